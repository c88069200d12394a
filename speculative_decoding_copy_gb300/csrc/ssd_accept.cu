// Vocabulary rows, acceptance, longest-block choice and the final draw.
//
// Speculative Decoding 해부 page: §2 Phase 3 — drafts are checked in order, the
// first rejection truncates the draft and a token from the residual replaces
// it; if every draft is accepted a bonus token is drawn from the next target
// distribution. §3.1 — accept x with probability min(1, p(x)/q(x)), read as
// u*q(x) < p(x). §3.2 — residual max(0, p - q) normalised. SwitchSD page,
// "무엇과 다른가" — after verifying W candidates at once the longest verified
// continuation is adopted. 추측 디코딩은 왜… page, "2단계 · 일괄 검증" — greedy:
// a match is accepted, the first mismatch truncates.
//
// Kernels (one stream, in order):
//   k_vocab_stats   grid (chunks, rows, B): per needed row and vocabulary chunk,
//                   max, sum of exp(l - max) and argmax (lowest index on ties);
//                   a single streaming pass over the logits (HBM-bound);
//   k_accept_select grid B: merges the chunks of each needed row, runs the
//                   acceptance scan of every block (one warp per block, one
//                   lane per token, ballot for the leading run), picks the
//                   longest block and writes the accepted tokens;
//   k_sample_final  grid (chunks, B), sample mode only: integer weights of the
//                   stop row per chunk, then the last CTA of each sequence
//                   finds the chunk and the index where the prefix sum crosses
//                   the threshold (no spin-wait: a completion counter);
//   k_probs_out     optional diagnostic copy of p for every needed row.
#include <math.h>

#include "ssd_accept.cuh"

namespace ssd {

constexpr int kVocabThreads = 256;
constexpr int kSelectThreads = 256;
constexpr int kMaxRows = 2048;          // 1 + NB*Dmax + K
constexpr long long kOneWeight = 1LL << 40;

__device__ __forceinline__ float load_val(const void* base, int64_t i, int bf16) {
  return bf16 ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(base) + i))
              : __ldg(static_cast<const float*>(base) + i);
}

// p of one entry: exp(l - max) / Z in fp32, or the value itself for probabilities
__device__ __forceinline__ float prob_of(float v, const RowStat& st, int probs) {
  return probs ? v : expf(v - st.m) / st.s;
}

// P = floor(p * 2^40): exact for fp32 p in [0, 1]
__device__ __forceinline__ long long weight_of(float p) {
  return __double2ll_rd(static_cast<double>(p) * 1099511627776.0);
}

__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * expf(m - M) + s2 * expf(m2 - M);
  m = M;
}

__device__ __forceinline__ void amax_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ bool row_needed(const AcceptParams& p, int b, int r) {
  if (r == 0) return true;
  if (r < p.NR) {
    const int sl = r - 1, k = sl / p.Dmax, pos = sl % p.Dmax;
    return pos < p.blk_len[b * p.NB + k];
  }
  const int i = r - p.NR;   // < K by the grid
  return p.chain_blk >= 0 && i < p.blk_len[b * p.NB + p.chain_blk];
}

__device__ __forceinline__ const void* row_ptr(const AcceptParams& p, int b, int r) {
  const size_t es = p.bf16 ? 2 : 4;
  if (r < p.NR)
    return static_cast<const char*>(p.tgt) + (static_cast<int64_t>(b) * p.NR + r) * p.V * es;
  return static_cast<const char*>(p.drf) + (static_cast<int64_t>(b) * p.K + (r - p.NR)) * p.V * es;
}

// ------------------------------------------------------------------ stats
__device__ void vocab_stats_one(const AcceptParams& p, int b, int r, int c);

__global__ void __launch_bounds__(kVocabThreads)
k_vocab_stats(AcceptParams p) {
  const int c = blockIdx.x % p.nch, r = blockIdx.x / p.nch;
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) vocab_stats_one(p, b, r, c);
}

__device__ void vocab_stats_one(const AcceptParams& p, int b, int r, int c) {
  if (!row_needed(p, b, r)) return;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int64_t lo = static_cast<int64_t>(c) * p.chunk;
  const int64_t hi = min(p.V, lo + p.chunk);
  const void* row = row_ptr(p, b, r);

  float m = -INFINITY, s = 0.f, av = -INFINITY;
  int ai = 0x7fffffff;
  if (lo < hi) {
    const bool vec_ok = aligned_dev(row, 16);
    const int64_t n = hi - lo;
    if (!p.bf16) {
      const float* f = static_cast<const float*>(row);
      int64_t nv = vec_ok ? n / 4 : 0;
      const float4* f4 = reinterpret_cast<const float4*>(f + lo);
      for (int64_t v = tid; v < nv; v += kVocabThreads) {
        const float4 x = __ldg(f4 + v);
        const int i0 = static_cast<int>(lo + v * 4);
        if (x.x > av) { av = x.x; ai = i0; }
        if (x.y > av) { av = x.y; ai = i0 + 1; }
        if (x.z > av) { av = x.z; ai = i0 + 2; }
        if (x.w > av) { av = x.w; ai = i0 + 3; }
        if (!p.probs) {
          const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
          if (mx > m) { s *= expf(m - mx); m = mx; }
          s += expf(x.x - m) + expf(x.y - m) + expf(x.z - m) + expf(x.w - m);
        }
      }
      for (int64_t i = lo + nv * 4 + tid; i < hi; i += kVocabThreads) {
        const float x = __ldg(f + i);
        if (x > av) { av = x; ai = static_cast<int>(i); }
        if (!p.probs) {
          if (x > m) { s *= expf(m - x); m = x; }
          s += expf(x - m);
        }
      }
    } else {
      const uint16_t* hb = static_cast<const uint16_t*>(row);
      int64_t nv = vec_ok ? n / 8 : 0;
      const uint4* h8 = reinterpret_cast<const uint4*>(hb + lo);
      for (int64_t v = tid; v < nv; v += kVocabThreads) {
        const uint4 u = __ldg(h8 + v);
        const int i0 = static_cast<int>(lo + v * 8);
        float x[8];
        x[0] = __uint_as_float(u.x << 16); x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16); x[3] = __uint_as_float(u.y & 0xffff0000u);
        x[4] = __uint_as_float(u.z << 16); x[5] = __uint_as_float(u.z & 0xffff0000u);
        x[6] = __uint_as_float(u.w << 16); x[7] = __uint_as_float(u.w & 0xffff0000u);
        float mx = x[0];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (x[q] > av) { av = x[q]; ai = i0 + q; }
          mx = fmaxf(mx, x[q]);
        }
        if (mx > m) { s *= expf(m - mx); m = mx; }
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) acc += expf(x[q] - m);
        s += acc;
      }
      for (int64_t i = lo + nv * 8 + tid; i < hi; i += kVocabThreads) {
        const float x = bf16_to_f32(__ldg(hb + i));
        if (x > av) { av = x; ai = static_cast<int>(i); }
        if (x > m) { s *= expf(m - x); m = x; }
        s += expf(x - m);
      }
    }
  }
  // block reduction
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
    stat_merge(m, s, m2, s2);
    amax_merge(av, ai, v2, i2);
  }
  __shared__ RowStat red[kVocabThreads / 32];
  if (lane == 0) red[wid] = RowStat{m, s, av, ai};
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kVocabThreads / 32; ++w) {
      stat_merge(m, s, red[w].m, red[w].s);
      amax_merge(av, ai, red[w].amax_v, red[w].amax_i);
    }
    p.part[(static_cast<int64_t>(b) * p.NRD + r) * p.nch + c] = RowStat{m, s, av, ai};
  }
  __syncthreads();   // red[] is reused by the next sequence of this CTA
}

// ------------------------------------------------------------------ select
__global__ void __launch_bounds__(kSelectThreads)
k_accept_select(AcceptParams p) {
  __shared__ RowStat st[kMaxRows];
  __shared__ int acc_s[256];
  __shared__ int len_s[256];
  __shared__ int sel[4];   // best block, a, len, final (greedy)
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int nw = kSelectThreads / 32;

  // block lengths, clamped to the slots that exist (a chain block to K draft rows)
  for (int k = tid; k < p.NB; k += kSelectThreads) {
    const int raw = p.blk_len[b * p.NB + k];
    const int cap = (k == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
    const int L = min(max(raw, 0), cap);
    if (L != raw) record_error(p.hdr, SSD_ERR_DEVICE, 101);
    len_s[k] = L;
  }

  // 1. merge the chunks of every needed row
  for (int r = wid; r < p.NRD; r += nw) {
    if (!row_needed(p, b, r)) continue;
    float m = -INFINITY, s = 0.f, av = -INFINITY;
    int ai = 0x7fffffff;
    const RowStat* pr = p.part + (static_cast<int64_t>(b) * p.NRD + r) * p.nch;
    for (int c = lane; c < p.nch; c += 32) {
      const RowStat x = pr[c];
      stat_merge(m, s, x.m, x.s);
      amax_merge(av, ai, x.amax_v, x.amax_i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
      stat_merge(m, s, m2, s2);
      amax_merge(av, ai, v2, i2);
    }
    if (lane == 0) {
      const RowStat x{m, s, av, ai};
      st[r] = x;
      p.stat[static_cast<int64_t>(b) * p.NRD + r] = x;
    }
  }
  __syncthreads();

  // 2. acceptance scan: one warp per block, one lane per token
  for (int k = wid; k < p.NB; k += nw) {
    const int L = len_s[k];
    const bool chain = (k == p.chain_blk);
    int a = 0;
    for (int d0 = 0; d0 < L; d0 += 32) {
      const int d = d0 + lane;
      bool ok = false;
      if (d < L) {
        const int x = p.blk_tok[(static_cast<int64_t>(b) * p.NB + k) * p.Dmax + d];
        const int r = d == 0 ? 0 : 1 + k * p.Dmax + d - 1;
        if (x < 0 || x >= p.V) {
          record_error(p.hdr, SSD_ERR_DEVICE, 100);
        } else if (!p.sample) {
          ok = (x == st[r].amax_i);
        } else {
          const float px = prob_of(load_val(row_ptr(p, b, r), x, p.bf16), st[r], p.probs);
          float qx = 1.f;
          if (chain) qx = prob_of(load_val(row_ptr(p, b, p.NR + d), x, p.bf16), st[p.NR + d], p.probs);
          const float u = p.u_acc[(static_cast<int64_t>(b) * p.NB + k) * p.Dmax + d];
          ok = __dmul_rn(static_cast<double>(u), static_cast<double>(qx)) < static_cast<double>(px);
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      const int run = __ffs(~bal) - 1;          // leading accepted lanes (-1 if all 32)
      if (run < 0) {
        a += min(32, L - d0);
        if (L - d0 <= 32) break;
      } else {
        a += min(run, L - d0);
        break;
      }
    }
    if (lane == 0) {
      acc_s[k] = a;
      p.acc_len[b * p.NB + k] = a;
    }
  }
  __syncthreads();

  // 3. longest accepted run, lowest block index on ties
  if (tid == 0) {
    int best = -1, ba = -1;
    for (int k = 0; k < p.NB; ++k) {
      if (len_s[k] > 0 && acc_s[k] > ba) {
        ba = acc_s[k];
        best = k;
      }
    }
    const int a = best >= 0 ? ba : 0;
    const int L = best >= 0 ? len_s[best] : 0;
    const int stop = a == 0 ? 0 : 1 + best * p.Dmax + a - 1;
    sel[0] = best;
    sel[1] = a;
    sel[2] = L;
    sel[3] = st[stop].amax_i;
    p.best_blk[b] = best;
    p.n_out[b] = a + 1;
    if (p.sample) {
      StopInfo si;
      si.row = stop;
      si.a = a;
      si.drf_row = -1;
      si.excl = -1;
      si.bonus = (a >= L) ? 1 : 0;
      if (a < L) {
        if (best == p.chain_blk) si.drf_row = a;
        else si.excl = p.blk_tok[(static_cast<int64_t>(b) * p.NB + best) * p.Dmax + a];
      }
      p.stop[b] = si;
      p.cnt[b] = 0u;
    }
  }
  __syncthreads();

  // 4. emitted tokens (the sampler fills the final one in sample mode)
  const int best = sel[0], a = sel[1];
  for (int i = tid; i <= p.Dmax; i += kSelectThreads) {
    int v = -1;
    if (i < a) v = p.blk_tok[(static_cast<int64_t>(b) * p.NB + best) * p.Dmax + i];
    else if (i == a && !p.sample) v = sel[3];
    p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + i] = v;
  }
}

// ------------------------------------------------------------------ final draw
__device__ __forceinline__ void weights_at(const AcceptParams& p, const void* prow, const RowStat& ps,
                                           const void* qrow, const RowStat& qs, int excl, int bonus,
                                           int64_t i, long long& W, long long& P) {
  P = weight_of(prob_of(load_val(prow, i, p.bf16), ps, p.probs));
  if (bonus) {
    W = P;
    return;
  }
  long long Q;
  if (qrow != nullptr) Q = weight_of(prob_of(load_val(qrow, i, p.bf16), qs, p.probs));
  else Q = (i == excl) ? kOneWeight : 0LL;
  W = P > Q ? P - Q : 0LL;
}

__device__ void sample_final_one(const AcceptParams& p, int b, int c);

__global__ void __launch_bounds__(kVocabThreads)
k_sample_final(AcceptParams p) {
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    sample_final_one(p, b, blockIdx.x);
    __syncthreads();   // shared state is reused by the next sequence of this CTA
  }
}

__device__ void sample_final_one(const AcceptParams& p, int b, int c) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int nw = kVocabThreads / 32;
  __shared__ long long red_w[nw], red_p[nw];
  __shared__ int is_last;
  __shared__ long long t_rem;
  __shared__ int c_star, use_bonus;

  const StopInfo si = p.stop[b];
  const void* prow = row_ptr(p, b, si.row);
  const RowStat ps = p.stat[static_cast<int64_t>(b) * p.NRD + si.row];
  const void* qrow = si.drf_row >= 0 ? row_ptr(p, b, p.NR + si.drf_row) : nullptr;
  const RowStat qs = si.drf_row >= 0 ? p.stat[static_cast<int64_t>(b) * p.NRD + p.NR + si.drf_row] : ps;

  // phase 1: this chunk's residual and bonus weight sums
  const int64_t lo = static_cast<int64_t>(c) * p.schunk;
  const int64_t hi = min(p.V, lo + p.schunk);
  long long sw = 0, sp = 0;
  for (int64_t i = lo + tid; i < hi; i += kVocabThreads) {
    long long W, P;
    weights_at(p, prow, ps, qrow, qs, si.excl, si.bonus, i, W, P);
    sw += W;
    sp += P;
  }
  sw = warp_sum(sw);
  sp = warp_sum(sp);
  if (lane == 0) { red_w[wid] = sw; red_p[wid] = sp; }
  __syncthreads();
  if (tid == 0) {
    long long tw = 0, tp = 0;
    for (int w = 0; w < nw; ++w) { tw += red_w[w]; tp += red_p[w]; }
    p.csum[(static_cast<int64_t>(b) * p.nchs + c) * 2 + 0] = tw;
    p.csum[(static_cast<int64_t>(b) * p.nchs + c) * 2 + 1] = tp;
    __threadfence();
    const unsigned ticket = atomicAdd(p.cnt + b, 1u);
    is_last = (ticket == static_cast<unsigned>(p.nchs - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // phase 2 (last CTA of this sequence): threshold, chunk, index
  if (tid == 0) {
    const volatile long long* cs = p.csum + static_cast<int64_t>(b) * p.nchs * 2;
    long long SW = 0, SP = 0;
    for (int k = 0; k < p.nchs; ++k) { SW += cs[2 * k]; SP += cs[2 * k + 1]; }
    const int ub = (si.bonus || SW == 0) ? 1 : 0;
    const unsigned long long S = static_cast<unsigned long long>(ub ? SP : SW);
    const float u = fminf(fmaxf(p.u_fin[b], 0.f), 0.99999994f);   // contract: u in [0, 1)
    const unsigned long long U = static_cast<unsigned long long>(u * 16777216.0f);   // floor(u 2^24), exact
    const unsigned long long lo64 = U * S;
    const unsigned long long hi64 = __umul64hi(U, S);
    const long long T = static_cast<long long>((hi64 << 40) | (lo64 >> 24));
    long long acc = 0;
    int cs_i = p.nchs - 1;
    for (int k = 0; k < p.nchs; ++k) {
      const long long wk = cs[2 * k + (ub ? 1 : 0)];
      if (acc + wk > T) { cs_i = k; break; }
      acc += wk;
    }
    c_star = cs_i;
    t_rem = T - acc;
    use_bonus = ub;
    p.cnt[b] = 0u;
  }
  __syncthreads();
  const int64_t lo2 = static_cast<int64_t>(c_star) * p.schunk;
  const int64_t hi2 = min(p.V, lo2 + p.schunk);
  const int64_t per = (hi2 - lo2 + kVocabThreads - 1) / kVocabThreads;
  const int64_t my_lo = min(hi2, lo2 + tid * per), my_hi = min(hi2, my_lo + per);
  const int ub = use_bonus;
  long long mine = 0;
  for (int64_t i = my_lo; i < my_hi; ++i) {
    long long W, P;
    weights_at(p, prow, ps, qrow, qs, si.excl, si.bonus, i, W, P);
    mine += ub ? P : W;
  }
  // exclusive block scan of `mine`
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) red_w[wid] = incl;
  __syncthreads();
  long long wofs = 0;
  for (int w = 0; w < wid; ++w) wofs += red_w[w];
  const long long excl = wofs + incl - mine;
  const long long Tr = t_rem;
  if (mine > 0 && excl <= Tr && Tr < excl + mine) {
    long long acc = excl;
    int64_t tok = my_hi - 1;
    for (int64_t i = my_lo; i < my_hi; ++i) {
      long long W, P;
      weights_at(p, prow, ps, qrow, qs, si.excl, si.bonus, i, W, P);
      acc += ub ? P : W;
      if (acc > Tr) { tok = i; break; }
    }
    p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + si.a] = static_cast<int>(tok);
  }
}

// ------------------------------------------------------------------ diagnostics
__global__ void __launch_bounds__(kVocabThreads)
k_probs_out(AcceptParams p) {
  const int c = blockIdx.x % p.nch, r = blockIdx.x / p.nch;
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    if (!row_needed(p, b, r)) continue;
    const RowStat st = p.stat[static_cast<int64_t>(b) * p.NRD + r];
    const void* row = row_ptr(p, b, r);
    const int64_t lo = static_cast<int64_t>(c) * p.chunk;
    const int64_t hi = min(p.V, lo + p.chunk);
    float* out = p.probs_out + (static_cast<int64_t>(b) * p.NR + r) * p.V;
    for (int64_t i = lo + threadIdx.x; i < hi; i += kVocabThreads)
      out[i] = prob_of(load_val(row, i, p.bf16), st, p.probs);
  }
}

// ------------------------------------------------------------------ host
AcceptLayout accept_layout(const ssd_accept_args* a) {
  AcceptLayout L{};
  const int NR = 1 + a->NB * a->Dmax;
  const int NRD = NR + (a->chain_blk >= 0 ? a->K : 0);
  L.NR = NR;
  L.NRD = NRD;
  // vocabulary chunks per row: about 8 CTAs per SM in total, multiples of 8 elements
  const long long rows = static_cast<long long>(a->B) * NRD;
  long long nch = (8LL * 152 + rows - 1) / (rows > 0 ? rows : 1);
  const long long max_nch = (a->V + 2047) / 2048;            // at least 2048 elements per chunk
  if (nch > max_nch) nch = max_nch;
  if (nch > 64) nch = 64;
  if (nch < 1) nch = 1;
  long long chunk = (a->V + nch - 1) / nch;
  chunk = (chunk + 7) / 8 * 8;
  nch = (a->V + chunk - 1) / chunk;
  L.nch = static_cast<int>(nch);
  L.chunk = chunk;
  // sampler chunks: about 2 CTAs per SM over the batch
  long long nchs = (2LL * 152 + a->B - 1) / (a->B > 0 ? a->B : 1);
  const long long max_nchs = (a->V + 1023) / 1024;
  if (nchs > max_nchs) nchs = max_nchs;
  if (nchs > 128) nchs = 128;
  if (nchs < 1) nchs = 1;
  long long schunk = (a->V + nchs - 1) / nchs;
  schunk = (schunk + 7) / 8 * 8;
  nchs = (a->V + schunk - 1) / schunk;
  L.nchs = static_cast<int>(nchs);
  L.schunk = schunk;

  size_t off = sizeof(WsHeader);
  L.part_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * NRD * L.nch * sizeof(RowStat), 256);
  L.stat_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * NRD * sizeof(RowStat), 256);
  L.stop_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * sizeof(StopInfo), 256);
  L.csum_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * L.nchs * 2 * sizeof(long long), 256);
  L.cnt_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * sizeof(unsigned), 256);
  L.total = off;
  return L;
}

int accept_validate(const ssd_accept_args* a) {
  if (a == nullptr) return SSD_ERR_INVALID;
  if (a->mode != SSD_GREEDY && a->mode != SSD_SAMPLE) return SSD_ERR_INVALID;
  if (a->kind != SSD_LOGITS_F32 && a->kind != SSD_LOGITS_BF16 && a->kind != SSD_PROBS_F32) return SSD_ERR_INVALID;
  if (a->B < 0 || a->NB < 1 || a->Dmax < 1 || a->K < 0 || a->V < 2) return SSD_ERR_INVALID;
  if (a->V >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  if (a->Dmax > 256) return SSD_ERR_UNSUPPORTED;
  if (a->chain_blk < -1 || a->chain_blk >= a->NB) return SSD_ERR_INVALID;
  if (a->NB > 256) return SSD_ERR_UNSUPPORTED;
  const long long nrd = 1LL + static_cast<long long>(a->NB) * a->Dmax + (a->chain_blk >= 0 ? a->K : 0);
  if (nrd > kMaxRows) return SSD_ERR_UNSUPPORTED;
  if (a->chain_blk >= 0 && (a->K < 1 || a->K > a->Dmax)) return SSD_ERR_INVALID;
  if (a->B == 0) return SSD_OK;
  if (!a->tgt || !a->blk_tok || !a->blk_len || !a->acc_len || !a->best_blk || !a->n_out || !a->out_tok)
    return SSD_ERR_INVALID;
  if (a->chain_blk >= 0 && !a->drf) return SSD_ERR_INVALID;
  if (a->mode == SSD_SAMPLE && (!a->u_acc || !a->u_fin)) return SSD_ERR_INVALID;
  return SSD_OK;
}

AcceptParams accept_params(const ssd_accept_args* a, const AcceptLayout& L, char* base) {
  AcceptParams p{};
  p.tgt = a->tgt;
  p.drf = a->drf;
  p.V = a->V;
  p.blk_tok = a->blk_tok;
  p.blk_len = a->blk_len;
  p.B = a->B; p.NB = a->NB; p.Dmax = a->Dmax; p.K = a->chain_blk >= 0 ? a->K : 0; p.chain_blk = a->chain_blk;
  p.NR = L.NR; p.NRD = L.NRD;
  p.u_acc = a->u_acc; p.u_fin = a->u_fin;
  p.acc_len = a->acc_len; p.best_blk = a->best_blk; p.n_out = a->n_out; p.out_tok = a->out_tok;
  p.probs_out = a->probs_out;
  p.sample = a->mode == SSD_SAMPLE;
  p.bf16 = a->kind == SSD_LOGITS_BF16;
  p.probs = a->kind == SSD_PROBS_F32;
  p.nch = L.nch; p.chunk = L.chunk; p.nchs = L.nchs; p.schunk = L.schunk;
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.part = reinterpret_cast<RowStat*>(base + L.part_off);
  p.stat = reinterpret_cast<RowStat*>(base + L.stat_off);
  p.stop = reinterpret_cast<StopInfo*>(base + L.stop_off);
  p.csum = reinterpret_cast<long long*>(base + L.csum_off);
  p.cnt = reinterpret_cast<unsigned*>(base + L.cnt_off);
  return p;
}

int accept_launch(const AcceptParams& p, cudaStream_t s) {
  const unsigned by = static_cast<unsigned>(p.B < 65535 ? p.B : 65535);
  dim3 g1(static_cast<unsigned>(p.nch * p.NRD), by);
  {
    KernelTimer t(SSD_KERNEL_VOCAB_STATS, s);
    k_vocab_stats<<<g1, kVocabThreads, 0, s>>>(p);
  }
  {
    KernelTimer t(SSD_KERNEL_ACCEPT_SELECT, s);
    k_accept_select<<<p.B, kSelectThreads, 0, s>>>(p);
  }
  int n = 2;
  if (p.sample) {
    dim3 g3(static_cast<unsigned>(p.nchs), by);
    KernelTimer t(SSD_KERNEL_SAMPLE_FINAL, s);
    k_sample_final<<<g3, kVocabThreads, 0, s>>>(p);
    ++n;
  }
  if (p.probs_out != nullptr) {
    dim3 g4(static_cast<unsigned>(p.nch * p.NR), by);
    k_probs_out<<<g4, kVocabThreads, 0, s>>>(p);
    ++n;
  }
  count_launch(n);
  return check_launch();
}

}  // namespace ssd

using namespace ssd;

extern "C" size_t ssd_accept_workspace_size(const ssd_accept_args* a) {
  if (accept_validate(a) != SSD_OK) return 0;
  return accept_layout(a).total;
}

extern "C" int ssd_accept(const ssd_accept_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = accept_validate(a);
  if (st != SSD_OK) return st;
  if (a->B == 0) return SSD_OK;
  if (ws == nullptr || !aligned(ws, 256)) return SSD_ERR_WORKSPACE;
  const AcceptLayout L = accept_layout(a);
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const AcceptParams p = accept_params(a, L, static_cast<char*>(ws));
  return accept_launch(p, static_cast<cudaStream_t>(stream));
}
