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
// Kernels (one stream, in order; each later kernel is launched with
// programmatic dependent launch and waits for its predecessor's results):
//   k_vocab_stats   persistent CTAs over (sequence, row, chunk) tasks: one
//                   16-byte-vector pass over the logits, a whole 32 KB chunk
//                   in registers per task and the next task's loads in flight
//                   while the current one is reduced to max, argmax (lowest
//                   index on ties) and sum of 2^((l - max) log2 e);
//   k_accept_select grid B: merges the chunks of every needed row, runs the
//                   acceptance test of every candidate token (one thread per
//                   token slot, loads issued together), picks the longest
//                   accepted block and writes the accepted tokens;
//   k_sample_final  grid (chunks, B), sample mode only: integer weights of the
//                   stop row per chunk; the last CTA of each sequence (a
//                   completion counter, no spin-wait) finds the chunk and the
//                   index where the prefix sum crosses the threshold with
//                   block-wide scans;
//   k_probs_out     optional diagnostic copy of p for every needed row.
#include <math.h>

#include <mutex>

#include "ssd_accept.cuh"

namespace ssd {

constexpr int kVocabThreads = 256;
constexpr int kVec = 8;                 // 16-byte vectors per thread per stats chunk
constexpr int kSelectThreads = 256;
constexpr int kMaxRows = 1024;          // 1 + NB*Dmax + K
constexpr int kMaxSlots = 1024;         // NB*Dmax
constexpr int kSampleChunk = 2048;      // vocabulary entries per sampler CTA
constexpr int kSamplePer = kSampleChunk / kVocabThreads;
constexpr long long kOneWeight = 1LL << 40;

__device__ __forceinline__ float load_val(const void* base, int64_t i, int bf16) {
  return bf16 ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(base) + i))
              : __ldg(static_cast<const float*>(base) + i);
}

// p of one entry: 2^((l - max) log2 e) / Z in fp32, or the value itself for probabilities
__device__ __forceinline__ float prob_of(float v, const RowStat& st, int probs) {
  return probs ? v : ex2_approx(fmaf(v, kLog2e, -st.m * kLog2e)) * __frcp_rn(st.s);
}

// P = floor(p * 2^40) for fp32 p in [0, 1], exactly, from the bits of p
__device__ __forceinline__ long long weight_of(float p) {
  const uint32_t u = __float_as_uint(p);
  if (static_cast<int32_t>(u) <= 0) return 0;            // +0 or negative
  const int e = static_cast<int>(u >> 23);                // biased exponent (0: subnormal, < 2^-126)
  if (e == 0) return 0;
  const long long mant = static_cast<long long>((u & 0x7fffffu) | 0x800000u);
  const int sh = e - 110;                                 // p * 2^40 = mant * 2^(e - 127 - 23 + 40)
  if (sh >= 0) return mant << min(sh, 30);
  return sh <= -24 ? 0 : (mant >> (-sh));
}

__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * ex2_approx((m - M) * kLog2e) + s2 * ex2_approx((m2 - M) * kLog2e);
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

// block-wide exclusive prefix sum over the 256 threads; *total gets the sum
__device__ __forceinline__ long long block_excl_scan(long long v, long long* warp_tot, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kVocabThreads / 32; ++w) {
    const long long t = warp_tot[w];
    if (w < wid) before += t;
    all += t;
  }
  *total = all;
  return before + incl - v;
}

// ------------------------------------------------------------------ stats
// element e (0..EPV-1) of a 16-byte vector
template <bool BF16>
__device__ __forceinline__ float vec_elem(const uint4& u, int e) {
  const uint32_t w = e < (BF16 ? 2 : 1) ? u.x : e < (BF16 ? 4 : 2) ? u.y : e < (BF16 ? 6 : 3) ? u.z : u.w;
  if (BF16) return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  return __uint_as_float(w);
}

// One chunk of one row as 16-byte vectors held in registers (32 per thread).
// Elements past the row end (or an unaligned row) are gathered one by one; the
// padding is -inf.
template <bool BF16>
__device__ __forceinline__ void load_chunk(const void* row, int64_t lo, int64_t hi, bool vec_ok, uint4* raw) {
  constexpr int EPV = BF16 ? 8 : 4;    // elements per 16-byte vector
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int64_t i0 = lo + static_cast<int64_t>(v * kVocabThreads + threadIdx.x) * EPV;
    if (vec_ok && i0 + EPV <= hi) {
      raw[v] = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(row) + i0 * (BF16 ? 2 : 4)));
    } else {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) w[q] = BF16 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        if (i0 + e < hi) {
          if (BF16) {
            const uint32_t h = __ldg(static_cast<const uint16_t*>(row) + i0 + e);
            w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0xffffu) | (h << 16)) : ((w[e >> 1] & 0xffff0000u) | h);
          } else {
            w[e] = __float_as_uint(__ldg(static_cast<const float*>(row) + i0 + e));
          }
        }
      }
      raw[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// max, argmax (lowest index on ties) and sum of 2^((x - max) log2 e) of this thread's elements
template <bool BF16>
__device__ __forceinline__ void reduce_chunk(const uint4* raw, int64_t lo, bool probs, float& m, float& s, float& av,
                                             int& ai) {
  constexpr int EPV = BF16 ? 8 : 4;
  av = -INFINITY;
  ai = 0x7fffffff;
#pragma unroll
  for (int v = 0; v < kVec; ++v) {
    const int i0 = static_cast<int>(lo + static_cast<int64_t>(v * kVocabThreads + threadIdx.x) * EPV);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float x = vec_elem<BF16>(raw[v], e);
      if (x > av) {                      // indices increase: strict > keeps the lowest on ties
        av = x;
        ai = i0 + e;
      }
    }
  }
  m = av;
  s = 0.f;
  if (!probs && m > -INFINITY) {
    const float c = -m * kLog2e;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
#pragma unroll
      for (int e = 0; e < EPV; e += 2) {
        s0 += ex2_approx(fmaf(vec_elem<BF16>(raw[v], e), kLog2e, c));
        s1 += ex2_approx(fmaf(vec_elem<BF16>(raw[v], e + 1), kLog2e, c));
      }
    }
    s = s0 + s1;
  }
}

// ------------------------------------------------------------------ select
constexpr int kSlotsPer = kMaxSlots / kSelectThreads;

struct SelectSmem {
  RowStat st[kMaxRows];
  int len_s[256];
  int acc_s[256];
  unsigned char ok_s[kMaxSlots];
  int sel[4];   // best block, a, len, final (greedy)
};

// Acceptance and choice of block for sequence b, by one CTA of 256 threads,
// once every needed row's chunk statistics are in p.part.
__device__ void select_one(const AcceptParams& p, int b, SelectSmem& sm) {
  RowStat* st = sm.st;
  int* len_s = sm.len_s;
  int* acc_s = sm.acc_s;
  unsigned char* ok_s = sm.ok_s;
  int* sel = sm.sel;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int nw = kSelectThreads / 32;
  const int nslots = p.NB * p.Dmax;

  // 1. per token slot: its token, its block's length, its uniform and the logits
  //    the acceptance test needs; every load is issued before the row merge
  int x_[kSlotsPer], row_[kSlotsPer];
  bool live_[kSlotsPer];
  float lp_[kSlotsPer], lq_[kSlotsPer], u_[kSlotsPer];
#pragma unroll
  for (int k = 0; k < kSlotsPer; ++k) {
    const int sl = tid + k * kSelectThreads;
    live_[k] = false;
    x_[k] = 0;
    row_[k] = 0;
    lp_[k] = 0.f;
    lq_[k] = 0.f;
    u_[k] = 0.f;
    if (sl < nslots) {
      const int blk = sl / p.Dmax, d = sl % p.Dmax;
      const int raw = p.blk_len[b * p.NB + blk];
      const int cap = (blk == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
      const int L = min(max(raw, 0), cap);
      if (d < L) {
        const int x = p.blk_tok[static_cast<int64_t>(b) * nslots + sl];
        if (x < 0 || x >= p.V) {
          record_error(p.hdr, SSD_ERR_DEVICE, 100);
        } else {
          live_[k] = true;
          x_[k] = x;
          row_[k] = d == 0 ? 0 : 1 + blk * p.Dmax + d - 1;
          if (p.sample) {
            lp_[k] = load_val(row_ptr(p, b, row_[k]), x, p.bf16);
            if (blk == p.chain_blk) lq_[k] = load_val(row_ptr(p, b, p.NR + d), x, p.bf16);
            u_[k] = p.u_acc[static_cast<int64_t>(b) * nslots + sl];
          }
        }
      }
    }
  }
  for (int k = tid; k < p.NB; k += kSelectThreads) {
    const int raw = p.blk_len[b * p.NB + k];
    const int cap = (k == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
    const int L = min(max(raw, 0), cap);
    if (L != raw) record_error(p.hdr, SSD_ERR_DEVICE, 101);
    len_s[k] = L;
  }

  __syncthreads();   // len_s
  // 2. merge the vocabulary chunks of every needed row: one thread per row, its
  //    chunk partials loaded together, max first, then one scaled sum
  for (int r = tid; r < p.NRD; r += kSelectThreads) {
    bool needed = r == 0;
    if (r > 0 && r < p.NR) needed = ((r - 1) % p.Dmax) < len_s[(r - 1) / p.Dmax];
    else if (r >= p.NR) needed = p.chain_blk >= 0 && (r - p.NR) < len_s[p.chain_blk];
    if (!needed) continue;
    const RowStat* src = p.part + (static_cast<int64_t>(b) * p.NRD + r) * p.nch;
    float M = -INFINITY, S = 0.f, av = -INFINITY;
    int ai = 0x7fffffff;
    for (int c0 = 0; c0 < p.nch; c0 += 16) {
      float4 v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q)
        v[q] = (c0 + q < p.nch) ? __ldcg(reinterpret_cast<const float4*>(src + c0 + q))
                                : make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(0x7fffffff));
      float Mb = -INFINITY;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        Mb = fmaxf(Mb, v[q].x);
        amax_merge(av, ai, v[q].z, __float_as_int(v[q].w));
      }
      const float Mn = fmaxf(M, Mb);
      if (Mn > -INFINITY) {
        float acc = (M > -INFINITY) ? S * ex2_approx((M - Mn) * kLog2e) : 0.f;
#pragma unroll
        for (int q = 0; q < 16; ++q)
          if (v[q].x > -INFINITY) acc += v[q].y * ex2_approx((v[q].x - Mn) * kLog2e);
        S = acc;
        M = Mn;
      }
    }
    const RowStat x{M, S, av, ai};
    st[r] = x;
    p.stat[static_cast<int64_t>(b) * p.NRD + r] = x;
  }
  __syncthreads();

  // 3. acceptance test of every present token
#pragma unroll
  for (int k = 0; k < kSlotsPer; ++k) {
    const int sl = tid + k * kSelectThreads;
    if (sl >= nslots) continue;
    bool ok = false;
    if (live_[k]) {
      const int blk = sl / p.Dmax, d = sl % p.Dmax;
      if (!p.sample) {
        ok = (x_[k] == st[row_[k]].amax_i);
      } else {
        const float px = prob_of(lp_[k], st[row_[k]], p.probs);
        const float qx = (blk == p.chain_blk) ? prob_of(lq_[k], st[p.NR + d], p.probs) : 1.f;
        ok = __dmul_rn(static_cast<double>(u_[k]), static_cast<double>(qx)) < static_cast<double>(px);
      }
    }
    ok_s[sl] = ok ? 1 : 0;
  }
  __syncthreads();

  // 4. leading accepted run of every block
  for (int k = tid; k < p.NB; k += kSelectThreads) {
    const int L = len_s[k];
    int a = 0;
    while (a < L && ok_s[k * p.Dmax + a]) ++a;
    acc_s[k] = a;
    p.acc_len[b * p.NB + k] = a;
  }
  __syncthreads();

  // 5. longest accepted run, lowest block index on ties
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
      si.ps = st[stop];
      si.a = a;
      si.drf_row = -1;
      si.excl = -1;
      si.bonus = (a >= L) ? 1 : 0;
      si.qs = si.ps;
      if (a < L) {
        if (best == p.chain_blk) {
          si.drf_row = a;
          si.qs = st[p.NR + a];
        }
        else {
          si.excl = p.blk_tok[static_cast<int64_t>(b) * nslots + best * p.Dmax + a];
        }
      }
      p.stop[b] = si;
      p.cnt[b] = 0u;
    }
  }
  __syncthreads();

  // 6. emitted tokens (the sampler fills the final one in sample mode)
  const int best = sel[0], a = sel[1];
  for (int i = tid; i <= p.Dmax; i += kSelectThreads) {
    int v = -1;
    if (i < a) v = p.blk_tok[static_cast<int64_t>(b) * nslots + best * p.Dmax + i];
    else if (i == a && !p.sample) v = sel[3];
    p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + i] = v;
  }
  __syncthreads();
}

// next task (sequence, row, chunk) of this CTA whose row some token needs, or
// ntask; tasks are numbered ((b * NRD) + r) * nch + c (fits in 32 bits)
__device__ __forceinline__ int next_task(const AcceptParams& p, int t, int ntask) {
  for (; t < ntask; t += gridDim.x) {
    const int br = t / p.nch;
    const int b = br / p.NRD, r = br - b * p.NRD;
    if (row_needed(p, b, r)) break;
  }
  return t;
}

// Persistent CTAs walk the (sequence, row, chunk) tasks; the loads of the next
// task are in flight while the current one is reduced.
template <bool BF16>
__global__ void __launch_bounds__(kVocabThreads, 2)
k_vocab_stats(AcceptParams p) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  __shared__ RowStat red[kVocabThreads / 32];
  // let the next kernel of the stream start its launch while this one runs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // blk_len comes from the previous kernel of the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int ntask = p.nch * p.NRD * p.B;
  uint4 cur[kVec], nxt[kVec];
  int t = next_task(p, blockIdx.x, ntask);
  if (t < ntask) {
    const int br = t / p.nch, c = t - br * p.nch;
    const int b = br / p.NRD, r = br - b * p.NRD;
    const int64_t lo = static_cast<int64_t>(c) * p.chunk;
    const void* row = row_ptr(p, b, r);
    load_chunk<BF16>(row, lo, min(p.V, lo + p.chunk), aligned_dev(row, 16), cur);
  }
  while (t < ntask) {
    const int br = t / p.nch, c = t - br * p.nch;
    const int b = br / p.NRD, r = br - b * p.NRD;
    const int64_t lo = static_cast<int64_t>(c) * p.chunk;
    // prefetch the next task
    const int t2 = next_task(p, t + gridDim.x, ntask);
    if (t2 < ntask) {
      const int br2 = t2 / p.nch, c2 = t2 - br2 * p.nch;
      const int b2 = br2 / p.NRD, r2 = br2 - b2 * p.NRD;
      const int64_t lo2 = static_cast<int64_t>(c2) * p.chunk;
      const void* row2 = row_ptr(p, b2, r2);
      load_chunk<BF16>(row2, lo2, min(p.V, lo2 + p.chunk), aligned_dev(row2, 16), nxt);
    }
    float m, s, av;
    int ai;
    reduce_chunk<BF16>(cur, lo, p.probs, m, s, av, ai);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
      stat_merge(m, s, m2, s2);
      amax_merge(av, ai, v2, i2);
    }
    if (lane == 0) red[wid] = RowStat{m, s, av, ai};
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kVocabThreads / 32; ++w) {
        stat_merge(m, s, red[w].m, red[w].s);
        amax_merge(av, ai, red[w].amax_v, red[w].amax_i);
      }
      p.part[(static_cast<int64_t>(b) * p.NRD + r) * p.nch + c] = RowStat{m, s, av, ai};
    }
    __syncthreads();   // red[] is reused by the next task of this CTA
#pragma unroll
    for (int v = 0; v < kVec; ++v) cur[v] = nxt[v];
    t = t2;
  }
}

// one CTA per sequence, once every chunk statistic is in
__global__ void __launch_bounds__(kSelectThreads)
k_accept_select(AcceptParams p) {
  __shared__ SelectSmem sm;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");     // partials come from the stats kernel
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) select_one(p, b, sm);
}

// ------------------------------------------------------------------ final draw
// residual (or bonus) weight of entry i given its p and q values
__device__ __forceinline__ void weights_of(const AcceptParams& p, float pv, const RowStat& ps, bool has_q, float qv,
                                           const RowStat& qs, int excl, int bonus, int64_t i, long long& W,
                                           long long& P) {
  P = weight_of(prob_of(pv, ps, p.probs));
  if (bonus) {
    W = P;
    return;
  }
  const long long Q = has_q ? weight_of(prob_of(qv, qs, p.probs)) : ((i == excl) ? kOneWeight : 0LL);
  W = P > Q ? P - Q : 0LL;
}

__device__ void sample_final_one(const AcceptParams& p, int b, int c) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int nw = kVocabThreads / 32;
  __shared__ long long red_w[nw], red_p[nw];
  __shared__ int is_last, c_star, use_bonus;
  __shared__ long long t_rem;

  const StopInfo si = p.stop[b];
  const void* prow = row_ptr(p, b, si.row);
  const RowStat ps = si.ps;
  const bool has_q = si.drf_row >= 0;
  const void* qrow = has_q ? row_ptr(p, b, p.NR + si.drf_row) : prow;
  const RowStat qs = si.qs;

  // phase 1: this chunk's residual and bonus weight sums (all loads first)
  const int64_t lo = static_cast<int64_t>(c) * kSampleChunk;
  float pv[kSamplePer], qv[kSamplePer];
#pragma unroll
  for (int k = 0; k < kSamplePer; ++k) {
    const int64_t i = lo + k * kVocabThreads + tid;
    pv[k] = i < p.V ? load_val(prow, i, p.bf16) : 0.f;
    qv[k] = (has_q && i < p.V) ? load_val(qrow, i, p.bf16) : 0.f;
  }
  long long sw = 0, sp = 0;
#pragma unroll
  for (int k = 0; k < kSamplePer; ++k) {
    const int64_t i = lo + k * kVocabThreads + tid;
    if (i < p.V) {
      long long W, P;
      weights_of(p, pv[k], ps, has_q, qv[k], qs, si.excl, si.bonus, i, W, P);
      sw += W;
      sp += P;
    }
  }
  sw = warp_sum(sw);
  sp = warp_sum(sp);
  if (lane == 0) {
    red_w[wid] = sw;
    red_p[wid] = sp;
  }
  __syncthreads();
  if (tid == 0) {
    long long tw = 0, tp = 0;
    for (int w = 0; w < nw; ++w) {
      tw += red_w[w];
      tp += red_p[w];
    }
    p.csum[(static_cast<int64_t>(b) * p.nchs + c) * 2 + 0] = tw;
    p.csum[(static_cast<int64_t>(b) * p.nchs + c) * 2 + 1] = tp;
    __threadfence();
    const unsigned ticket = atomicAdd(p.cnt + b, 1u);
    is_last = (ticket == static_cast<unsigned>(p.nchs - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // phase 2 (last CTA of this sequence): totals, threshold, chunk
  // each thread owns a contiguous run of chunks
  const int cpt = (p.nchs + kVocabThreads - 1) / kVocabThreads;
  const int c_lo = min(p.nchs, tid * cpt), c_hi = min(p.nchs, c_lo + cpt);
  const volatile long long* cs = p.csum + static_cast<int64_t>(b) * p.nchs * 2;
  if (tid == 0) {            // defaults if no weight is positive (degenerate rows)
    c_star = 0;
    t_rem = 0;
    use_bonus = 1;
  }
  long long mw = 0, mp = 0;
  for (int k = c_lo; k < c_hi; ++k) {
    mw += cs[2 * k];
    mp += cs[2 * k + 1];
  }
  long long SW, SP;
  const long long ew = block_excl_scan(mw, red_w, &SW);
  const long long ep = block_excl_scan(mp, red_p, &SP);
  const int ub = (si.bonus || SW == 0) ? 1 : 0;
  const unsigned long long S = static_cast<unsigned long long>(ub ? SP : SW);
  const float u = fminf(fmaxf(p.u_fin[b], 0.f), 0.99999994f);               // contract: u in [0, 1)
  const unsigned long long U = static_cast<unsigned long long>(u * 16777216.0f);   // floor(u 2^24), exact
  const long long T = static_cast<long long>((__umul64hi(U, S) << 40) | ((U * S) >> 24));
  const long long mine = ub ? mp : mw, excl = ub ? ep : ew;
  if (mine > 0 && excl <= T && T < excl + mine) {
    long long acc = excl;
    int cst = c_hi - 1;
    for (int k = c_lo; k < c_hi; ++k) {
      const long long wk = cs[2 * k + ub];
      if (acc + wk > T) {
        cst = k;
        break;
      }
      acc += wk;
    }
    c_star = cst;
    t_rem = T - acc;
    use_bonus = ub;
  }
  if (tid == 0) p.cnt[b] = 0u;
  __syncthreads();

  // phase 3: the index inside chunk c_star; each thread owns kSamplePer contiguous entries
  const int64_t lo2 = static_cast<int64_t>(c_star) * kSampleChunk + tid * kSamplePer;
  const int ub2 = use_bonus;
#pragma unroll
  for (int k = 0; k < kSamplePer; ++k) {
    const int64_t i = lo2 + k;
    pv[k] = i < p.V ? load_val(prow, i, p.bf16) : 0.f;
    qv[k] = (has_q && i < p.V) ? load_val(qrow, i, p.bf16) : 0.f;
  }
  long long wv[kSamplePer];
  long long my = 0;
#pragma unroll
  for (int k = 0; k < kSamplePer; ++k) {
    const int64_t i = lo2 + k;
    long long W = 0, P = 0;
    if (i < p.V) weights_of(p, pv[k], ps, has_q, qv[k], qs, si.excl, si.bonus, i, W, P);
    wv[k] = ub2 ? P : W;
    my += wv[k];
  }
  long long tot;
  const long long ex = block_excl_scan(my, red_w, &tot);
  const long long Tr = t_rem;
  if (my > 0 && ex <= Tr && Tr < ex + my) {
    long long acc = ex;
    int64_t tok = lo2 + kSamplePer - 1;
#pragma unroll
    for (int k = 0; k < kSamplePer; ++k) {
      acc += wv[k];
      if (acc > Tr) {
        tok = lo2 + k;
        break;
      }
    }
    p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + si.a] = static_cast<int>(tok);
  }
}

__global__ void __launch_bounds__(kVocabThreads)
k_sample_final(AcceptParams p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");     // stop rows come from the previous kernel
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    sample_final_one(p, b, blockIdx.x);
    __syncthreads();   // shared state is reused by the next sequence of this CTA
  }
}

// ------------------------------------------------------------------ diagnostics
__global__ void __launch_bounds__(kVocabThreads)
k_probs_out(AcceptParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  // a stats chunk is one 16-byte vector per thread per step: 8 x 256 vectors
  const int64_t epv = (a->kind == SSD_LOGITS_BF16) ? 8 : 4;
  L.chunk = static_cast<int64_t>(kVec) * kVocabThreads * epv;
  L.nch = static_cast<int>((a->V + L.chunk - 1) / L.chunk);
  L.schunk = kSampleChunk;
  L.nchs = static_cast<int>((a->V + kSampleChunk - 1) / kSampleChunk);

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
  if (a->Dmax > 256 || a->NB > 256) return SSD_ERR_UNSUPPORTED;
  if (a->chain_blk < -1 || a->chain_blk >= a->NB) return SSD_ERR_INVALID;
  if (static_cast<long long>(a->NB) * a->Dmax > kMaxSlots) return SSD_ERR_UNSUPPORTED;
  const long long nrd = 1LL + static_cast<long long>(a->NB) * a->Dmax + (a->chain_blk >= 0 ? a->K : 0);
  if (nrd > kMaxRows) return SSD_ERR_UNSUPPORTED;
  {
    const long long chunk = static_cast<long long>(kVec) * kVocabThreads * (a->kind == SSD_LOGITS_BF16 ? 8 : 4);
    if (((a->V + chunk - 1) / chunk) * nrd * a->B >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  }
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

// resident CTAs of the stats kernel on the whole device (persistent grid)
static long long stats_grid_cap(bool bf16) {
  static long long cap[2] = {0, 0};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  long long& c = cap[bf16 ? 1 : 0];
  if (c == 0) {
    int dev = 0, sms = 152, per = 1;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (bf16) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_vocab_stats<true>, kVocabThreads, 0);
    else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_vocab_stats<false>, kVocabThreads, 0);
    c = static_cast<long long>(sms) * (per > 0 ? per : 1);
  }
  return c;
}

int accept_launch(const AcceptParams& p, cudaStream_t s) {
  const unsigned by = static_cast<unsigned>(p.B < 65535 ? p.B : 65535);
  cudaError_t e;
  {
    // statistics of every needed row; the last CTA of each sequence runs the select
    const long long ntask = static_cast<long long>(p.nch) * p.NRD * p.B;
    const long long cap = stats_grid_cap(p.bf16 != 0);
    const dim3 g1(static_cast<unsigned>(ntask < cap ? ntask : cap));
    KernelTimer t(SSD_KERNEL_VOCAB_STATS, s);
    e = p.bf16 ? launch_pdl(k_vocab_stats<true>, g1, dim3(kVocabThreads), 0, s, p)
               : launch_pdl(k_vocab_stats<false>, g1, dim3(kVocabThreads), 0, s, p);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
  }
  {
    KernelTimer t(SSD_KERNEL_ACCEPT_SELECT, s);
    const unsigned gb = static_cast<unsigned>(p.B < 1048576 ? p.B : 1048576);
    e = launch_pdl(k_accept_select, dim3(gb), dim3(kSelectThreads), 0, s, p);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
  }
  int n = 2;
  if (p.sample) {
    const dim3 g3(static_cast<unsigned>(p.nchs), by);
    KernelTimer t(SSD_KERNEL_SAMPLE_FINAL, s);
    e = launch_pdl(k_sample_final, g3, dim3(kVocabThreads), 0, s, p);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    ++n;
  }
  if (p.probs_out != nullptr) {
    const dim3 g4(static_cast<unsigned>(p.nch * p.NR), by);
    e = launch_pdl(k_probs_out, g4, dim3(kVocabThreads), 0, s, p);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
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

// ------------------------------------------------------------------ no-allocation variant
// Scratch for ssd_accept_static: a fixed array in device memory that exists on
// every GPU where this library's device code is loaded, for the life of the
// process. Host code must not use the symbol itself as a device address (it is
// a host-side stand-in); the real address is fetched once per device below.
namespace ssd {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB
static __device__ __align__(256) unsigned char g_accept_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up on the
// first call for that device (the lookup loads the module there if needed).
static int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) return SSD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SSD_OK;
}

}  // namespace ssd

extern "C" int ssd_accept_static(const ssd_accept_args* a, void* stream) {
  const int st = accept_validate(a);
  if (st != SSD_OK) return st;
  if (a->B == 0) return SSD_OK;
  const AcceptLayout L = accept_layout(a);
  if (L.total > kStaticScratchBytes) return SSD_ERR_WORKSPACE;   // batch too large for the fixed scratch
  void* ws = nullptr;
  const int rc = static_scratch(&ws);
  if (rc != SSD_OK) return rc;
  // Nothing in the scratch has to start at zero: the select kernel sets every
  // sampler completion counter before the sampler reads it.
  const AcceptParams p = accept_params(a, L, static_cast<char*>(ws));
  return accept_launch(p, static_cast<cudaStream_t>(stream));
}
