// Probe gate, kappa-gram check and recency-ranked retrieval.
//
// SwitchSD page, "어떻게 동작하나": the probe is a bias-free linear projection
// p = sigma(w^T h) of a mid-layer hidden state. "무엇과 다른가": the copy path
// opens only when the score is at least tau AND the kappa-gram (kappa = 5)
// ending at the current token occurred earlier in the context; then up to W
// continuations of length D are taken, most recent first.
//
// One CTA per sequence. The context is scanned from its end in chunks staged
// in shared memory with coalesced loads; match ends are ranked by a block-wide
// ballot so that the W largest ends come out in descending order and the scan
// stops as soon as W are known.
#include <math.h>

#include "ssd_common.cuh"

namespace ssd {

constexpr int kGateThreads = 256;
constexpr int kChunk = 4096;     // match ends examined per staged chunk
constexpr int kMaxKappa = 64;
constexpr int kMaxW = 64;

constexpr int kPerThread = 16;           // positions examined per thread per chunk (kChunk / kGateThreads)
constexpr int kStageLoads = (kChunk + kMaxKappa + kGateThreads - 1) / kGateThreads;

struct ScanSmem {
  int tile[kChunk + kMaxKappa];
  int g[kMaxKappa];
  int warp_val[kGateThreads / 32];
  int cnt[kPerThread][kGateThreads / 32];  // matches per (round, warp) of one chunk
  int ends[kMaxW];
  int nfound;
  long long warp_sum[kGateThreads / 32];
};

// Stage ctx[j_lo-kappa+1 .. j_hi] into shared memory: every load of the chunk is
// issued before the first store, so the chunk costs one memory latency.
__device__ __forceinline__ void stage_chunk(ScanSmem& s, const int32_t* row, int j_lo, int j_hi, int kappa) {
  const int base = j_lo - kappa + 1;
  const int cnt = j_hi - base + 1;
  int v[kStageLoads];
#pragma unroll
  for (int u = 0; u < kStageLoads; ++u) {
    const int i = threadIdx.x + u * kGateThreads;
    v[u] = i < cnt ? __ldg(row + base + i) : 0;
  }
#pragma unroll
  for (int u = 0; u < kStageLoads; ++u) {
    const int i = threadIdx.x + u * kGateThreads;
    if (i < cnt) s.tile[i] = v[u];
  }
}

__device__ __forceinline__ bool match_at(const ScanSmem& s, int j, int j_lo, int kappa) {
  // tile index of ctx[j - kappa + 1] is (j - kappa + 1) - (j_lo - kappa + 1) = j - j_lo
  const int* t = s.tile + (j - j_lo);
  bool ok = true;
  for (int i = 0; i < kappa; ++i) ok &= (t[i] == s.g[i]);
  return ok;
}

// Bit u of the result: position j_hi - (u * kGateThreads + threadIdx.x) is a match end.
__device__ __forceinline__ unsigned match_mask(const ScanSmem& s, int j_lo, int j_hi, int kappa) {
  unsigned mask = 0;
#pragma unroll
  for (int u = 0; u < kPerThread; ++u) {
    const int j = j_hi - (u * kGateThreads + static_cast<int>(threadIdx.x));
    if (j >= j_lo && match_at(s, j, j_lo, kappa)) mask |= 1u << u;
  }
  return mask;
}

__global__ void __launch_bounds__(kGateThreads)
k_gate_match(const int32_t* __restrict__ ctx, int64_t stride, const int32_t* __restrict__ ctx_len,
             const void* __restrict__ h, int h_bf16, int64_t h_stride, const float* __restrict__ w, int d,
             int thr_mode, long long thr, int kappa,
             float* __restrict__ score, int32_t* __restrict__ gate, int32_t* __restrict__ last,
             int32_t* __restrict__ probe_on) {
  __shared__ ScanSmem s;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  // ---- probe: exact products, fixed point 2^-32, integer sum (8 loads in flight per thread)
  long long acc = 0;
  const uint16_t* hb = static_cast<const uint16_t*>(h) + b * h_stride;
  const float* hf = static_cast<const float*>(h) + b * h_stride;
  for (int base = 0; base < d; base += kGateThreads * 8) {
    float hv[8], wv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = base + k * kGateThreads + tid;
      hv[k] = 0.f;
      wv[k] = 0.f;
      if (i < d) {
        hv[k] = h_bf16 ? bf16_to_f32(__ldg(hb + i)) : __ldg(hf + i);
        wv[k] = __ldg(w + i);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const double p = static_cast<double>(hv[k]) * static_cast<double>(wv[k]);
      acc += __double2ll_rz(p * 4294967296.0);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) s.warp_sum[wid] = acc;

  // ---- kappa-gram: largest earlier end j
  const int n = ctx_len[b];
  const int32_t* row = ctx + b * stride;
  if (tid < kappa && n >= kappa) s.g[tid] = row[n - kappa + tid];
  __syncthreads();

  int found = -1;
  if (n >= kappa + 1) {
    const int j_min = kappa - 1;
    for (int j_hi = n - 2; j_hi >= j_min && found < 0;) {
      const int j_lo = max(j_min, j_hi - kChunk + 1);
      stage_chunk(s, row, j_lo, j_hi, kappa);
      __syncthreads();
      const unsigned mask = match_mask(s, j_lo, j_hi, kappa);
      // lowest set bit = largest j of this thread
      int best = mask ? j_hi - ((__ffs(mask) - 1) * kGateThreads + tid) : -1;
      best = __reduce_max_sync(0xffffffffu, best);
      if (lane == 0) s.warp_val[wid] = best;
      __syncthreads();
      int m = -1;
#pragma unroll
      for (int i = 0; i < kGateThreads / 32; ++i) m = max(m, s.warp_val[i]);
      found = m;
      __syncthreads();
      j_hi = j_lo - 1;
    }
  }

  if (tid == 0) {
    long long S = 0;
#pragma unroll
    for (int i = 0; i < kGateThreads / 32; ++i) S += s.warp_sum[i];
    bool on = thr_mode == 1 ? true : thr_mode == 2 ? false : (S >= thr);
    const double x = static_cast<double>(S) * 2.3283064365386962890625e-10;  // 2^-32
    score[b] = static_cast<float>(1.0 / (1.0 + exp(-x)));
    last[b] = found;
    gate[b] = (on && found >= 0) ? 1 : 0;
    if (probe_on != nullptr) probe_on[b] = on ? 1 : 0;
  }
}

__global__ void __launch_bounds__(kGateThreads)
k_retrieve(const int32_t* __restrict__ ctx, int64_t stride, const int32_t* __restrict__ ctx_len,
           const int32_t* __restrict__ gate, const int32_t* __restrict__ last, int kappa, int W, int D,
           int K, int chain_policy, const int32_t* __restrict__ chain_tok, int NB, int Dmax,
           int32_t* __restrict__ blk_tok, int32_t* __restrict__ blk_len, int32_t* __restrict__ n_cand) {
  __shared__ ScanSmem s;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = ctx_len[b];
  const int32_t* row = ctx + b * stride;
  const bool on = gate[b] != 0;

  if (tid == 0) s.nfound = 0;
  if (tid < kappa && n >= kappa) s.g[tid] = row[n - kappa + tid];
  __syncthreads();

  int j_start = n - 2;
  if (last != nullptr) j_start = min(j_start, static_cast<int>(last[b]));   // -1: nothing to find
  if (on && n >= kappa + 1) {
    const int j_min = kappa - 1;
    for (int j_hi = j_start; j_hi >= j_min;) {
      const int j_lo = max(j_min, j_hi - kChunk + 1);
      stage_chunk(s, row, j_lo, j_hi, kappa);
      __syncthreads();
      // rank every match of the chunk in descending j order: position
      // j_hi - (u * 256 + tid) precedes every (u', tid') with a larger u'*256+tid'
      const unsigned mask = match_mask(s, j_lo, j_hi, kappa);
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const unsigned bal = __ballot_sync(0xffffffffu, (mask >> u) & 1u);
        if (lane == 0) s.cnt[u][wid] = __popc(bal);
      }
      __syncthreads();
      if (wid == 0) {
        // exclusive prefix over the 128 (round, warp) counts, round-major, offset by
        // the matches of earlier chunks
        constexpr int nc = kPerThread * (kGateThreads / 32);
        constexpr int per = nc / 32;
        int* flat = &s.cnt[0][0];
        int v[per];
        int local = 0;
#pragma unroll
        for (int q = 0; q < per; ++q) {
          v[q] = flat[lane * per + q];
          local += v[q];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int before = s.nfound;
        int run = before + incl - local;
#pragma unroll
        for (int q = 0; q < per; ++q) {
          flat[lane * per + q] = run;
          run += v[q];
        }
        __syncwarp();
        if (lane == 31) s.warp_val[0] = before + incl;   // matches found so far
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const bool m = (mask >> u) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (m) {
          const int rank = s.cnt[u][wid] + __popc(bal & ((1u << lane) - 1u));
          if (rank < W) s.ends[rank] = j_hi - (u * kGateThreads + tid);
        }
      }
      __syncthreads();
      if (tid == 0) s.nfound = s.warp_val[0];
      __syncthreads();
      if (s.nfound >= W) break;
      j_hi = j_lo - 1;
    }
  }
  __syncthreads();
  const int nf = on ? min(s.nfound, W) : 0;
  const bool chain_on = chain_policy == SSD_CHAIN_ALWAYS || (chain_policy == SSD_CHAIN_WHEN_GATE_OFF && !on);

  // outputs: every slot of every block
  int32_t* bt = blk_tok + static_cast<int64_t>(b) * NB * Dmax;
  for (int i = tid; i < NB * Dmax; i += kGateThreads) {
    const int k = i / Dmax, pos = i % Dmax;
    int v = -1;
    if (k < W) {
      if (k < nf) {
        const int j = s.ends[k];
        const int len = min(D, n - 1 - j);
        if (pos < len) v = __ldg(row + j + 1 + pos);
      }
    } else if (chain_on && pos < K) {
      v = __ldg(chain_tok + static_cast<int64_t>(b) * K + pos);
    }
    bt[i] = v;
  }
  for (int k = tid; k < NB; k += kGateThreads) {
    int len = 0;
    if (k < W) {
      if (k < nf) len = min(D, n - 1 - s.ends[k]);
    } else if (chain_on) {
      len = K;
    }
    blk_len[static_cast<int64_t>(b) * NB + k] = len;
  }
  if (tid == 0) n_cand[b] = nf;
}

}  // namespace ssd

using namespace ssd;

extern "C" int ssd_gate_match(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                              const void* h, int h_dtype, int64_t h_stride, const float* w, int d,
                              float tau, int kappa, float* score, int32_t* gate,
                              int32_t* last_match_end, int32_t* probe_on, void* stream) {
  if (B < 0 || kappa < 1 || kappa > kMaxKappa || d < 1) return SSD_ERR_INVALID;
  if (h_dtype != SSD_F32 && h_dtype != SSD_BF16) return SSD_ERR_INVALID;
  if (B == 0) return SSD_OK;
  if (!ctx || !ctx_len || !h || !w || !score || !gate || !last_match_end) return SSD_ERR_INVALID;
  if (ctx_stride < 1 || h_stride < d) return SSD_ERR_INVALID;
  if (ctx_stride > INT32_MAX) return SSD_ERR_UNSUPPORTED;
  int thr_mode = 0;
  long long thr = 0;
  const double t = static_cast<double>(tau);
  if (!(t > 0.0)) {
    thr_mode = 1;                      // sigma(s) >= tau for every s
  } else if (t >= 1.0) {
    thr_mode = 2;                      // sigma(s) < 1 for every finite s
  } else {
    thr = static_cast<long long>(ceil(log(t / (1.0 - t)) * 4294967296.0));
  }
  KernelTimer timer(SSD_KERNEL_GATE_MATCH, static_cast<cudaStream_t>(stream));
  k_gate_match<<<B, kGateThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      ctx, ctx_stride, ctx_len, h, h_dtype == SSD_BF16, h_stride, w, d, thr_mode, thr, kappa, score, gate,
      last_match_end, probe_on);
  count_launch();
  return check_launch();
}

extern "C" int ssd_retrieve(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                            const int32_t* gate, const int32_t* last_match_end, int kappa, int W, int D, int K,
                            int chain_policy, const int32_t* chain_tok, int32_t* blk_tok, int32_t* blk_len,
                            int32_t* n_cand, void* stream) {
  if (B < 0 || kappa < 1 || kappa > kMaxKappa || W < 1 || W > kMaxW || D < 1 || D > 256 || K < 0 || K > 256)
    return SSD_ERR_INVALID;
  if (chain_policy < SSD_CHAIN_NONE || chain_policy > SSD_CHAIN_ALWAYS) return SSD_ERR_INVALID;
  if (chain_policy != SSD_CHAIN_NONE && (K < 1 || chain_tok == nullptr)) return SSD_ERR_INVALID;
  if (B == 0) return SSD_OK;
  if (!ctx || !ctx_len || !gate || !blk_tok || !blk_len || !n_cand) return SSD_ERR_INVALID;
  if (ctx_stride < 1) return SSD_ERR_INVALID;
  if (ctx_stride > INT32_MAX) return SSD_ERR_UNSUPPORTED;
  const int NB = W + (chain_policy != SSD_CHAIN_NONE ? 1 : 0);
  const int Dmax = chain_policy != SSD_CHAIN_NONE ? (D > K ? D : K) : D;
  KernelTimer timer(SSD_KERNEL_RETRIEVE, static_cast<cudaStream_t>(stream));
  k_retrieve<<<B, kGateThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      ctx, ctx_stride, ctx_len, gate, last_match_end, kappa, W, D, K, chain_policy, chain_tok, NB, Dmax, blk_tok,
      blk_len, n_cand);
  count_launch();
  return check_launch();
}
