// Probe gate, kappa-gram check and recency-ranked retrieval.
//
// SwitchSD page, "어떻게 동작하나": the probe is a bias-free linear projection
// p = sigma(w^T h) of a mid-layer hidden state. "무엇과 다른가": the copy path
// opens only when the score is at least tau AND the kappa-gram (kappa = 5)
// ending at the current token occurred earlier in the context; then up to W
// continuations of length D are taken, most recent first.
//
// One kernel, k_front<GATE, RETRIEVE>, one CTA per sequence, serves the three
// entry points (gate only, retrieval only, both fused). Every global load of a
// phase is issued before its first use:
//   1. ctx_len and the probe operands (h, w) together;
//   2. one staged chunk of the context ending at the current token, extended
//      by D positions so that continuations can be copied from shared memory;
//   3. the probe sum in exact integer arithmetic (no fp64: the product of two
//      fp32 significands is formed as a 64-bit integer and shifted into the
//      2^-32 fixed point, identical to the exact real product truncated);
//   4. match ends ranked in descending order with per-warp ballots and one
//      prefix over the (round, warp) counts; the scan stops once W are known.
#include <math.h>

#include "ssd_common.cuh"

namespace ssd {

constexpr int kGateThreads = 1024;
constexpr int kChunk = 8192;                 // match ends examined per staged chunk
constexpr int kPerThread = kChunk / kGateThreads;
constexpr int kMaxKappa = 64;
constexpr int kMaxW = 64;
constexpr int kMaxD = 256;
constexpr int kTile = kChunk + kMaxKappa + kMaxD;
constexpr int kStageLoads = (kTile + kGateThreads - 1) / kGateThreads;
constexpr int kProbeBatch = 8;               // probe elements per thread in flight

struct FrontSmem {
  int tile[kTile];                           // ctx[base .. base + cnt)
  int cnt[kPerThread][kGateThreads / 32];    // matches per (round, warp), then their prefix
  int g[kMaxKappa];                          // the final kappa-gram
  int ends[kMaxW];
  int nfound;
  int total;
  long long warp_sum[kGateThreads / 32];
};

// trunc(a * b * 2^32) for finite fp32 a, b with |a*b| < 2^31, exactly
__device__ __forceinline__ long long fixed_prod32(float a, float b) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  int ea = static_cast<int>((ua >> 23) & 0xffu), eb = static_cast<int>((ub >> 23) & 0xffu);
  uint32_t ma = ua & 0x7fffffu, mb = ub & 0x7fffffu;
  if (ea == 0) ea = 1; else ma |= 0x800000u;        // subnormals have no implicit bit
  if (eb == 0) eb = 1; else mb |= 0x800000u;
  const uint64_t prod = static_cast<uint64_t>(ma) * mb;   // < 2^48, exact
  // value = prod * 2^(ea - 150 + eb - 150) ; scaled by 2^32
  const int sh = ea + eb - 300 + 32;
  uint64_t mag;
  if (sh >= 0) mag = prod << min(sh, 15);            // |a*b| < 2^31 keeps sh <= 15
  else mag = (-sh >= 64) ? 0 : (prod >> (-sh));
  const bool neg = ((ua ^ ub) >> 31) != 0;
  return neg ? -static_cast<long long>(mag) : static_cast<long long>(mag);
}

template <bool GATE, bool RETRIEVE>
__global__ void __launch_bounds__(kGateThreads, 1)
k_front(const int32_t* __restrict__ ctx, int64_t stride, const int32_t* __restrict__ ctx_len,
        const void* __restrict__ h, int h_bf16, int64_t h_stride, const float* __restrict__ w, int d,
        int thr_mode, long long thr, int kappa, int W, int D, int K, int chain_policy,
        const int32_t* __restrict__ chain_tok, int NB, int Dmax,
        float* __restrict__ score, int32_t* __restrict__ gate, int32_t* __restrict__ last,
        int32_t* __restrict__ probe_on, int32_t* __restrict__ blk_tok, int32_t* __restrict__ blk_len,
        int32_t* __restrict__ n_cand) {
  __shared__ FrontSmem s;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // the next kernel may start its launch
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int32_t* row = ctx + b * stride;

  // ---- 1. context length and the probe operands, all loads in flight together
  const int n = __ldg(ctx_len + b);
  long long acc = 0;
  if (GATE) {
    const uint16_t* hb = static_cast<const uint16_t*>(h) + b * h_stride;
    const float* hf = static_cast<const float*>(h) + b * h_stride;
    for (int base = 0; base < d; base += kGateThreads * kProbeBatch) {
      float hv[kProbeBatch], wv[kProbeBatch];
#pragma unroll
      for (int k = 0; k < kProbeBatch; ++k) {
        const int i = base + k * kGateThreads + tid;
        hv[k] = 0.f;
        wv[k] = 0.f;
        if (i < d) {
          hv[k] = h_bf16 ? bf16_to_f32(__ldg(hb + i)) : __ldg(hf + i);
          wv[k] = __ldg(w + i);
        }
      }
#pragma unroll
      for (int k = 0; k < kProbeBatch; ++k) acc += fixed_prod32(hv[k], wv[k]);
    }
    acc = warp_sum(acc);
    if (lane == 0) s.warp_sum[wid] = acc;
  }
  bool on = true;
  if (RETRIEVE && !GATE) on = __ldg(gate + b) != 0;
  if (tid == 0) s.nfound = 0;
  __syncthreads();

  // ---- 2..4. scan for earlier occurrences of the final kappa-gram
  // GATE needs the largest end; RETRIEVE the W largest (only when the gate is on,
  // which for the fused kernel is known once the probe sum is in).
  const int want = RETRIEVE ? W : 1;
  bool scan = n >= kappa + 1;
  if (RETRIEVE && !GATE) scan = scan && on;
  int first = -1;
  if (scan) {
    const int j_min = kappa - 1;
    for (int j_hi = n - 2; j_hi >= j_min;) {
      const int j_lo = max(j_min, j_hi - kChunk + 1);
      // stage ctx[j_lo-kappa+1 .. min(n-1, j_hi+D)] (the final kappa-gram and every
      // continuation of a match in this chunk lie inside)
      const int base = j_lo - kappa + 1;
      const int top = min(n - 1, j_hi + (RETRIEVE ? D : 0) + 1);
      const int cnt = top - base + 1;
      {
        int v[kStageLoads];
#pragma unroll
        for (int u = 0; u < kStageLoads; ++u) {
          const int i = tid + u * kGateThreads;
          v[u] = i < cnt ? __ldg(row + base + i) : 0;
        }
        __syncthreads();   // the previous chunk's tile is no longer read
#pragma unroll
        for (int u = 0; u < kStageLoads; ++u) {
          const int i = tid + u * kGateThreads;
          if (i < cnt) s.tile[i] = v[u];
        }
      }
      __syncthreads();
      // the final kappa-gram ctx[n-kappa .. n-1] lies in the first chunk's tile
      if (j_hi == n - 2) {
        if (tid < kappa) s.g[tid] = s.tile[n - kappa + tid - base];
        __syncthreads();
      }
      unsigned mask = 0;
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const int j = j_hi - (u * kGateThreads + tid);
        if (j >= j_lo) {
          const int* t = s.tile + (j - kappa + 1 - base);
          bool ok = true;
          for (int i = 0; i < kappa && ok; ++i) ok = t[i] == s.g[i];
          if (ok) mask |= 1u << u;
        }
      }
      // rank: position j_hi - (u*256 + tid) precedes every (u', tid') with a larger u'*256+tid'
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const unsigned bal = __ballot_sync(0xffffffffu, (mask >> u) & 1u);
        if (lane == 0) s.cnt[u][wid] = __popc(bal);
      }
      __syncthreads();
      if (wid == 0) {
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
        if (lane == 31) s.total = before + incl;
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const bool m = (mask >> u) & 1u;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (m) {
          const int rank = s.cnt[u][wid] + __popc(bal & ((1u << lane) - 1u));
          const int j = j_hi - (u * kGateThreads + tid);
          if (rank < want) {
            s.ends[rank] = j;
            if (RETRIEVE && blk_tok != nullptr) {
              // continuation tokens straight from the tile into block `rank`
              const int len = min(D, n - 1 - j);
              int32_t* bt = blk_tok + (static_cast<int64_t>(b) * NB + rank) * Dmax;
              for (int q = 0; q < len; ++q) bt[q] = s.tile[j + 1 + q - base];
            }
          }
        }
      }
      __syncthreads();
      if (tid == 0) s.nfound = s.total;
      __syncthreads();
      if (s.nfound >= want) break;
      j_hi = j_lo - 1;
    }
    first = s.nfound > 0 ? s.ends[0] : -1;
  }

  // ---- gate decision
  if (GATE) {
    __syncthreads();
    long long S = 0;
#pragma unroll
    for (int i = 0; i < kGateThreads / 32; ++i) S += s.warp_sum[i];
    on = thr_mode == 1 ? true : thr_mode == 2 ? false : (S >= thr);
    if (tid == 0) {
      const float x = static_cast<float>(S) * 2.3283064365386962890625e-10f;   // 2^-32
      score[b] = 1.f / (1.f + expf(-x));
      last[b] = first;
      gate[b] = (on && first >= 0) ? 1 : 0;
      if (probe_on != nullptr) probe_on[b] = on ? 1 : 0;
    }
    on = on && first >= 0;
  }

  // ---- retrieval outputs: lengths, padding, chain block
  if (RETRIEVE) {
    const int nf = on ? min(s.nfound, W) : 0;
    const bool chain_on = chain_policy == SSD_CHAIN_ALWAYS || (chain_policy == SSD_CHAIN_WHEN_GATE_OFF && !on);
    int32_t* bt = blk_tok + static_cast<int64_t>(b) * NB * Dmax;
    for (int i = tid; i < NB * Dmax; i += kGateThreads) {
      const int k = i / Dmax, pos = i % Dmax;
      if (k < W) {
        // copy blocks were written during the scan (only when the gate is on)
        const int len = k < nf ? min(D, n - 1 - s.ends[k]) : 0;
        if (pos >= len || k >= nf) bt[i] = -1;
      } else {
        bt[i] = (chain_on && pos < K) ? __ldg(chain_tok + static_cast<int64_t>(b) * K + pos) : -1;
      }
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
}

struct Threshold {
  int mode;
  long long thr;
};

static Threshold probe_threshold(float tau) {
  Threshold t{0, 0};
  const double x = static_cast<double>(tau);
  if (!(x > 0.0)) t.mode = 1;             // sigma(s) >= tau for every s
  else if (x >= 1.0) t.mode = 2;          // sigma(s) < 1 for every finite s
  else t.thr = static_cast<long long>(ceil(log(x / (1.0 - x)) * 4294967296.0));
  return t;
}

}  // namespace ssd

using namespace ssd;

static int check_gate_args(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B, const void* h,
                           int h_dtype, int64_t h_stride, const float* w, int d, int kappa) {
  if (B < 0 || kappa < 1 || kappa > kMaxKappa || d < 1) return SSD_ERR_INVALID;
  if (h_dtype != SSD_F32 && h_dtype != SSD_BF16) return SSD_ERR_INVALID;
  if (B == 0) return SSD_OK;
  if (!ctx || !ctx_len || !h || !w) return SSD_ERR_INVALID;
  if (ctx_stride < 1 || h_stride < d) return SSD_ERR_INVALID;
  if (ctx_stride > INT32_MAX) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

static int check_retrieve_args(int W, int D, int K, int chain_policy, const int32_t* chain_tok, int32_t* blk_tok,
                               int32_t* blk_len, int32_t* n_cand, int B) {
  if (W < 1 || W > kMaxW || D < 1 || D > kMaxD || K < 0 || K > 256) return SSD_ERR_INVALID;
  if (chain_policy < SSD_CHAIN_NONE || chain_policy > SSD_CHAIN_ALWAYS) return SSD_ERR_INVALID;
  if (chain_policy != SSD_CHAIN_NONE && (K < 1 || chain_tok == nullptr)) return SSD_ERR_INVALID;
  if (B > 0 && (!blk_tok || !blk_len || !n_cand)) return SSD_ERR_INVALID;
  return SSD_OK;
}

extern "C" int ssd_gate_match(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                              const void* h, int h_dtype, int64_t h_stride, const float* w, int d,
                              float tau, int kappa, float* score, int32_t* gate,
                              int32_t* last_match_end, int32_t* probe_on, void* stream) {
  int rc = check_gate_args(ctx, ctx_stride, ctx_len, B, h, h_dtype, h_stride, w, d, kappa);
  if (rc != SSD_OK || B == 0) return rc;
  if (!score || !gate || !last_match_end) return SSD_ERR_INVALID;
  const Threshold t = probe_threshold(tau);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  KernelTimer timer(SSD_KERNEL_GATE_MATCH, s);
  k_front<true, false><<<B, kGateThreads, 0, s>>>(ctx, ctx_stride, ctx_len, h, h_dtype == SSD_BF16, h_stride, w, d,
                                                  t.mode, t.thr, kappa, 1, 1, 0, 0, nullptr, 1, 1, score, gate,
                                                  last_match_end, probe_on, nullptr, nullptr, nullptr);
  count_launch();
  return check_launch();
}

extern "C" int ssd_retrieve(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                            const int32_t* gate, const int32_t* last_match_end, int kappa, int W, int D, int K,
                            int chain_policy, const int32_t* chain_tok, int32_t* blk_tok, int32_t* blk_len,
                            int32_t* n_cand, void* stream) {
  (void)last_match_end;   // the scan restarts from the end: the first chunk holds the latest matches
  if (B < 0 || kappa < 1 || kappa > kMaxKappa) return SSD_ERR_INVALID;
  int rc = check_retrieve_args(W, D, K, chain_policy, chain_tok, blk_tok, blk_len, n_cand, B);
  if (rc != SSD_OK || B == 0) return rc;
  if (!ctx || !ctx_len || !gate) return SSD_ERR_INVALID;
  if (ctx_stride < 1) return SSD_ERR_INVALID;
  if (ctx_stride > INT32_MAX) return SSD_ERR_UNSUPPORTED;
  const int NB = W + (chain_policy != SSD_CHAIN_NONE ? 1 : 0);
  const int Dmax = chain_policy != SSD_CHAIN_NONE ? (D > K ? D : K) : D;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  KernelTimer timer(SSD_KERNEL_RETRIEVE, s);
  k_front<false, true><<<B, kGateThreads, 0, s>>>(ctx, ctx_stride, ctx_len, nullptr, 0, 0, nullptr, 0, 0, 0, kappa, W,
                                                  D, K, chain_policy, chain_tok, NB, Dmax, nullptr,
                                                  const_cast<int32_t*>(gate), nullptr, nullptr, blk_tok, blk_len,
                                                  n_cand);
  count_launch();
  return check_launch();
}

extern "C" int ssd_gate_retrieve(const int32_t* ctx, int64_t ctx_stride, const int32_t* ctx_len, int B,
                                 const void* h, int h_dtype, int64_t h_stride, const float* w, int d, float tau,
                                 int kappa, int W, int D, int K, int chain_policy, const int32_t* chain_tok,
                                 float* score, int32_t* gate, int32_t* last_match_end, int32_t* probe_on,
                                 int32_t* blk_tok, int32_t* blk_len, int32_t* n_cand, void* stream) {
  int rc = check_gate_args(ctx, ctx_stride, ctx_len, B, h, h_dtype, h_stride, w, d, kappa);
  if (rc != SSD_OK) return rc;
  rc = check_retrieve_args(W, D, K, chain_policy, chain_tok, blk_tok, blk_len, n_cand, B);
  if (rc != SSD_OK || B == 0) return rc;
  if (!score || !gate || !last_match_end) return SSD_ERR_INVALID;
  const Threshold t = probe_threshold(tau);
  const int NB = W + (chain_policy != SSD_CHAIN_NONE ? 1 : 0);
  const int Dmax = chain_policy != SSD_CHAIN_NONE ? (D > K ? D : K) : D;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  KernelTimer timer(SSD_KERNEL_GATE_MATCH, s);
  k_front<true, true><<<B, kGateThreads, 0, s>>>(ctx, ctx_stride, ctx_len, h, h_dtype == SSD_BF16, h_stride, w, d,
                                                 t.mode, t.thr, kappa, W, D, K, chain_policy, chain_tok, NB, Dmax,
                                                 score, gate, last_match_end, probe_on, blk_tok, blk_len, n_cand);
  count_launch();
  return check_launch();
}
