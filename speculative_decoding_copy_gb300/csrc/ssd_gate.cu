// Probe gate, kappa-gram check and recency-ranked retrieval.
//
// SwitchSD page, "어떻게 동작하나": the probe is a bias-free linear projection
// p = sigma(w^T h) of a mid-layer hidden state. "무엇과 다른가": the copy path
// opens only when the score is at least tau AND the kappa-gram (kappa = 5)
// ending at the current token occurred earlier in the context; then up to W
// continuations of length D are taken, most recent first.
//
// One kernel, k_front<GATE, RETRIEVE>, one CTA of 512 threads per sequence,
// serves the three entry points (gate only, retrieval only, both fused):
//   1. ctx_len and the first pass of the probe operands (h, w) are loaded;
//   2. the loads of the first context chunk (ending at the current token,
//      extended by D positions so that continuations come from shared memory)
//      are issued as soon as ctx_len is in, before the probe arithmetic;
//   3. the probe sum in exact integer arithmetic (no fp64: the product of two
//      fp32 significands is formed as a 64-bit integer and shifted into the
//      2^-32 fixed point, identical to the exact real product truncated);
//   4. each thread tests 8 consecutive match ends; one block scan of the
//      per-thread counts ranks the matches in descending order; the
//      continuations of the W most recent are copied from the tile by all
//      threads; further chunks are staged only if fewer than W were found;
//   5. one warp sums the probe partials and takes the gate decision.
#include <math.h>

#include "ssd_common.cuh"

namespace ssd {

constexpr int kFrontThreads = 512;
constexpr int kWarps = kFrontThreads / 32;
constexpr int kPer = 8;                      // match ends per thread per chunk (contiguous, descending)
constexpr int kChunk = kFrontThreads * kPer; // match ends examined per staged chunk
constexpr int kMaxKappa = 64;
constexpr int kMaxW = 64;
constexpr int kMaxD = 256;
constexpr int kTile = kChunk + kMaxKappa + kMaxD;
constexpr int kStageLoads = (kTile + kFrontThreads - 1) / kFrontThreads;
constexpr int kProbePer = 8;                 // probe elements per thread per pass

struct FrontSmem {
  int tile[kTile];                           // ctx[base .. base + cnt)
  int g[kMaxKappa];                          // the final kappa-gram
  int ends[kMaxW];                           // match ends, most recent first
  int warp_cnt[kWarps];                      // matches per warp in the current chunk
  long long warp_sum[kWarps];                // probe partial sums
  int nfound;
  int on;
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
__global__ void __launch_bounds__(kFrontThreads, 1)
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
  const uint16_t* hb = static_cast<const uint16_t*>(h) + b * h_stride;
  const float* hf = static_cast<const float*>(h) + b * h_stride;

  // ---- 1. loads that do not depend on the context length: ctx_len, the first probe pass
  int n = __ldg(ctx_len + b);
  if (!in_range(n, stride + 1, nullptr, 200)) n = 0;          // a length past the row: nothing is read
  float hv[kProbePer], wv[kProbePer];
  if (GATE) {
#pragma unroll
    for (int k = 0; k < kProbePer; ++k) {
      const int i = tid * kProbePer + k;
      hv[k] = 0.f;
      wv[k] = 0.f;
      if (i < d) {
        hv[k] = h_bf16 ? bf16_to_f32(__ldg(hb + i)) : __ldg(hf + i);
        wv[k] = __ldg(w + i);
      }
    }
  }
  bool on = true;
  if (RETRIEVE && !GATE) on = __ldg(gate + b) != 0;
  const int want = RETRIEVE ? W : 1;
  bool scan = n >= kappa + 1;
  if (RETRIEVE && !GATE) scan = scan && on;

  // ---- 2. the first chunk of the context (ending at the current token): its loads
  // are in flight while the probe sum is formed. A chunk covers match ends
  // [j_lo, j_hi]; its tile adds the kappa-1 tokens before j_lo and, for
  // retrieval, the D tokens after j_hi, so continuations come from shared memory.
  const int j_min = kappa - 1;
  int j_hi = n - 2, j_lo = 0, base = 0, cnt = 0;
  int v[kStageLoads];
  auto stage_loads = [&]() {
    j_lo = max(j_min, j_hi - kChunk + 1);
    base = j_lo - kappa + 1;
    const int top = min(n - 1, j_hi + (RETRIEVE ? D : 0) + 1);
    cnt = top - base + 1;
#pragma unroll
    for (int u = 0; u < kStageLoads; ++u) {
      const int i = tid + u * kFrontThreads;
      v[u] = i < cnt ? __ldg(row + base + i) : 0;
    }
  };
  if (scan) stage_loads();

  // ---- 3. the probe sum in exact integer fixed point (2^-32)
  if (GATE) {
    long long acc = 0;
#pragma unroll
    for (int k = 0; k < kProbePer; ++k) acc += fixed_prod32(hv[k], wv[k]);
    for (int i0 = kFrontThreads * kProbePer; i0 < d; i0 += kFrontThreads * kProbePer) {
#pragma unroll
      for (int k = 0; k < kProbePer; ++k) {
        const int i = i0 + tid * kProbePer + k;
        if (i < d) acc += fixed_prod32(h_bf16 ? bf16_to_f32(__ldg(hb + i)) : __ldg(hf + i), __ldg(w + i));
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) s.warp_sum[wid] = acc;
  }
  if (tid == 0) s.nfound = 0;

  // ---- 4. scan chunks from the end until `want` match ends are known
  if (scan) {
    for (;;) {
#pragma unroll
      for (int u = 0; u < kStageLoads; ++u) {
        const int i = tid + u * kFrontThreads;
        if (i < cnt) s.tile[i] = v[u];
      }
      __syncthreads();
      if (j_hi == n - 2) {   // the final kappa-gram ctx[n-kappa .. n-1] lies in the first chunk's tile
        if (tid < kappa && in_range(n - kappa + tid - base, cnt, nullptr, 201)) s.g[tid] = s.tile[n - kappa + tid - base];
        __syncthreads();
      }
      const int before = s.nfound;
      // this thread's match ends j = j_hi - (tid*kPer + u), u = 0.. (descending)
      unsigned mask = 0;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int j = j_hi - (tid * kPer + u);
        if (j >= j_lo) {
          const int* t = s.tile + (j - kappa + 1 - base);
          bool ok = true;
          for (int i = 0; i < kappa && ok; ++i) ok = t[i] == s.g[i];
          if (ok) mask |= 1u << u;
        }
      }
      // rank of a match = matches at larger j: in earlier threads, then at lower u here
      const int c = __popc(mask);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) s.warp_cnt[wid] = incl;
      __syncthreads();
      int woff = 0, total = 0;
#pragma unroll
      for (int q = 0; q < kWarps; ++q) {
        const int x = s.warp_cnt[q];
        woff += q < wid ? x : 0;
        total += x;
      }
      int rank = before + woff + incl - c;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if ((mask >> u) & 1u) {
          if (rank < want) s.ends[rank] = j_hi - (tid * kPer + u);
          ++rank;
        }
      }
      __syncthreads();
      // continuation tokens of the ends found in this chunk, straight from the tile
      const int r_lo = before, r_hi = min(want, before + total);
      if (RETRIEVE && blk_tok != nullptr && r_hi > r_lo) {
        for (int idx = tid; idx < (r_hi - r_lo) * D; idx += kFrontThreads) {
          const int rr = r_lo + idx / D, q = idx - (idx / D) * D;
          const int j = s.ends[rr];
          if (q < min(D, n - 1 - j) && in_range(j + 1 + q - base, cnt, nullptr, 202) &&
              in_range(rr * Dmax + q, static_cast<long long>(NB) * Dmax, nullptr, 203))
            blk_tok[(static_cast<int64_t>(b) * NB + rr) * Dmax + q] = s.tile[j + 1 + q - base];
        }
      }
      const bool done = before + total >= want || j_lo == j_min;
      __syncthreads();                               // the tile, ends and count are no longer read
      if (tid == 0) s.nfound = before + total;
      if (done) break;
      j_hi = j_lo - 1;
      stage_loads();
    }
  }
  __syncthreads();
  const int nfound = s.nfound;
  const int first = nfound > 0 ? s.ends[0] : -1;

  // ---- 5. gate decision: one warp sums the probe partials
  if (GATE) {
    if (wid == 0) {
      long long S = lane < kWarps ? s.warp_sum[lane] : 0;
      S = warp_sum(S);
      if (lane == 0) {
        const bool pon = thr_mode == 1 ? true : thr_mode == 2 ? false : (S >= thr);
        const float x = static_cast<float>(S) * 2.3283064365386962890625e-10f;   // 2^-32
        score[b] = 1.f / (1.f + expf(-x));
        last[b] = first;
        gate[b] = (pon && first >= 0) ? 1 : 0;
        if (probe_on != nullptr) probe_on[b] = pon ? 1 : 0;
        s.on = (pon && first >= 0) ? 1 : 0;
      }
    }
    __syncthreads();
    on = s.on != 0;
  }

  // ---- 6. retrieval outputs: lengths, padding, chain block
  if (RETRIEVE) {
    const int nf = on ? min(nfound, W) : 0;
    const bool chain_on = chain_policy == SSD_CHAIN_ALWAYS || (chain_policy == SSD_CHAIN_WHEN_GATE_OFF && !on);
    int32_t* bt = blk_tok + static_cast<int64_t>(b) * NB * Dmax;
    for (int i = tid; i < NB * Dmax; i += kFrontThreads) {
      const int k = i / Dmax, pos = i - (i / Dmax) * Dmax;
      if (k < W) {
        // copy blocks were written during the scan (only when the gate is on)
        const int len = k < nf ? min(D, n - 1 - s.ends[k]) : 0;
        if (pos >= len) bt[i] = -1;
      } else {
        bt[i] = (chain_on && pos < K) ? __ldg(chain_tok + static_cast<int64_t>(b) * K + pos) : -1;
      }
    }
    for (int k = tid; k < NB; k += kFrontThreads) {
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
  k_front<true, false><<<B, kFrontThreads, 0, s>>>(ctx, ctx_stride, ctx_len, h, h_dtype == SSD_BF16, h_stride, w, d,
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
  k_front<false, true><<<B, kFrontThreads, 0, s>>>(ctx, ctx_stride, ctx_len, nullptr, 0, 0, nullptr, 0, 0, 0, kappa, W,
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
  k_front<true, true><<<B, kFrontThreads, 0, s>>>(ctx, ctx_stride, ctx_len, h, h_dtype == SSD_BF16, h_stride, w, d,
                                                 t.mode, t.thr, kappa, W, D, K, chain_policy, chain_tok, NB, Dmax,
                                                 score, gate, last_match_end, probe_on, blk_tok, blk_len, n_cand);
  count_launch();
  return check_launch();
}
