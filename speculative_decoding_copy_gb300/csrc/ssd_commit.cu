// After the step: commit of the accepted candidates' keys and values to the prefix
// cache, and the copy-attempt / speculation-tax counts.
//
// Speculative Decoding 해부 page, §6 "KV 캐시 롤백(Rollback) 및 페이징 메모리 오버헤드
// 관리": the target holds the candidates' K/V to verify them, and what follows the first
// rejection must be released. The candidates' K/V sit beside the cache here, so the
// accepted ones are appended (the rejected ones never enter it).
//
// k_commit_kv: one CTA per sequence; after griddepcontrol.wait (best_blk and n_out come
// from the acceptance, the kernel before it) every thread copies 16-byte words (or
// elements, for unaligned rows) of the a accepted rows of every kv head, then thread 0
// advances prefix_len once every copy of the CTA has been issued.
#include "ssd_common.cuh"

namespace ssd {

constexpr int kCommitThreads = 256;

template <bool VEC>
__global__ void __launch_bounds__(kCommitThreads)
k_commit_kv(ssd_commit_args a, WsHeader* hdr) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x;
  const int k = a.best_blk[b];
  const int n = k >= 0 ? a.n_out[b] - 1 : 0;
  if (n <= 0) return;
  const int64_t P = a.prefix_len[b];
  if (k >= a.NB || n > a.Dmax || P < 0 || P + n > a.P_max) {   // no room, or inputs not from this shape
    if (threadIdx.x == 0) record_error(hdr, SSD_ERR_DEVICE, 300);
    return;
  }
  const int es = a.dtype == SSD_BF16 ? 2 : 4;
  const int64_t row_bytes = static_cast<int64_t>(a.dh) * es;
  const int NT = a.NB * a.Dmax;
  const int64_t rows = static_cast<int64_t>(n) * a.Hkv;       // (token, kv head) rows of K, and as many of V
  if (VEC) {
    const int wpr = static_cast<int>(row_bytes / 16);         // 16-byte words per row
    const int64_t words = rows * wpr;
    for (int64_t w = threadIdx.x; w < 2 * words; w += kCommitThreads) {
      const bool is_v = w >= words;
      const int64_t ww = is_v ? w - words : w;
      const int64_t r = ww / wpr;
      const int c = static_cast<int>(ww - r * wpr);
      const int i = static_cast<int>(r / a.Hkv), h = static_cast<int>(r - static_cast<int64_t>(i) * a.Hkv);
      const int64_t src_row = (static_cast<int64_t>(b) * NT + k * a.Dmax + i) * a.Hkv + h;
      const int64_t dst_row = (static_cast<int64_t>(b) * a.Hkv + h) * a.P_max + P + i;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(is_v ? a.v_cand : a.k_cand) +
                                                        src_row * row_bytes);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(is_v ? a.v_cache : a.k_cache) + dst_row * row_bytes);
      dst[c] = src[c];
    }
  } else {
    const int64_t elems = rows * a.dh;
    for (int64_t e = threadIdx.x; e < 2 * elems; e += kCommitThreads) {
      const bool is_v = e >= elems;
      const int64_t ee = is_v ? e - elems : e;
      const int64_t r = ee / a.dh;
      const int c = static_cast<int>(ee - r * a.dh);
      const int i = static_cast<int>(r / a.Hkv), h = static_cast<int>(r - static_cast<int64_t>(i) * a.Hkv);
      const int64_t src_row = (static_cast<int64_t>(b) * NT + k * a.Dmax + i) * a.Hkv + h;
      const int64_t dst_row = (static_cast<int64_t>(b) * a.Hkv + h) * a.P_max + P + i;
      const char* src = static_cast<const char*>(is_v ? a.v_cand : a.k_cand) + (src_row * a.dh + c) * es;
      char* dst = static_cast<char*>(is_v ? a.v_cache : a.k_cache) + (dst_row * a.dh + c) * es;
      if (es == 2)
        *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(src);
      else
        *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) a.prefix_len[b] = static_cast<int32_t>(P + n);
}

}  // namespace ssd

extern "C" int ssd_commit_kv(const ssd_commit_args* a, void* ws, size_t ws_bytes, void* stream) {
  using namespace ssd;
  if (a == nullptr) return SSD_ERR_INVALID;
  if (a->dtype != SSD_F32 && a->dtype != SSD_BF16) return SSD_ERR_INVALID;
  if (a->B < 0 || a->NB < 1 || a->Dmax < 1 || a->Hkv < 1 || a->dh < 1 || a->P_max < 0) return SSD_ERR_INVALID;
  if (a->B == 0) return SSD_OK;
  if (!a->k_cache || !a->v_cache || !a->k_cand || !a->v_cand || !a->prefix_len || !a->best_blk || !a->n_out)
    return SSD_ERR_INVALID;
  if (static_cast<long long>(a->B) * a->NB * a->Dmax * a->Hkv >= (1LL << 40)) return SSD_ERR_UNSUPPORTED;
  if (a->B > 2147483647) return SSD_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < sizeof(WsHeader)) return SSD_ERR_WORKSPACE;
  const int es = a->dtype == SSD_BF16 ? 2 : 4;
  const bool vec = (static_cast<long long>(a->dh) * es) % 16 == 0 && aligned(a->k_cache, 16) && aligned(a->v_cache, 16) &&
                   aligned(a->k_cand, 16) && aligned(a->v_cand, 16);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(ws);
  const cudaError_t e = vec ? launch_pdl(k_commit_kv<true>, dim3(a->B), dim3(kCommitThreads), 0, s, *a, hdr)
                            : launch_pdl(k_commit_kv<false>, dim3(a->B), dim3(kCommitThreads), 0, s, *a, hdr);
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  count_launch();
  return check_launch();
}

namespace ssd {
constexpr int kStatThreads = 256;

// one CTA: block sums of the four counts, added to the running totals
__global__ void __launch_bounds__(kStatThreads)
k_copy_stats(const int32_t* __restrict__ gate, const int32_t* __restrict__ n_cand, const int32_t* __restrict__ acc_len,
             int B, int NB, int W, unsigned long long* counts) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ unsigned long long part[3][kStatThreads / 32];
  unsigned long long c[3] = {0, 0, 0};
  for (int b = threadIdx.x; b < B; b += kStatThreads) {
    if (gate[b] == 0 || n_cand[b] <= 0) continue;
    int run = 0;
    for (int k = 0; k < W; ++k) run = max(run, acc_len[static_cast<int64_t>(b) * NB + k]);
    c[0] += 1;
    c[1] += run == 0 ? 1 : 0;
    c[2] += static_cast<unsigned long long>(run);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c[i] += __shfl_xor_sync(0xffffffffu, c[i], o);
    if (lane == 0) part[i][wid] = c[i];
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    unsigned long long t = 0;
    for (int w = 0; w < kStatThreads / 32; ++w) t += part[threadIdx.x][w];
    atomicAdd(counts + threadIdx.x, t);
  }
  if (threadIdx.x == 3) atomicAdd(counts + 3, static_cast<unsigned long long>(B));
}
}  // namespace ssd

extern "C" int ssd_copy_stats(const int32_t* gate, const int32_t* n_cand, const int32_t* acc_len, int B, int NB, int W,
                              int64_t* counts, void* stream) {
  using namespace ssd;
  if (B < 0 || W < 0 || NB < W || NB < 1) return SSD_ERR_INVALID;
  if (B == 0) return SSD_OK;
  if (!gate || !n_cand || !acc_len || !counts || !aligned(counts, 8)) return SSD_ERR_INVALID;
  if (launch_pdl(k_copy_stats, dim3(1), dim3(kStatThreads), 0, static_cast<cudaStream_t>(stream), gate, n_cand, acc_len,
                 B, NB, W, reinterpret_cast<unsigned long long*>(counts)) != cudaSuccess)
    return SSD_ERR_CUDA;
  count_launch();
  return check_launch();
}
