// Verification attention under the block-triangular mask.
//
// SwitchSD page, "무엇과 다른가": all W candidates are verified in one target
// pass; a candidate token attends to the whole prefix and to the earlier tokens
// of its own candidate, never to another candidate. A chain draft is one block
// under the ordinary causal mask (Speculative Decoding 해부 page, §2 Phase 2).
//
// The work splits into a dense part (every token of a sequence sees the same
// prefix keys, so q-heads of one kv head and all candidate tokens pack into
// the rows of one matrix product against each prefix tile) and a tiny masked
// part (at most Dmax own-block keys per token). Two kernels:
//   prefix partial: split-KV flash pass over the prefix; per (row, split) it
//                   leaves the running max m, sum l and un-normalised o
//                   (log2 units) in the workspace;
//   combine:        one warp per row merges the splits, adds the row's own
//                   block keys, normalises and stores the output.
// bf16 inputs with head dim 128 use the fused tcgen05 kernel (ssd_attn_tc.cu),
// which covers both parts in one launch; the SIMT pair below serves fp32, head
// dim 64 and every other shape.
#include <math.h>

#include "ssd_attn.cuh"

namespace ssd {

std::atomic<uint64_t> g_launches{0};

constexpr int kSimtThreads = 128;
constexpr int kSimtRowsPerWarp = 2;
constexpr int kSimtRows = (kSimtThreads / 32) * kSimtRowsPerWarp;   // 8 packed rows per CTA
constexpr int kKeyTile = 32;

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p, int64_t i) { return __ldg(p + i); }
template <>
__device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t* p, int64_t i) { return bf16_to_f32(__ldg(p + i)); }

template <typename T>
__device__ __forceinline__ void st_elem(T* p, int64_t i, float v);
template <>
__device__ __forceinline__ void st_elem<float>(float* p, int64_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st_elem<uint16_t>(uint16_t* p, int64_t i, float v) { p[i] = f32_to_bf16(v); }

__device__ __forceinline__ bool token_present(const int32_t* blk_len, int b, int NB, int Dmax, int t) {
  const int k = t / Dmax, pos = t % Dmax;
  return pos < blk_len[b * NB + k];
}

// grid (B*Hkv, ceil(NT*G / 8), S), block 128
template <typename T, int DH>
__global__ void __launch_bounds__(kSimtThreads)
k_attn_prefix_simt(AttnParams p) {
  constexpr int EPL = DH / 32;   // output dims per lane
  __shared__ float q_s[kSimtRows][DH];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float k_s[kKeyTile][DH + 1];
  __shared__ float v_s[kKeyTile][DH];

  const int split = blockIdx.z;
  const int bk = blockIdx.x;
  const int b = bk / p.Hkv, kvh = bk % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int NT = p.NB * p.Dmax;
  const int rows_total = NT * G;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int P = p.prefix_len[b];
  if (!in_range(P, p.P_max + 1, p.hdr, 28)) P = 0;       // a prefix longer than the cache
  const int k0 = split * p.chunk;
  const int k1 = min(P, k0 + p.chunk);

  const T* q = static_cast<const T*>(p.q);
  const T* kc = static_cast<const T*>(p.k_cache) + (static_cast<int64_t>(b) * p.Hkv + kvh) * p.P_max * DH;
  const T* vc = static_cast<const T*>(p.v_cache) + (static_cast<int64_t>(b) * p.Hkv + kvh) * p.P_max * DH;

  // stage the CTA's q rows, pre-scaled into log2 units
  const int r_base = blockIdx.y * kSimtRows;
  for (int i = tid; i < kSimtRows * DH; i += kSimtThreads) {
    const int rr = i / DH, e = i % DH;
    const int r = r_base + rr;
    float v = 0.f;
    if (r < rows_total) {
      const int t = r / G, h = kvh * G + r % G;
      v = ld_elem(q, ((static_cast<int64_t>(b) * NT + t) * p.Hq + h) * DH + e) * p.scale_log2;
    }
    q_s[rr][e] = v;
  }

  float m[kSimtRowsPerWarp], l[kSimtRowsPerWarp], o[kSimtRowsPerWarp][EPL];
#pragma unroll
  for (int j = 0; j < kSimtRowsPerWarp; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[j][e] = 0.f;
  }

  for (int kt = k0; kt < k1; kt += kKeyTile) {
    __syncthreads();
    for (int i = tid; i < kKeyTile * DH; i += kSimtThreads) {
      const int kk = i / DH, e = i % DH;
      const int key = kt + kk;
      float kv = 0.f, vv = 0.f;
      if (key < k1) {
        kv = ld_elem(kc, static_cast<int64_t>(key) * DH + e);
        vv = ld_elem(vc, static_cast<int64_t>(key) * DH + e);
      }
      k_s[kk][e] = kv;
      v_s[kk][e] = vv;
    }
    __syncthreads();
    const bool key_ok = (kt + lane) < k1;
#pragma unroll
    for (int j = 0; j < kSimtRowsPerWarp; ++j) {
      const float* qr = q_s[wid * kSimtRowsPerWarp + j];
      float s = 0.f;
#pragma unroll 8
      for (int e = 0; e < DH; ++e) s = fmaf(qr[e], k_s[lane][e], s);
      s = key_ok ? s : -INFINITY;
      const float m_new = fmaxf(m[j], warp_max(s));
      const float corr = exp2f(m[j] - m_new);          // m = -inf -> 0
      const float pj = exp2f(s - m_new);
      l[j] = l[j] * corr + warp_sum(pj);
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[j][e] *= corr;
      for (int kk = 0; kk < kKeyTile; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, pj, kk);
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(pk, v_s[kk][lane + 32 * e], o[j][e]);
      }
      m[j] = m_new;
    }
  }

  // leave (m, l, o) for every packed row of a present token
#pragma unroll
  for (int j = 0; j < kSimtRowsPerWarp; ++j) {
    const int r = r_base + wid * kSimtRowsPerWarp + j;
    if (r >= rows_total) continue;
    const int t = r / G, h = kvh * G + r % G;
    if (!p.all_rows && !token_present(p.blk_len, b, p.NB, p.Dmax, t)) continue;
    const int64_t R = (static_cast<int64_t>(b) * NT + t) * p.Hq + h;
    float* ml = p.ws_ml + (R * p.S + split) * 2;
    float* ow = p.ws_o + (R * p.S + split) * DH;
    if (lane == 0) {
      ml[0] = m[j];
      ml[1] = l[j];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) ow[lane + 32 * e] = o[j][e];
  }
}

// one warp per (b, t, h); grid ceil(B*NT*Hq / 4), block 128
template <typename T, int DH>
__global__ void __launch_bounds__(128)
k_attn_combine(AttnParams p) {
  constexpr int EPL = DH / 32;
  __shared__ float sc_s[4][256];
  asm volatile("griddepcontrol.wait;" ::: "memory");     // partials come from the prefix pass
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int NT = p.NB * p.Dmax;
  const int64_t R = static_cast<int64_t>(blockIdx.x) * 4 + wid;
  if (R >= static_cast<int64_t>(p.B) * NT * p.Hq) return;
  const int h = static_cast<int>(R % p.Hq);
  const int t = static_cast<int>((R / p.Hq) % NT);
  const int b = static_cast<int>(R / (static_cast<int64_t>(p.Hq) * NT));
  if (!p.all_rows && !token_present(p.blk_len, b, p.NB, p.Dmax, t)) return;
  const int G = p.Hq / p.Hkv;
  const int kvh = h / G;
  const int k = t / p.Dmax, pos = t % p.Dmax;

  constexpr int KG = 8;          // own-block keys whose loads are issued together
  const T* q = static_cast<const T*>(p.q) + R * DH;
  const T* kd = static_cast<const T*>(p.k_cand);
  const T* vd = static_cast<const T*>(p.v_cand);
  const int64_t kv_row0 = (static_cast<int64_t>(b) * NT + k * p.Dmax) * p.Hkv + kvh;   // slot k*Dmax, head kvh
  const int64_t kv_step = static_cast<int64_t>(p.Hkv) * DH;                            // next slot
  float qv[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] = ld_elem(q, lane + 32 * e) * p.scale_log2;

  // per-split running max: lane s holds split s
  const float* ml = p.ws_ml + R * p.S * 2;
  float M = -INFINITY;
  for (int s = lane; s < p.S; s += 32) M = fmaxf(M, ml[2 * s]);
  M = warp_max(M);

  // own-block keys: slots k*Dmax .. t, scores in groups of KG
  for (int c0 = 0; c0 <= pos; c0 += KG) {
    float kk[KG][EPL];
#pragma unroll
    for (int g = 0; g < KG; ++g) {
      const int c = c0 + g;
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        kk[g][e] = c <= pos ? ld_elem(kd, (kv_row0 + c * (p.Hkv)) * DH + lane + 32 * e) : 0.f;
    }
    float sc[KG];
#pragma unroll
    for (int g = 0; g < KG; ++g) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) s = fmaf(qv[e], kk[g][e], s);
      sc[g] = s;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int g = 0; g < KG; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], o);
#pragma unroll
    for (int g = 0; g < KG; ++g) {
      if (c0 + g <= pos) {
        if (lane == 0) sc_s[wid][c0 + g] = sc[g];
        M = fmaxf(M, sc[g]);
      }
    }
  }
  __syncwarp();
  (void)kv_step;

  float L = 0.f, O[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) O[e] = 0.f;
  // splits: loads of four splits in flight at a time
  const float* ow = p.ws_o + R * p.S * DH;
  for (int s0 = 0; s0 < p.S; s0 += 4) {
    float ms[4], ls[4], ov[4][EPL];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int s = s0 + g;
      ms[g] = s < p.S ? ml[2 * s] : -INFINITY;
      ls[g] = s < p.S ? ml[2 * s + 1] : 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ov[g][e] = s < p.S ? ow[s * DH + lane + 32 * e] : 0.f;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (ms[g] == -INFINITY) continue;
      const float f = exp2f(ms[g] - M);
      L += ls[g] * f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) O[e] = fmaf(f, ov[g][e], O[e]);
    }
  }
  for (int c0 = 0; c0 <= pos; c0 += KG) {
    float vv[KG][EPL];
#pragma unroll
    for (int g = 0; g < KG; ++g) {
      const int c = c0 + g;
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        vv[g][e] = c <= pos ? ld_elem(vd, (kv_row0 + c * (p.Hkv)) * DH + lane + 32 * e) : 0.f;
    }
#pragma unroll
    for (int g = 0; g < KG; ++g) {
      if (c0 + g > pos) continue;
      const float f = exp2f(sc_s[wid][c0 + g] - M);
      L += f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) O[e] = fmaf(f, vv[g][e], O[e]);
    }
  }
  const float inv = 1.f / L;
  if (p.out_f32) {
    float* out = static_cast<float*>(p.out) + R * DH;
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = O[e] * inv;
  } else {
    T* out = static_cast<T*>(p.out) + R * DH;
#pragma unroll
    for (int e = 0; e < EPL; ++e) st_elem(out, lane + 32 * e, O[e] * inv);
  }
}

// ---------------------------------------------------------------- host
static int choose_splits(const ssd_attn_args* a, int* chunk_out) {
  const int NT = a->NB * a->Dmax;
  const int G = a->Hq / a->Hkv;
  const long long rowgrps = (static_cast<long long>(NT) * G + kSimtRows - 1) / kSimtRows;
  const long long ctas = rowgrps * a->B * a->Hkv;
  const long long P = a->P_max > 0 ? a->P_max : 1;
  long long S = (8LL * 152 + ctas - 1) / ctas;
  const long long S_cap = (P + kKeyTile - 1) / kKeyTile;
  if (S > S_cap) S = S_cap;
  if (S > 64) S = 64;
  if (S < 1) S = 1;
  long long chunk = (P + S - 1) / S;
  chunk = (chunk + kKeyTile - 1) / kKeyTile * kKeyTile;
  S = (P + chunk - 1) / chunk;
  if (S < 1) S = 1;
  *chunk_out = static_cast<int>(chunk);
  return static_cast<int>(S);
}

static int validate(const ssd_attn_args* a) {
  if (a == nullptr) return SSD_ERR_INVALID;
  if (a->B < 0 || a->NB < 1 || a->Dmax < 1 || a->Hq < 1 || a->Hkv < 1 || a->P_max < 0) return SSD_ERR_INVALID;
  if (a->dtype != SSD_F32 && a->dtype != SSD_BF16) return SSD_ERR_INVALID;
  if (a->out_dtype != a->dtype && a->out_dtype != SSD_F32) return SSD_ERR_INVALID;
  if (a->Hq % a->Hkv != 0) return SSD_ERR_INVALID;
  if (a->skip_absent < 0 || a->skip_absent > 2) return SSD_ERR_INVALID;
  if (a->all_rows != 0 && a->all_rows != 1) return SSD_ERR_INVALID;
  if (a->all_rows && a->skip_absent) return SSD_ERR_INVALID;
  if (a->max_ctas < 0) return SSD_ERR_INVALID;
  if (a->Dmax > 256 || a->NB * a->Dmax > 8192 || a->Hq / a->Hkv > 64) return SSD_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->B) * a->Hkv > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  if (a->dh != 64 && a->dh != 128) return SSD_ERR_UNSUPPORTED;
  if (a->P_max > (1LL << 30)) return SSD_ERR_UNSUPPORTED;
  if (a->block_table != nullptr) {
    if (a->dtype != SSD_BF16 || a->dh != 128) return SSD_ERR_UNSUPPORTED;
    if (a->pages_per_seq < 1 || a->num_pages < 1) return SSD_ERR_INVALID;
    if (a->num_pages * a->Hkv * 128LL >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
    if (a->P_max > 128LL * a->pages_per_seq) return SSD_ERR_INVALID;
  }
  if (a->B == 0) return SSD_OK;
  if (!a->q || !a->k_cand || !a->v_cand || !a->out || !a->prefix_len) return SSD_ERR_INVALID;
  if (!a->all_rows && !a->blk_len) return SSD_ERR_INVALID;
  if (a->P_max > 0 && (!a->k_cache || !a->v_cache)) return SSD_ERR_INVALID;
  return SSD_OK;
}

struct AttnLayout {
  size_t ml_off, o_off, total;
  int S, chunk;
};

static AttnLayout attn_layout(const ssd_attn_args* a) {
  AttnLayout L{};
  L.S = choose_splits(a, &L.chunk);
  const size_t R = static_cast<size_t>(a->B) * a->NB * a->Dmax * a->Hq;
  L.ml_off = sizeof(WsHeader);
  L.o_off = round_up(L.ml_off + R * L.S * 2 * sizeof(float), 256);
  L.total = round_up(L.o_off + R * L.S * a->dh * sizeof(float), 256);
  return L;
}

}  // namespace ssd

using namespace ssd;

extern "C" size_t ssd_verify_attn_workspace_size(const ssd_attn_args* a) {
  if (validate(a) != SSD_OK) return 0;
  if (a->B == 0) return sizeof(WsHeader);
  // the path the call will take: the tensor-core kernel merges on chip and needs only the
  // header; the SIMT passes keep every split's partial rows
  if (attn_tc_applies(a)) return attn_tc_workspace_size(a);
  return attn_layout(a).total;
}

extern "C" int ssd_verify_attn(const ssd_attn_args* a, void* ws, size_t ws_bytes, void* stream) {
  int st = validate(a);
  if (st != SSD_OK) return st;
  if (a->B == 0) return SSD_OK;
  if (ws == nullptr || !aligned(ws, 256)) return SSD_ERR_WORKSPACE;
  if (ws_bytes < ssd_verify_attn_workspace_size(a)) return SSD_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (attn_tc_applies(a)) return attn_tc_launch(a, ws, s);
  if (a->block_table != nullptr) return SSD_ERR_UNSUPPORTED;   // paged caches: tensor-core path only

  const AttnLayout L = attn_layout(a);
  AttnParams p{};
  p.q = a->q; p.k_cache = a->k_cache; p.v_cache = a->v_cache; p.k_cand = a->k_cand; p.v_cand = a->v_cand;
  p.out = a->out; p.prefix_len = a->prefix_len; p.blk_len = a->blk_len;
  p.B = a->B; p.NB = a->NB; p.Dmax = a->Dmax; p.Hq = a->Hq; p.Hkv = a->Hkv; p.P_max = a->P_max;
  const float scale = a->scale != 0.f ? a->scale : 1.f / sqrtf(static_cast<float>(a->dh));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.S = L.S; p.chunk = L.chunk;
  p.out_f32 = (a->out_dtype == SSD_F32) ? 1 : 0;
  p.all_rows = a->all_rows;
  char* base = static_cast<char*>(ws);
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.ws_ml = reinterpret_cast<float*>(base + L.ml_off);
  p.ws_o = reinterpret_cast<float*>(base + L.o_off);

  const int NT = a->NB * a->Dmax;
  const int G = a->Hq / a->Hkv;
  dim3 g1(a->B * a->Hkv, (NT * G + kSimtRows - 1) / kSimtRows, L.S);
  {
    KernelTimer t(SSD_KERNEL_VERIFY_ATTN, s);
    if (a->dtype == SSD_F32) {
      if (a->dh == 64) k_attn_prefix_simt<float, 64><<<g1, kSimtThreads, 0, s>>>(p);
      else k_attn_prefix_simt<float, 128><<<g1, kSimtThreads, 0, s>>>(p);
    } else {
      if (a->dh == 64) k_attn_prefix_simt<uint16_t, 64><<<g1, kSimtThreads, 0, s>>>(p);
      else k_attn_prefix_simt<uint16_t, 128><<<g1, kSimtThreads, 0, s>>>(p);
    }
  }
  const int rc = check_launch();
  if (rc != SSD_OK) return rc;
  count_launch(2);
  return attn_combine_launch(p, a->dtype, a->dh, s);
}

namespace ssd {
int attn_combine_launch(const AttnParams& p, int dtype, int dh, cudaStream_t s) {
  const int NT = p.NB * p.Dmax;
  const long long rows = static_cast<long long>(p.B) * NT * p.Hq;
  dim3 g2(static_cast<unsigned>((rows + 3) / 4));
  KernelTimer t(SSD_KERNEL_ATTN_COMBINE, s);
  cudaError_t e;
  if (dtype == SSD_F32) {
    if (dh == 64) e = launch_pdl(k_attn_combine<float, 64>, g2, dim3(128), 0, s, p);
    else e = launch_pdl(k_attn_combine<float, 128>, g2, dim3(128), 0, s, p);
  } else {
    if (dh == 64) e = launch_pdl(k_attn_combine<uint16_t, 64>, g2, dim3(128), 0, s, p);
    else e = launch_pdl(k_attn_combine<uint16_t, 128>, g2, dim3(128), 0, s, p);
  }
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  return check_launch();
}
}  // namespace ssd
