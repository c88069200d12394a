// The SlimSpec low-rank draft LM head on the tensor cores (sm_103a).
//
// SlimSpec page, "방법론: SlimSpec" / "아키텍처": the drafter's head is
// z = W_up (W_down h) with W_down [r][d] and W_up [V][r] (r such as d/8) instead
// of the full-rank W_full [V][d]. The draft distribution q = softmax(z) over the
// whole vocabulary is summarised per row by its max, natural log-sum-exp and
// first argmax (the greedy draft token); the logits themselves are written when
// the caller asks for them.
//
// Three kernels, chained by programmatic dependent launch:
//  k_head_down     u = W_down h. Grid (8, ceil(r/128)), clusters of 8 along d:
//                  a CTA multiplies a 128-row tile of W_down (the M of the MMA)
//                  by h (the N, the batch rows padded to 16) over its eighth of
//                  d, in TMEM; the eight partial tiles meet in distributed shared
//                  memory, where each CTA adds 16 of the rows in rank order and
//                  writes them as bf16 (the second product's operand).
//  k_head_up       z = W_up u and its statistics. One CTA per SM, a contiguous
//                  range of 128-row vocabulary tiles each. u stays in shared
//                  memory; W_up streams through a TMA ring whose first loads go
//                  out before the wait for k_head_down (the weights do not
//                  depend on it). The MMA thread fills one of two TMEM
//                  accumulators while four epilogue warps reduce the other: per
//                  batch column, the max, sum of exp and first argmax over the
//                  tile's rows by warp reductions that transpose as they go.
//  k_head_combine  one CTA per batch row merges the per-CTA statistics in CTA
//                  order.
// Warp roles in the first two: warps 0-3 epilogue (one TMEM lane each), warp 4
// TMEM allocation and TMA producer, warp 5 the single MMA-issuing thread.
// Every mbarrier wait is bounded; on expiry SSD_ERR_TIMEOUT is recorded in the
// workspace header, the remaining waits return at once and the kernel exits
// through its barriers after its copies in flight have landed.
#include <limits.h>
#include <math.h>

#include "ssd_tc.cuh"

namespace ssd {
namespace head {
using namespace tc;

constexpr int BM = 128;                    // rows of a W_down / W_up tile
constexpr int KAT = 64;                    // K elements per 128-byte swizzle atom
constexpr uint32_t kATile = BM * 128;      // one atom of a 128-row tile: 16 KB
constexpr int kMaxRows = 64;               // rows of h per call
constexpr int kMaxRank = 1024;
constexpr int kCluster = 8;                // split of d in k_head_down
constexpr int kThreads = 192;
constexpr int kDownStages = 6;
constexpr int kMaxUpStages = 16;
constexpr int kPartStride = kMaxRows + 4;  // floats per row of a partial tile (conflict-free float4 rows)
constexpr int kSmemLimit = 232448;
constexpr unsigned long long kWaitClocks = 1ull << 32;
constexpr unsigned long long kDrainClocks = 1ull << 30;

struct HeadParams {
  uint16_t* u;          // [M][r] bf16, workspace
  void* logits;         // [M][V] or NULL
  float* row_max;
  float* lse;
  int32_t* argmax;
  float4* parts;        // [grid of k_head_up][64]: (max, sum of exp(z - max), argmax bits, 0)
  WsHeader* hdr;
  int M, N, d, r, V;    // N = M rounded up to 16
  int tiles;            // ceil(V / 128)
  int up_stages;
  int logits_bf16;
};

struct DownBars {
  uint64_t full[kDownStages], empty[kDownStages];
  uint64_t acc_full;
  uint32_t tmem_base;
  int failed;
};

struct UpBars {
  uint64_t full[kMaxUpStages], empty[kMaxUpStages];
  uint64_t u_full;
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int failed;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait for copies already issued to land, without the CTA's failure flag (used
// after a failure, before the shared memory they write is released).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = clock64();
  while (!mbar_probe(bar, parity))
    if (clock64() - t0 > kDrainClocks) return;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ------------------------------------------------------------------ k_head_down
// grid (8, ceil(r/128)), cluster (8, 1, 1)
__global__ void __launch_bounds__(kThreads, 1)
k_head_down(const __grid_constant__ CUtensorMap map_wd, const __grid_constant__ CUtensorMap map_h, HeadParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bstride = kATile + static_cast<uint32_t>(p.N) * 128;   // W_down atom + h atom
  float* part = reinterpret_cast<float*>(smem + kDownStages * bstride);
  DownBars& bars = *reinterpret_cast<DownBars*>(smem + kDownStages * bstride + BM * kPartStride * 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = static_cast<int>(cluster_rank());
  const int rt = blockIdx.y;
  const int natoms = (p.d + KAT - 1) / KAT;
  const int a0 = q * natoms / kCluster, n_at = (q + 1) * natoms / kCluster - a0;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kDownStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.acc_full, 1);
    bars.failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(64)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  auto wait = [&](uint64_t* bar, uint32_t parity, int where) {
    return mbar_wait_bounded(bar, parity, &bars.failed, p.hdr, where, kWaitClocks);
  };

  if (warp == 4 && lane == 0) {
    prefetch_tmap(&map_wd);
    prefetch_tmap(&map_h);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // h comes from the preceding kernel
    int issued = 0;
    for (int i = 0; i < n_at; ++i) {
      const int s = i % kDownStages;
      if (!wait(&bars.empty[s], ((i / kDownStages) & 1) ^ 1, 60)) break;
      mbar_expect_tx(&bars.full[s], bstride);
      const uint32_t dst = sbase + s * bstride;
      tma_load_2d(dst, &map_wd, (a0 + i) * KAT, rt * BM, &bars.full[s]);
      tma_load_2d(dst + kATile, &map_h, (a0 + i) * KAT, 0, &bars.full[s]);
      ++issued;
    }
    for (int s = 0; s < kDownStages && s < issued; ++s) {
      const int n_s = (issued - 1 - s) / kDownStages + 1;   // loads that went to stage s
      drain_wait(&bars.full[s], (n_s - 1) & 1);
    }
  } else if (warp == 5 && lane == 0) {
    const uint32_t idesc = idesc_bf16(false, static_cast<uint32_t>(p.N));
    for (int i = 0; i < n_at; ++i) {
      const int s = i % kDownStages;
      if (!wait(&bars.full[s], (i / kDownStages) & 1, 61)) break;
      tc_fence_after();
      const uint32_t a = sbase + s * bstride;
#pragma unroll
      for (int k = 0; k < KAT / 16; ++k)
        mma_bf16(tmem, sw128_desc(a + k * 32, 16, 1024), sw128_desc(a + kATile + k * 32, 16, 1024), idesc,
                 (i | k) != 0 ? 1u : 0u);
      mma_commit(&bars.empty[s]);
    }
    if (n_at > 0) mma_commit(&bars.acc_full);
  } else if (warp < 4) {
    // this thread's row of the partial tile, N columns, to shared memory
    float* prow = part + (warp * 32 + lane) * kPartStride;
    int ok = 0;
    if (lane == 0) ok = n_at > 0 && wait(&bars.acc_full, 0, 62);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after();
      for (int c0 = 0; c0 < p.N; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          if (c0 + j < p.N)
            *reinterpret_cast<float4*>(prow + c0 + j) = make_float4(
                __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      }
    } else {
      for (int c = 0; c < p.N; c += 4) *reinterpret_cast<float4*>(prow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's partial tile is in its shared memory

  // this CTA adds rows [16q, 16q + 16) of the tile over the 8 ranks, in rank order
  if (tid < 128) {
    const int row = q * (BM / kCluster) + (tid >> 3);
    const int rg = rt * BM + row;
    const uint32_t raddr = smem_u32(part + row * kPartStride);
    for (int c4 = tid & 7; c4 < p.N / 4; c4 += 8) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int pr = 0; pr < kCluster; ++pr) {
        const float4 x = ld_dsmem_f4(map_peer(raddr + c4 * 16, static_cast<uint32_t>(pr)));
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      if (rg < p.r) {
        const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = c4 * 4 + e;
          if (m < p.M) p.u[static_cast<size_t>(m) * p.r + rg] = f32_to_bf16(vals[e]);
        }
      }
    }
  }
  cluster_sync();   // peers keep their partial tiles until every CTA has read them
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(64) : "memory");
  }
}

// ------------------------------------------------------------------ k_head_up
// Warp-wide reduction of 32 columns (one value per lane and column) that
// transposes as it goes: at each step a lane keeps half of its columns and
// trades the other half with its partner, so after five steps lane L holds
// column L reduced over all 32 lanes, for 31 shuffles instead of 160.
template <int S, typename Op>
__device__ __forceinline__ void transpose_step(float* t, int lane, Op op) {
  const bool up = (lane & S) != 0;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const float send = up ? t[i] : t[i + S];
    const float keep = up ? t[i + S] : t[i];
    t[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, S));
  }
}

template <typename Op>
__device__ __forceinline__ float transpose_reduce(float* t, int lane, Op op) {
  transpose_step<16>(t, lane, op);
  transpose_step<8>(t, lane, op);
  transpose_step<4>(t, lane, op);
  transpose_step<2>(t, lane, op);
  transpose_step<1>(t, lane, op);
  return t[0];
}

// Statistics of 32 batch columns over the warp's 32 rows (lane = row, z[j] =
// column j): lane L receives column L's max, sum of exp(z - max) and the first
// lane holding the max (-1 if no row is valid).
__device__ __forceinline__ void column_stats(const float* z, bool valid, int lane, float& cmax, float& csum,
                                             int& crow) {
  float t[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) t[j] = valid ? z[j] : -INFINITY;
  cmax = transpose_reduce(t, lane, [](float a, float b) { return fmaxf(a, b); });
  crow = -1;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float mj = __shfl_sync(0xffffffffu, cmax, j);
    const unsigned hit = __ballot_sync(0xffffffffu, valid && z[j] == mj);
    if (lane == j) crow = hit != 0u ? __ffs(static_cast<int>(hit)) - 1 : -1;
    t[j] = valid ? ex2_approx((z[j] - mj) * kLog2e) : 0.f;
  }
  csum = transpose_reduce(t, lane, [](float a, float b) { return a + b; });
}

// (m, s, a) <- (m, s, a) merged with (m2, s2, a2); s is a sum of exp(z - m); the
// argmax is the lowest index among equal maxima.
__device__ __forceinline__ void merge_stats(float& m, float& s, int& a, float m2, float s2, int a2) {
  if (m2 > m) {
    s = s * ex2_approx((m - m2) * kLog2e) + s2;
    m = m2;
    a = a2;
  } else if (m2 > -INFINITY) {
    s += s2 * ex2_approx((m2 - m) * kLog2e);
    if (m2 == m && a2 < a) a = a2;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
k_head_up(const __grid_constant__ CUtensorMap map_wu, const __grid_constant__ CUtensorMap map_u, HeadParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const int KA = (p.r + KAT - 1) / KAT;
  const uint32_t uatom = static_cast<uint32_t>(p.N) * 128;
  const uint32_t ubytes = KA * uatom;
  const uint32_t ring = sbase + ubytes;
  float4* scratch = reinterpret_cast<float4*>(smem + ubytes + p.up_stages * kATile);
  UpBars& bars = *reinterpret_cast<UpBars*>(smem + ubytes + p.up_stages * kATile + 4 * kMaxRows * sizeof(float4));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int base = p.tiles / G, rem = p.tiles % G;
  const int t0 = c * base + min(c, rem), nt = base + (c < rem ? 1 : 0);
  const int total = nt * KA;   // ring loads of this CTA

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < p.up_stages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.u_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.acc_full[i], 1);
      mbar_init(&bars.acc_empty[i], 4);
    }
    bars.failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(128)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  auto wait = [&](uint64_t* bar, uint32_t parity, int where) {
    return mbar_wait_bounded(bar, parity, &bars.failed, p.hdr, where, kWaitClocks);
  };

  if (warp == 4 && lane == 0) {
    prefetch_tmap(&map_wu);
    prefetch_tmap(&map_u);
    // ring load i: vocabulary tile t0 + i / KA, K atom i % KA
    auto issue = [&](int i) {
      const int s = i % p.up_stages;
      if (!wait(&bars.empty[s], ((i / p.up_stages) & 1) ^ 1, 70)) return false;
      mbar_expect_tx(&bars.full[s], kATile);
      tma_load_2d(ring + s * kATile, &map_wu, (i % KA) * KAT, (t0 + i / KA) * BM, &bars.full[s]);
      return true;
    };
    int i = 0;
    const int pre = min(total, p.up_stages);
    for (; i < pre; ++i) issue(i);                         // weights: independent of the preceding kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");     // u comes from k_head_down
    mbar_expect_tx(&bars.u_full, ubytes);
    for (int kc = 0; kc < KA; ++kc) tma_load_2d(sbase + kc * uatom, &map_u, kc * KAT, 0, &bars.u_full);
    for (; i < total; ++i)
      if (!issue(i)) break;
    drain_wait(&bars.u_full, 0);
    for (int s = 0; s < p.up_stages && s < i; ++s) {
      const int n_s = (i - 1 - s) / p.up_stages + 1;
      drain_wait(&bars.full[s], (n_s - 1) & 1);
    }
  } else if (warp == 5 && lane == 0) {
    const uint32_t idesc = idesc_bf16(false, static_cast<uint32_t>(p.N));
    bool ok = wait(&bars.u_full, 0, 71);
    int i = 0;
    for (int t = 0; ok && t < nt; ++t) {
      const int a = t & 1;
      if (!wait(&bars.acc_empty[a], ((t >> 1) & 1) ^ 1, 72)) break;
      tc_fence_after();
      for (int kc = 0; kc < KA; ++kc, ++i) {
        const int s = i % p.up_stages;
        if (!wait(&bars.full[s], (i / p.up_stages) & 1, 73)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t A = ring + s * kATile, B = sbase + kc * uatom;
#pragma unroll
        for (int k = 0; k < KAT / 16; ++k)
          mma_bf16(tmem + a * 64, sw128_desc(A + k * 32, 16, 1024), sw128_desc(B + k * 32, 16, 1024), idesc,
                   (kc | k) != 0 ? 1u : 0u);
        mma_commit(&bars.empty[s]);
      }
      mma_commit(&bars.acc_full[a]);
    }
  } else if (warp < 4) {
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int ng = (p.M + 31) / 32;
    float rm[2] = {-INFINITY, -INFINITY}, rs[2] = {0.f, 0.f};
    int ra[2] = {INT_MAX, INT_MAX};
    for (int t = 0; t < nt; ++t) {
      const int a = t & 1;
      int ok = 0;
      if (lane == 0) ok = wait(&bars.acc_full[a], (t >> 1) & 1, 74);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int row0 = (t0 + t) * BM + warp * 32;
      const int v = row0 + lane;
      const bool valid = v < p.V;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (g >= ng) break;
        uint32_t raw[32];
        tmem_ld32(tmem + lane_off + a * 64 + g * 32, raw);
        tmem_wait_ld();
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(raw[j]);
        if (p.logits != nullptr && valid) {
          const int mend = min(32, p.M - g * 32);
          if (p.logits_bf16) {
            uint16_t* L = static_cast<uint16_t*>(p.logits) + static_cast<size_t>(g * 32) * p.V + v;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < mend) L[static_cast<size_t>(j) * p.V] = f32_to_bf16(z[j]);
          } else {
            float* L = static_cast<float*>(p.logits) + static_cast<size_t>(g * 32) * p.V + v;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < mend) L[static_cast<size_t>(j) * p.V] = z[j];
          }
        }
        float cmax, csum;
        int crow;
        column_stats(z, valid, lane, cmax, csum, crow);
        merge_stats(rm[g], rs[g], ra[g], cmax, csum, crow >= 0 ? row0 + crow : INT_MAX);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.acc_empty[a]);
    }
    // the four warps' statistics, merged in warp order per column
#pragma unroll
    for (int g = 0; g < 2; ++g)
      scratch[warp * kMaxRows + g * 32 + lane] = make_float4(rm[g], rs[g], __int_as_float(ra[g]), 0.f);
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (tid < p.M) {
      float4 s0 = scratch[tid];
      float m = s0.x, s = s0.y;
      int am = __float_as_int(s0.z);
      for (int w = 1; w < 4; ++w) {
        const float4 x = scratch[w * kMaxRows + tid];
        merge_stats(m, s, am, x.x, x.y, __float_as_int(x.z));
      }
      p.parts[c * kMaxRows + tid] = make_float4(m, s, __int_as_float(am), 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128) : "memory");
  }
}

// ------------------------------------------------------------------ k_head_combine
// grid M, 256 threads: row blockIdx.x, the G per-CTA statistics merged in a fixed order
__global__ void __launch_bounds__(256) k_head_combine(HeadParams p, int G) {
  __shared__ float4 wst[8];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int m = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mx = -INFINITY, s = 0.f;
  int a = INT_MAX;
  for (int c = tid; c < G; c += 256) {
    const float4 x = p.parts[c * kMaxRows + m];
    merge_stats(mx, s, a, x.x, x.y, __float_as_int(x.z));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
    merge_stats(mx, s, a, m2, s2, a2);
  }
  if (lane == 0) wst[warp] = make_float4(mx, s, __int_as_float(a), 0.f);
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < 8; ++w) merge_stats(mx, s, a, wst[w].x, wst[w].y, __float_as_int(wst[w].z));
    p.row_max[m] = mx;
    p.lse[m] = mx + logf(s);
    p.argmax[m] = a;
  }
}

// ------------------------------------------------------------------ host
static bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(KAT), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static int up_grid(const ssd_head_args* a) {
  const int tiles = (a->V + BM - 1) / BM;
  const int n = num_sms();
  return n > 0 ? min(n, tiles) : 0;
}

static size_t u_bytes(const ssd_head_args* a) { return round_up(static_cast<size_t>(a->M) * a->r * 2, 256); }

static int validate(const ssd_head_args* a) {
  if (a == nullptr || a->h == nullptr || a->w_down == nullptr || a->w_up == nullptr) return SSD_ERR_INVALID;
  if (a->row_max == nullptr || a->lse == nullptr || a->argmax == nullptr) return SSD_ERR_INVALID;
  if (a->M < 1 || a->M > kMaxRows || a->d < 8 || a->r < 8 || a->V < 1) return SSD_ERR_INVALID;
  if (a->logits != nullptr && a->logits_dtype != SSD_F32 && a->logits_dtype != SSD_BF16) return SSD_ERR_INVALID;
  if ((a->d % 8) != 0 || (a->r % 8) != 0 || a->r > kMaxRank) return SSD_ERR_UNSUPPORTED;
  if (!aligned(a->h, 16) || !aligned(a->w_down, 16) || !aligned(a->w_up, 16)) return SSD_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->V) + BM >= (1LL << 31)) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

static bool device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3 && encode_fn() != nullptr;
}

}  // namespace head
}  // namespace ssd

using namespace ssd;
using namespace ssd::head;

extern "C" size_t ssd_lowrank_head_workspace_size(const ssd_head_args* a) {
  if (validate(a) != SSD_OK) return 0;
  const int G = up_grid(a);
  if (G <= 0) return 0;
  return sizeof(WsHeader) + u_bytes(a) + static_cast<size_t>(G) * kMaxRows * sizeof(float4);
}

extern "C" int ssd_lowrank_head(const ssd_head_args* a, void* ws, size_t ws_bytes, void* stream) {
  const int st = validate(a);
  if (st != SSD_OK) return st;
  if (!device_ok()) return SSD_ERR_UNSUPPORTED;
  const size_t need = ssd_lowrank_head_workspace_size(a);
  if (need == 0) return SSD_ERR_CUDA;
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < need) return SSD_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(k_head_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_head_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;

  HeadParams p{};
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  p.hdr = reinterpret_cast<WsHeader*>(wsb);
  p.u = reinterpret_cast<uint16_t*>(wsb + sizeof(WsHeader));
  p.parts = reinterpret_cast<float4*>(wsb + sizeof(WsHeader) + u_bytes(a));
  p.logits = a->logits;
  p.logits_bf16 = (a->logits != nullptr && a->logits_dtype == SSD_BF16) ? 1 : 0;
  p.row_max = a->row_max;
  p.lse = a->lse;
  p.argmax = a->argmax;
  p.M = a->M;
  p.N = (a->M + 15) / 16 * 16;
  p.d = a->d;
  p.r = a->r;
  p.V = a->V;
  p.tiles = (a->V + BM - 1) / BM;
  const int G = up_grid(a);
  const int KA = (a->r + KAT - 1) / KAT;
  const size_t ubytes = static_cast<size_t>(KA) * p.N * 128;
  const size_t up_fixed = 1024 + ubytes + 4 * kMaxRows * sizeof(float4) + sizeof(UpBars);
  p.up_stages = min(kMaxUpStages, static_cast<int>((kSmemLimit - up_fixed) / kATile));
  if (p.up_stages < 2) return SSD_ERR_UNSUPPORTED;
  const size_t up_smem = up_fixed + static_cast<size_t>(p.up_stages) * kATile;
  const size_t down_smem =
      1024 + kDownStages * (kATile + static_cast<size_t>(p.N) * 128) + BM * kPartStride * 4 + sizeof(DownBars);
  if (down_smem > static_cast<size_t>(kSmemLimit)) return SSD_ERR_UNSUPPORTED;

  CUtensorMap m_wd, m_h, m_wu, m_u;
  if (!make_map(&m_wd, a->w_down, a->d, a->r, BM) || !make_map(&m_h, a->h, a->d, a->M, p.N) ||
      !make_map(&m_wu, a->w_up, a->r, a->V, BM) || !make_map(&m_u, p.u, a->r, a->M, p.N))
    return SSD_ERR_CUDA;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCluster, static_cast<unsigned>((a->r + BM - 1) / BM), 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = down_smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    KernelTimer timer(SSD_KERNEL_HEAD_DOWN, s);
    if (cudaLaunchKernelEx(&cfg, k_head_down, m_wd, m_h, p) != cudaSuccess) return SSD_ERR_CUDA;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = up_smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    KernelTimer timer(SSD_KERNEL_HEAD_UP, s);
    if (cudaLaunchKernelEx(&cfg, k_head_up, m_wu, m_u, p) != cudaSuccess) return SSD_ERR_CUDA;
  }
  {
    KernelTimer timer(SSD_KERNEL_HEAD_COMBINE, s);
    if (launch_pdl(k_head_combine, dim3(static_cast<unsigned>(a->M)), dim3(256), 0, s, p, G) != cudaSuccess)
      return SSD_ERR_CUDA;
  }
  count_launch(3);
  return check_launch();
}
