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
//  k_head_down     u = W_down h. Grid (CS, ceil(r/128)), clusters of CS = 16 CTAs
//                  along d (8 where a 16-CTA cluster cannot be scheduled): a CTA
//                  multiplies a 128-row tile of W_down (the M of the MMA) by h
//                  (the N, the batch rows padded to 16) over its 1/CS of d, in
//                  TMEM; the partial tiles meet in distributed shared memory,
//                  where each CTA adds 128/CS of the rows in rank order and
//                  writes them as bf16 (the second product's operand).
//  k_head_up       z = W_up u and its statistics. One CTA per SM, a contiguous
//                  range of 128-row vocabulary tiles each. u stays in shared
//                  memory; W_up streams through a TMA ring whose first loads go
//                  out before the wait for k_head_down (the weights do not
//                  depend on it). The MMA thread fills one of two TMEM
//                  accumulators while eight epilogue warps (a TMEM lane quarter
//                  and 32 batch columns each) empty the other and fold it into
//                  per-lane running statistics: for each batch column, the max,
//                  the sum of exp(z - max) (one exponential per logit) and the
//                  first row at the max. At the end of its range a warp merges
//                  its 32 lanes per column with shuffles that transpose as they
//                  go, and the four lane quarters are merged in order.
//  k_head_combine  one CTA per batch row merges the per-CTA statistics in CTA
//                  order.
// Warp roles: in k_head_down warps 0-3 epilogue (one TMEM lane each), warp 4 TMEM
// allocation and TMA producer, warp 5 the single MMA-issuing thread; in k_head_up
// warps 0-7 epilogue, warp 8 TMEM allocation and producer, warp 9 MMA.
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
constexpr int kClusterMax = 16;            // split of d in k_head_down (16, else 8 where 16 cannot be scheduled)
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
// grid (CS, ceil(r/128)), cluster (CS, 1, 1)
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
  const int CS = gridDim.x;                  // cluster size: the grid is one cluster wide
  const int rt = blockIdx.y;
  const int natoms = (p.d + KAT - 1) / KAT;
  const int a0 = q * natoms / CS, n_at = (q + 1) * natoms / CS - a0;

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

  // this CTA adds rows [q RP, (q + 1) RP) of the tile over the CS ranks, in rank order
  const int RP = BM / CS, nq = p.N / 4;
  for (int it = tid; it < RP * nq; it += kThreads) {
    const int row = q * RP + it / nq, c4 = it % nq;
    const int rg = rt * BM + row;
    const uint32_t addr = smem_u32(part + row * kPartStride + c4 * 4);
    {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int pr = 0; pr < CS; ++pr) {
        const float4 x = ld_dsmem_f4(map_peer(addr, static_cast<uint32_t>(pr)));
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
constexpr int kUpEpiWarps = 8;                        // TMEM lane quarter w % 4, column group w / 4
constexpr int kUpThreads = 32 * (kUpEpiWarps + 2);    // + warp 8 producer, warp 9 MMA

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

// One step of a warp-wide merge of 32 column states (one per lane and column) that
// transposes as it goes: a lane keeps half of its columns and trades the other half
// with its partner, so after the five steps S = 16 .. 1 lane L holds column L merged
// over all 32 lanes, for 31 exchanges per lane.
template <int S>
__device__ __forceinline__ void transpose_merge_step(float* m, float* s, int* a, int lane) {
  const bool up = (lane & S) != 0;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    const float send_m = up ? m[i] : m[i + S], send_s = up ? s[i] : s[i + S];
    const int send_a = up ? a[i] : a[i + S];
    float km = up ? m[i + S] : m[i], ks = up ? s[i + S] : s[i];
    int ka = up ? a[i + S] : a[i];
    const float rm = __shfl_xor_sync(0xffffffffu, send_m, S);
    const float rs = __shfl_xor_sync(0xffffffffu, send_s, S);
    const int ra = __shfl_xor_sync(0xffffffffu, send_a, S);
    merge_stats(km, ks, ka, rm, rs, ra);
    m[i] = km;
    s[i] = ks;
    a[i] = ka;
  }
}

__global__ void __launch_bounds__(kUpThreads, 1)
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
  const int ng = (p.M + 31) / 32;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < p.up_stages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.u_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.acc_full[i], 1);
      mbar_init(&bars.acc_empty[i], 4 * ng);   // one arrival per epilogue warp with columns
    }
    bars.failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kUpEpiWarps) {
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

  if (warp == kUpEpiWarps && lane == 0) {
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
  } else if (warp == kUpEpiWarps + 1 && lane == 0) {
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
  } else if (warp < kUpEpiWarps) {
    // rows 32*q4 .. +31 of each tile (this warp's TMEM lanes), columns 32*g .. 32*g + jn - 1
    const int q4 = warp & 3, g = warp >> 2;
    const int jn = min(32, p.M - 32 * g);
    if (jn > 0) {
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + g * 32;
      // per lane and column: running max, sum of exp(z - max), first row at the max
      float m[32], s[32];
      int a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        m[j] = -INFINITY;
        s[j] = 0.f;
        a[j] = INT_MAX;
      }
      for (int t = 0; t < nt; ++t) {
        const int b = t & 1;
        int ok = 0;
        if (lane == 0) ok = wait(&bars.acc_full[b], (t >> 1) & 1, 74);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        tc_fence_after();
        uint32_t raw[32];
        tmem_ld32(taddr + b * 64, raw);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.acc_empty[b]);   // the accumulator is in registers
        const int v = (t0 + t) * BM + q4 * 32 + lane;
        if (v < p.V) {
          if (p.logits != nullptr) {
            if (p.logits_bf16) {
              uint16_t* L = static_cast<uint16_t*>(p.logits) + static_cast<size_t>(g * 32) * p.V + v;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < jn) L[static_cast<size_t>(j) * p.V] = f32_to_bf16(__uint_as_float(raw[j]));
            } else {
              float* L = static_cast<float*>(p.logits) + static_cast<size_t>(g * 32) * p.V + v;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < jn) L[static_cast<size_t>(j) * p.V] = __uint_as_float(raw[j]);
            }
          }
          // online update: of exp(m - x) and exp(x - m) one factor is 1, so one exponential
          // of -|x - m| serves both the rescale (new max) and the new term
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < jn) {
              const float x = __uint_as_float(raw[j]);
              const float mn = fmaxf(m[j], x);
              const float e = ex2_approx((fminf(m[j], x) - mn) * kLog2e);
              const bool grows = x > m[j];
              s[j] = grows ? fmaf(s[j], e, 1.f) : s[j] + e;
              a[j] = grows ? v : a[j];
              m[j] = mn;
            }
          }
        }
      }
      // the warp's 32 rows merged per column: lane L ends with column 32*g + L
      transpose_merge_step<16>(m, s, a, lane);
      transpose_merge_step<8>(m, s, a, lane);
      transpose_merge_step<4>(m, s, a, lane);
      transpose_merge_step<2>(m, s, a, lane);
      transpose_merge_step<1>(m, s, a, lane);
      scratch[q4 * kMaxRows + g * 32 + lane] = make_float4(m[0], s[0], __int_as_float(a[0]), 0.f);
    }
    // the four lane quarters merged in order, one thread per column
    asm volatile("bar.sync 1, %0;" ::"r"(kUpEpiWarps * 32) : "memory");
    if (tid < p.M) {
      const float4 s0 = scratch[tid];
      float mm = s0.x, ss = s0.y;
      int am = __float_as_int(s0.z);
      for (int w = 1; w < 4; ++w) {
        const float4 x = scratch[w * kMaxRows + tid];
        merge_stats(mm, ss, am, x.x, x.y, __float_as_int(x.z));
      }
      p.parts[c * kMaxRows + tid] = make_float4(mm, ss, __int_as_float(am), 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kUpEpiWarps) {
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

static size_t down_smem_bytes(int N) {
  return 1024 + kDownStages * (kATile + static_cast<size_t>(N) * 128) + BM * kPartStride * 4 + sizeof(DownBars);
}

// 16 CTAs per cluster where the device can hold such a cluster of k_head_down at its
// largest shared-memory size, else the portable 8 (per device, decided once)
static int down_cluster_size() {
  static int cache[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 8;
  std::call_once(once[dev], [dev] {
    int cs = 8;
    if (cudaFuncSetAttribute(k_head_down, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
        cudaFuncSetAttribute(k_head_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kClusterMax, 1, 1);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = down_smem_bytes(kMaxRows);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kClusterMax;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k_head_down, &cfg) == cudaSuccess && n >= 1) cs = kClusterMax;
    }
    cudaGetLastError();
    cache[dev] = cs;
  });
  return cache[dev];
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

  static std::once_flag attr_once[kMaxDevices];
  static cudaError_t attr_err[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return SSD_ERR_CUDA;
  std::call_once(attr_once[dev], [dev] {
    attr_err[dev] = cudaFuncSetAttribute(k_head_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (attr_err[dev] == cudaSuccess)
      attr_err[dev] = cudaFuncSetAttribute(k_head_up, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  });
  if (attr_err[dev] != cudaSuccess) return SSD_ERR_CUDA;

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
  const size_t down_smem = down_smem_bytes(p.N);
  if (down_smem > static_cast<size_t>(kSmemLimit)) return SSD_ERR_UNSUPPORTED;
  const int CS = down_cluster_size();

  CUtensorMap m_wd, m_h, m_wu, m_u;
  if (!make_map(&m_wd, a->w_down, a->d, a->r, BM) || !make_map(&m_h, a->h, a->d, a->M, p.N) ||
      !make_map(&m_wu, a->w_up, a->r, a->V, BM) || !make_map(&m_u, p.u, a->r, a->M, p.N))
    return SSD_ERR_CUDA;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(CS);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(CS), static_cast<unsigned>((a->r + BM - 1) / BM), 1);
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
    cfg.blockDim = dim3(kUpThreads);
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
