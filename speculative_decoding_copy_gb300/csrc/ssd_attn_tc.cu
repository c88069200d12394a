// Verification attention for bf16, head dim 128, on the tensor cores.
//
// SwitchSD page, "무엇과 다른가": a candidate token attends to the whole prefix
// and to the earlier tokens of its own candidate, never to another candidate.
// Every candidate token of a sequence sees the same prefix keys, so for one kv
// head the G query heads of all NT candidate slots pack into NT*G rows of one
// dense product with each key tile. A CTA owns 128 packed rows (the M of the
// MMA) and one split of the prefix; the S CTAs of a row tile form a thread-block
// cluster, rank 0 also takes the own-block keys as masked tiles, and the splits
// are merged on chip through distributed shared memory: no partial results go
// to HBM and no second kernel runs.
//
// Per CTA (192 threads, one CTA per SM):
//   warps 0-3  one thread per packed row: stage Q, online softmax from the S
//              row in TMEM (tcgen05.ld) with the row's key mask (a contiguous
//              range per tile), O rescale in TMEM, P as bf16 into shared
//              memory; after the loop the O row, max and sum are staged in
//              shared memory for the cluster merge;
//   warp 4     TMA producer: K and V tiles of 64 keys (two 64-wide halves of
//              the head dim, 128-byte swizzle) into a 4-stage ring, from the
//              prefix cache (2-D map) or the candidate keys (3-D map);
//   warp 5     TMEM allocation and the single MMA-issuing thread:
//              S = Q K^T (M128 N64, K16 x 8) into one of two TMEM buffers and
//              O += P V (M128 N128, K16 x 4), kind::f16 with bf16 operands and
//              fp32 accumulators in TMEM. S of tile j+1 is issued before P V of
//              tile j so the tensor core works while the rows run the softmax;
//              P is double-buffered in shared memory.
// Merge: each CTA of the cluster normalises 128/S rows, reading every split's
// O, max and sum from its peers' shared memory, and writes the bf16 output of
// the tokens that exist. The kernel may be launched before the retrieval that
// decides which tokens exist has finished (programmatic dependent launch): it
// reads the block lengths only after griddepcontrol.wait, just before writing.
// Every mbarrier wait is bounded (about 2^32 clocks); on expiry the CTA
// records SSD_ERR_TIMEOUT in the workspace header, skips the remaining waits,
// frees its TMEM and exits through the cluster barriers.
#include <cuda.h>
#include <math.h>

#include <mutex>

#include "ssd_attn.cuh"

namespace ssd {
namespace tc {

constexpr int DH = 128;
constexpr int BM = 128;                   // packed rows per CTA
constexpr int BN = 64;                    // keys per tile
constexpr int STAGES = 4;                 // K/V ring depth
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;       // S buffers: cols 0-63 and 64-127, O: cols 128-255
constexpr uint32_t kQHalf = BM * 128;     // 128 rows x 64 bf16 (one 128-byte-swizzled half): 16 KB
constexpr uint32_t kKVHalf = BN * 128;    // 64 keys x 64 bf16: 8 KB
constexpr uint32_t kPBuf = BM * 128;      // 128 rows x 64 keys bf16: 16 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + 2 * kQHalf;
constexpr uint32_t OFF_V = OFF_K + STAGES * 2 * kKVHalf;
constexpr uint32_t OFF_P = OFF_V + STAGES * 2 * kKVHalf;
constexpr uint32_t OFF_BAR = OFF_P + 2 * kPBuf;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;   // + slack to align the base to 1024
constexpr unsigned long long kWaitClocks = 1ull << 32;
struct Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t q_full;
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint32_t tmem_base;
  int failed;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; false once this CTA has given up (then every later wait returns at once).
__device__ __forceinline__ bool mbar_wait(Bars& bars, uint64_t* bar, uint32_t parity, WsHeader* hdr, int where) {
  volatile int* failed = &bars.failed;
  if (*failed) return false;
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*failed) return false;
    if (clock64() - t0 > kWaitClocks) {
      *failed = 1;
      record_error(hdr, SSD_ERR_TIMEOUT, where);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// whole-cluster barrier: arrive (release) + wait (acquire); every thread of every CTA
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// shared-memory address of the same location in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor, 128-byte swizzle (sm_100 format)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;            // descriptor version
  d |= 2ull << 61;            // SWIZZLE_128B
  return d;
}

// instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128, N = n
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major, uint32_t n) {
  return (1u << 4)            // D: f32
         | (1u << 7)          // A: bf16
         | (1u << 10)         // B: bf16
         | ((b_mn_major ? 1u : 0u) << 16)
         | ((n >> 3) << 17)     // N
         | ((128u >> 4) << 24); // M
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// two fp32 -> packed bf16x2 (round to nearest even), low half = first
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled half
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

// ------------------------------------------------------------------ kernel
constexpr int kMaxSplit = 8;              // cluster size limit (portable)
constexpr int kOStride = 132;             // fp32 per staged O row (padding against bank conflicts)
constexpr int kMergeItems = BM + kMaxSplit;   // bound on (rows merged by one CTA) x S

// grid (S, row tiles, B*Hkv), cluster (S, 1, 1): the S CTAs of one row tile split
// the prefix; cluster rank 0 also takes the own-block (candidate) keys.
__global__ void __launch_bounds__(kThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
          const __grid_constant__ CUtensorMap tmap_kc, const __grid_constant__ CUtensorMap tmap_vc, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars& bars = *reinterpret_cast<Bars*>(smem + OFF_BAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = static_cast<int>(cluster_rank());
  const int S = static_cast<int>(gridDim.x);
  const int mt = blockIdx.y;
  const int b = blockIdx.z / p.Hkv, kvh = blockIdx.z % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int NT = p.NB * p.Dmax;
  const int rows_total = NT * G;
  const int r0 = mt * BM;
  const int P = p.prefix_len[b];
  const int k0 = split * p.chunk;
  const int k1 = min(P, k0 + p.chunk);
  const int nP = k1 > k0 ? (k1 - k0 + BN - 1) / BN : 0;
  // candidate slots of this row tile: from the start of its first token's block to its last token
  const int t_first = r0 / G;
  const int t_last = min(NT - 1, (r0 + BM - 1) / G);
  const int s_base = (t_first / p.Dmax) * p.Dmax;
  const int nC = (split == 0 && t_first < NT) ? (t_last + 1 - s_base + BN - 1) / BN : 0;
  const int nT = nC + nP;

  // this thread's packed row: token t, q-head h, allowed own-block slots [c_lo, t]
  const int r = r0 + tid;
  const bool row_ok = tid < BM && r < rows_total;
  const int t = row_ok ? r / G : 0;
  const int h = row_ok ? kvh * G + r % G : 0;
  const int c_lo = (t / p.Dmax) * p.Dmax;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.q_full, BM);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], BM);
      mbar_init(&bars.p_full[i], BM);
      mbar_init(&bars.pv_done[i], 1);
    }
    bars.failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint32_t tmem_O = tmem + 128;
  float* ostage = reinterpret_cast<float*>(smem + OFF_K);          // [128][kOStride] after the main loop
  float* ml_s = reinterpret_cast<float*>(smem + OFF_P);            // [2][128] after the main loop

  if (warp < 4) {
    // ---------------------------------------------------------- softmax rows
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY, l = 0.f;        // reference max (log2 units) and sum
    if (nT > 0) {
      {
        // stage Q row `tid` (zeros past the last packed row), 128-byte swizzle
        const uint4* q4 = row_ok ? reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                                   ((static_cast<int64_t>(b) * NT + t) * p.Hq + h) * DH)
                                 : nullptr;
        uint4 qv[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) qv[c] = q4 ? __ldg(q4 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_shared_v4(sbase + OFF_Q + (c >> 3) * kQHalf + sw128_off(tid, c & 7), qv[c].x, qv[c].y, qv[c].z,
                       qv[c].w);
        fence_async_smem();
        mbar_arrive(&bars.q_full);
      }
      const float sl2 = p.scale_log2;
      for (int j = 0; j < nT; ++j) {
        const int sb = j & 1;
        mbar_wait(bars, &bars.s_full[sb], (j >> 1) & 1, p.hdr, 10);
        tc_fence_after();
        uint32_t sreg[BN];
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) tmem_ld32(tmem + sb * BN + lane_off + q * 32, sreg + q * 32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars.s_free[sb]);
        // valid columns: a contiguous range [v_lo, v_hi) of this tile
        int v_lo, v_hi;
        if (j < nC) {                                   // own-block keys: slots c_lo .. t
          const int s0 = s_base + j * BN;
          v_lo = row_ok ? c_lo - s0 : BN;
          v_hi = row_ok ? t + 1 - s0 : 0;
        } else {                                        // prefix keys below k1
          v_lo = 0;
          v_hi = k1 - (k0 + (j - nC) * BN);
        }
        if (v_lo > 0 || v_hi < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c < v_lo || c >= v_hi) sreg[c] = __float_as_uint(-INFINITY);
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < BN; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], __uint_as_float(sreg[c]));
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // reference max only moves when the row max grows by more than 2^8
        const float m_new = fmaxf(m, mx * sl2);
        const bool need = m_new > m + 8.f;
        const float mref = need ? m_new : m;
        const float alpha = need ? ex2_approx(m - m_new) : 1.f;
        uint32_t pk[BN / 2];
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
        if (mref > -INFINITY) {
#pragma unroll
          for (int c = 0; c < BN; c += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sreg[c]), sl2, -mref));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sreg[c + 1]), sl2, -mref));
            const uint32_t w = pack_bf16(p0, p1);
            pk[c / 2] = w;
            // sum the rounded values the MMA uses, so numerator and denominator agree
            rs[(c >> 1) & 1] += __uint_as_float(w << 16);
            rs[2 + ((c >> 1) & 1)] += __uint_as_float(w & 0xffff0000u);
          }
        } else {
#pragma unroll
          for (int c = 0; c < BN / 2; ++c) pk[c] = 0u;   // no allowed key yet in this row
        }
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O holds the sum up to tile j-1: wait for its last MMA, then rescale
          mbar_wait(bars, &bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.hdr, 11);
          tc_fence_after();
          uint32_t o[32];
#pragma unroll
          for (int q = 0; q < DH / 32; ++q) {
            tmem_ld32(tmem_O + lane_off + q * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem_O + lane_off + q * 32, o);
          }
          tmem_wait_st();
        }
        l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        m = mref;
        // P buffer sb was last read by the MMA of tile j-2
        if (j >= 2) mbar_wait(bars, &bars.pv_done[sb], ((j - 2) >> 1) & 1, p.hdr, 12);
#pragma unroll
        for (int c = 0; c < BN / 8; ++c)
          st_shared_v4(sbase + OFF_P + sb * kPBuf + sw128_off(tid, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                       pk[4 * c + 3]);
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&bars.p_full[sb]);
      }
      mbar_wait(bars, &bars.pv_done[(nT - 1) & 1], ((nT - 1) >> 1) & 1, p.hdr, 13);
      tc_fence_after();
    }
    // stage this CTA's un-normalised O row, reference max and sum for the cluster merge
    float* orow = ostage + tid * kOStride;
#pragma unroll
    for (int q = 0; q < DH / 32; ++q) {
      uint32_t o[32];
      if (nT > 0) {
        tmem_ld32(tmem_O + lane_off + q * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e)
        reinterpret_cast<float4*>(orow + q * 32)[e] =
            make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]), __uint_as_float(o[4 * e + 2]),
                        __uint_as_float(o[4 * e + 3]));
    }
    ml_s[tid] = m;
    ml_s[BM + tid] = l;
  } else if (warp == 4) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0 && nT > 0) {
      const int y0 = (b * p.Hkv + kvh) * static_cast<int>(p.P_max) + k0;
      for (int j = 0; j < nT; ++j) {
        const int s = j % STAGES;
        if (j >= STAGES) mbar_wait(bars, &bars.empty[s], ((j / STAGES) - 1) & 1, p.hdr, 20);
        if (bars.failed) break;
        mbar_expect_tx(&bars.full[s], 4 * kKVHalf);
        const uint32_t kd = sbase + OFF_K + s * 2 * kKVHalf, vd = sbase + OFF_V + s * 2 * kKVHalf;
        if (j < nC) {
          const int z = b * NT + s_base + j * BN;          // candidate slot (rows past NT are masked)
          tma_load_3d(kd, &tmap_kc, 0, kvh, z, &bars.full[s]);
          tma_load_3d(kd + kKVHalf, &tmap_kc, 64, kvh, z, &bars.full[s]);
          tma_load_3d(vd, &tmap_vc, 0, kvh, z, &bars.full[s]);
          tma_load_3d(vd + kKVHalf, &tmap_vc, 64, kvh, z, &bars.full[s]);
        } else {
          const int y = y0 + (j - nC) * BN;
          tma_load_2d(kd, &tmap_k, 0, y, &bars.full[s]);
          tma_load_2d(kd + kKVHalf, &tmap_k, 64, y, &bars.full[s]);
          tma_load_2d(vd, &tmap_v, 0, y, &bars.full[s]);
          tma_load_2d(vd + kKVHalf, &tmap_v, 64, y, &bars.full[s]);
        }
      }
    }
  } else {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nT > 0) {
      constexpr uint32_t idS = idesc_bf16(false, BN), idPV = idesc_bf16(true, DH);
      mbar_wait(bars, &bars.q_full, 0, p.hdr, 30);
      tc_fence_after();
      // S[j&1] = Q K_j^T : M128 N64, eight K16 steps over the head dim
      auto issue_S = [&](int j) {
        const uint32_t kb = sbase + OFF_K + (j % STAGES) * 2 * kKVHalf;
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const uint64_t a = sw128_desc(sbase + OFF_Q + (ks >> 2) * kQHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(kb + (ks >> 2) * kKVHalf + (ks & 3) * 32, 16, 1024);
          mma_bf16(tmem + (j & 1) * BN, a, bd, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[j & 1]);
      };
      mbar_wait(bars, &bars.full[0], 0, p.hdr, 31);
      tc_fence_after();
      issue_S(0);
      for (int j = 0; j < nT; ++j) {
        if (j + 1 < nT) {
          // S of the next tile into the other buffer, once its previous reader is done
          mbar_wait(bars, &bars.full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1, p.hdr, 32);
          if (j >= 1) mbar_wait(bars, &bars.s_free[(j + 1) & 1], ((j - 1) >> 1) & 1, p.hdr, 33);
          tc_fence_after();
          issue_S(j + 1);
        }
        // O += P_j V_j : M128 N128 (head dim), four K16 steps over the tile's keys
        mbar_wait(bars, &bars.p_full[j & 1], (j >> 1) & 1, p.hdr, 34);
        tc_fence_after();
        const uint32_t vb = sbase + OFF_V + (j % STAGES) * 2 * kKVHalf;
        const uint32_t pb = sbase + OFF_P + (j & 1) * kPBuf;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t a = sw128_desc(pb + ks * 32, 16, 1024);
          const uint64_t bd = sw128_desc(vb + ks * 16 * 128, kKVHalf, 1024);
          mma_bf16(tmem_O, a, bd, idPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&bars.pv_done[j & 1]);
        mma_commit(&bars.empty[j % STAGES]);
      }
    }
  }

  // ---- merge the S splits across the cluster through distributed shared memory
  __syncwarp();
  cluster_sync();                                   // every CTA's O, m, l are staged
  asm volatile("griddepcontrol.wait;" ::: "memory");   // blk_len (which rows exist) is final
  const int rpc = (BM + S - 1) / S;                 // rows merged by each CTA of the cluster
  const int rb = split * rpc, nr = max(0, min(BM, rb + rpc) - rb);
  // scratch after the staged m, l: per (row, split) max and sum, then weights; per-row presence
  float* mm = ml_s + 2 * BM;                        // [nr][S]
  float* ll = mm + kMergeItems;                     // [nr][S]
  float* fac = ll + kMergeItems;                    // [nr][S]: exp2(m_c - M) / L
  int* live = reinterpret_cast<int*>(fac + kMergeItems);   // [nr]
  if (tid < nr * S) {                               // (a) gather every split's max and sum of these rows
    const int i = tid / S, c = tid % S;
    mm[tid] = ld_peer_f32(map_peer(smem_u32(ml_s + rb + i), c));
    ll[tid] = ld_peer_f32(map_peer(smem_u32(ml_s + BM + rb + i), c));
  }
  if (tid < nr) {                                   // presence of the row's token
    const int gr = r0 + rb + tid;
    int ok = 0;
    if (gr < rows_total) {
      const int tt = gr / G;
      ok = (tt % p.Dmax) < p.blk_len[b * p.NB + tt / p.Dmax];
    }
    live[tid] = ok;
  }
  __syncthreads();
  if (tid < nr) {                                   // (b) merged max, sum and per-split weights
    float M = -INFINITY;
    for (int c = 0; c < S; ++c) M = fmaxf(M, mm[tid * S + c]);
    float L = 0.f;
    for (int c = 0; c < S; ++c) {
      const float mc = mm[tid * S + c];
      const float f = mc > -INFINITY ? ex2_approx(mc - M) : 0.f;
      fac[tid * S + c] = f;
      L = fmaf(ll[tid * S + c], f, L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int c = 0; c < S; ++c) fac[tid * S + c] *= inv;
    if (!(L > 0.f)) live[tid] = 0;
  }
  __syncthreads();
  // (c) one float4 of one row per item; a warp covers one row, its S peer loads in flight together
  for (int it = tid; it < nr * (DH / 4); it += kThreads) {
    const int i = it / (DH / 4), q4 = it % (DH / 4);
    if (!live[i]) continue;
    const uint32_t src = smem_u32(ostage + (rb + i) * kOStride + q4 * 4);
    float4 o[kMaxSplit];
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c)
      if (c < S) o[c] = ld_peer_f32x4(map_peer(src, c));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c)
      if (c < S) {
        const float f = fac[i * S + c];
        acc.x = fmaf(f, o[c].x, acc.x);
        acc.y = fmaf(f, o[c].y, acc.y);
        acc.z = fmaf(f, o[c].z, acc.z);
        acc.w = fmaf(f, o[c].w, acc.w);
      }
    const int gr = r0 + rb + i;
    const int tt = gr / G, hh = kvh * G + gr % G;
    const int64_t o_off = ((static_cast<int64_t>(b) * NT + tt) * p.Hq + hh) * DH + q4 * 4;
    if (p.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_off) = acc;
    } else {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + o_off) =
          make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
    }
  }
  cluster_sync();                                   // peers are done reading this CTA's staging

  // teardown: every role is done with TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

static bool make_kv_map(CUtensorMap* map, const void* base, uint64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(DH), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(DH) * 2};
  const cuuint32_t box[2] = {64, BN};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// candidate K or V [B*NT][Hkv][dh] as a 3-D tensor (dh, kv head, slot): a box of
// 64 slots of one kv head lands as a [64][64] tile like a prefix tile
static bool make_cand_map(CUtensorMap* map, const void* base, uint64_t slots, int Hkv) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(DH), static_cast<cuuint64_t>(Hkv), slots};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(DH) * 2, static_cast<cuuint64_t>(Hkv) * DH * 2};
  const cuuint32_t box[3] = {64, 1, BN};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How many clusters of S CTAs can be resident at once (0 if the query fails).
static int max_active_clusters(int S) {
  static int cache[kMaxSplit + 1][64];
  static bool done[kMaxSplit + 1][64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[S][dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_attn_tc, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[S][dev] = n;
    done[S][dev] = true;
  }
  return cache[S][dev];
}

// splits (cluster size <= 8): minimise (waves of clusters) x (key tiles per split + fixed cost)
static void choose_split(const ssd_attn_args* a, int mtiles, int* S_out, int* chunk_out) {
  const long long groups = static_cast<long long>(a->B) * a->Hkv * mtiles;   // clusters in the grid
  const long long nkt = a->P_max > 0 ? (a->P_max + BN - 1) / BN : 1;
  long long best_cost = -1;
  int best_S = 1;
  for (int S = 1; S <= kMaxSplit && S <= nkt; ++S) {
    const int active = max_active_clusters(S);
    if (active <= 0) continue;
    const long long tiles = (nkt + S - 1) / S;
    const long long waves = (groups + active - 1) / active;
    const long long cost = waves * (tiles + 3) * 16 + S;   // +3 tiles: prologue, candidate tile, merge
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_S = S;
    }
  }
  const long long tiles = (nkt + best_S - 1) / best_S;
  *chunk_out = static_cast<int>(tiles * BN);
  *S_out = best_S;
}

}  // namespace tc

static bool tc_disabled_by_env() {
  const char* e = getenv("SSD_ATTN_KERNEL");
  return e != nullptr && e[0] == 's';   // "simt" forces the SIMT prefix pass
}

bool attn_tc_applies(const ssd_attn_args* a) {
  if (tc_disabled_by_env()) return false;
  if (a->dtype != SSD_BF16 || a->dh != tc::DH || a->P_max < 1) return false;
  if (!aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->q, 16)) return false;
  if (!aligned(a->k_cand, 16) || !aligned(a->v_cand, 16) || !aligned(a->out, 16)) return false;
  if (static_cast<long long>(a->B) * a->Hkv * a->P_max >= (1LL << 31)) return false;
  if (static_cast<long long>(a->B) * a->NB * a->Dmax >= (1LL << 31)) return false;
  if (a->B * a->Hkv > 65535) return false;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3 && tc::encode_fn() != nullptr;
}

size_t attn_tc_workspace_size(const ssd_attn_args*) { return sizeof(WsHeader); }

int attn_tc_launch(const ssd_attn_args* a, void* ws, cudaStream_t s) {
  const int NT = a->NB * a->Dmax;
  const int G = a->Hq / a->Hkv;
  const int mtiles = (NT * G + tc::BM - 1) / tc::BM;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(tc::k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(tc::kSmemBytes));
  });
  if (attr_err != cudaSuccess) return SSD_ERR_CUDA;
  int S = 1, chunk = tc::BN;
  tc::choose_split(a, mtiles, &S, &chunk);
  CUtensorMap mk, mv, mkc, mvc;
  const uint64_t rows = static_cast<uint64_t>(a->B) * a->Hkv * a->P_max;
  const uint64_t slots = static_cast<uint64_t>(a->B) * NT;
  if (!tc::make_kv_map(&mk, a->k_cache, rows) || !tc::make_kv_map(&mv, a->v_cache, rows) ||
      !tc::make_cand_map(&mkc, a->k_cand, slots, a->Hkv) || !tc::make_cand_map(&mvc, a->v_cand, slots, a->Hkv))
    return SSD_ERR_CUDA;

  AttnParams p{};
  p.q = a->q; p.k_cache = a->k_cache; p.v_cache = a->v_cache; p.k_cand = a->k_cand; p.v_cand = a->v_cand;
  p.out = a->out; p.prefix_len = a->prefix_len; p.blk_len = a->blk_len;
  p.B = a->B; p.NB = a->NB; p.Dmax = a->Dmax; p.Hq = a->Hq; p.Hkv = a->Hkv; p.P_max = a->P_max;
  const float scale = a->scale != 0.f ? a->scale : 1.f / sqrtf(static_cast<float>(a->dh));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.S = S;
  p.chunk = chunk;
  p.out_f32 = (a->out_dtype == SSD_F32) ? 1 : 0;
  p.hdr = reinterpret_cast<WsHeader*>(ws);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(S), static_cast<unsigned>(mtiles), static_cast<unsigned>(a->B * a->Hkv));
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = tc::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  {
    KernelTimer timer(SSD_KERNEL_VERIFY_ATTN, s);
    if (cudaLaunchKernelEx(&cfg, tc::k_attn_tc, mk, mv, mkc, mvc, p) != cudaSuccess) return SSD_ERR_CUDA;
  }
  count_launch(1);
  return check_launch();
}

}  // namespace ssd
