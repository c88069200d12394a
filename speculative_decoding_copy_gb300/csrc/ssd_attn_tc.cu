// Verification attention for bf16, head dim 128, on the tensor cores.
//
// SwitchSD page, "무엇과 다른가": a candidate token attends to the whole prefix
// and to the earlier tokens of its own candidate, never to another candidate.
// Every candidate token of a sequence sees the same prefix keys, so for one kv
// head the G query heads of all NT candidate slots pack into NT*G rows of one
// dense product with each key tile. A CTA owns 128 packed rows (the M of the
// MMA) and one split of the prefix; the S CTAs of a row tile form a thread-block
// cluster, rank 0 also takes the own-block keys as masked tiles, and the splits
// are merged on chip through distributed shared memory.
//
// Per CTA (384 threads, one CTA per SM, all 512 TMEM columns):
//   warps 0-3  one thread per packed row: online softmax of a 128-key tile read
//              from TMEM (tcgen05.ld), masked to a contiguous key range; O is
//              rescaled in TMEM when the row max grows; P goes back to TMEM as
//              bf16 pairs (tcgen05.st) over the first half of the tile's S
//              buffer, where the P V product reads it as its A operand;
//   warp 4     TMEM allocation, then the TMA producer of Q (a 4-D map lays the G
//              heads of 128/G tokens out as 128 rows) and of the K tiles;
//   warp 6     the TMA producer of the V tiles. K and V tiles of 128 keys (two
//              64-wide halves of the head dim, 128-byte swizzle) share a 3-stage
//              ring, from the prefix cache (2-D map) or the candidate keys (3-D
//              map); a stage's K half is refilled once Q K^T of its tile is done,
//              its V half once P V is;
//   warp 5     the single MMA-issuing thread: S = Q K^T (M128 N128, eight K16
//              steps, both operands in shared memory) into one of three TMEM
//              buffers, three tiles ahead of the softmax, and O += P V (M128
//              N128, eight K16 steps, A from TMEM, V MN-major in shared memory);
//   warps 6-11 (warp 6 after its loads) add threads to the merge.
// TMEM columns: S buffers 0-127, 128-255 and 256-383 (P of a tile in the first 64
// columns of its buffer), O 384-511.
// Merge: each row's un-normalised O is staged in the CTA's idle ring as 16-bit
// integers, one power-of-two scale per 64-column half (warps 0-3 stage columns
// 0-63, warps 6-9 columns 64-127), with the row's max and sum; after a cluster
// barrier (every ring is idle) S-1 threads each send one other CTA of the
// cluster the rows it owns (128/S each) with one bulk copy completing on that
// CTA's mbarrier, and every owner thread weights and sums the S copies of one
// row's 16 columns and writes them for tokens that exist. Which tokens exist
// comes from the retrieval, so only warp 4's read of it waits for the preceding
// kernel (griddepcontrol.wait).
// Every mbarrier wait is bounded (about 2^32 clocks); on expiry the CTA
// records SSD_ERR_TIMEOUT in the workspace header, skips the remaining waits,
// frees its TMEM and exits through the cluster barriers.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "ssd_attn.cuh"
#include "ssd_tc.cuh"

namespace ssd {
namespace tc {

constexpr int DH = 128;
constexpr int BM = 128;                   // packed rows per CTA
constexpr int BN = 128;                   // keys per tile
constexpr int STAGES = 3;                 // K/V ring depth
constexpr int kThreads = 384;            // 6 role warps + 6 that join for the merge
constexpr uint32_t kTmemCols = 512;
constexpr int SBUF = 3;                   // S buffers: S runs three tiles ahead of the softmax
constexpr uint32_t TM_S = 0;              // SBUF S buffers of BN columns; P of a tile overwrites
                                          // the first BN/2 columns of its S buffer (bf16 pairs)
constexpr uint32_t TM_O = SBUF * BN;      // O: DH columns
static_assert(TM_O + DH <= kTmemCols, "TMEM budget");
constexpr uint32_t kHalf = 128 * 128;     // 128 rows x 64 bf16, one 128-byte-swizzled half: 16 KB
constexpr uint32_t kStage = 4 * kHalf;    // K and V tiles, two halves each: 64 KB
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_RING = OFF_Q + 2 * kHalf;
constexpr uint32_t OFF_BAR = OFF_RING + STAGES * kStage;
constexpr uint32_t kBarBytes = 1024;
constexpr uint32_t kSmemBytes = OFF_BAR + kBarBytes + 1024;   // + slack to align the base to 1024
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr unsigned long long kWaitClocks = 1ull << 32;
struct Bars {
  uint64_t full_k[STAGES], full_v[STAGES], empty_k[STAGES], empty_v[STAGES];
  uint64_t q_full;
  uint64_t s_full[SBUF], p_full[SBUF], pv_done[2];
  uint64_t recv_full;                     // every other split's copy of the owned rows has arrived
  uint32_t tmem_base;
  int failed;
  uint8_t exists[BM];                     // merged row belongs to a token that exists
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block");

// ------------------------------------------------------------------ waits
// Bounded wait; false once this CTA has given up (then every later wait returns at once).
__device__ __forceinline__ bool mbar_wait(Bars& bars, uint64_t* bar, uint32_t parity, WsHeader* hdr, int where) {
  return mbar_wait_bounded(bar, parity, &bars.failed, hdr, where, kWaitClocks);
}

// Merged rows travel as 16-bit integers (two per word, low half first) on the ALU pipes.
// Encode: for |x| < 2^22, x + 1.5*2^23 rounded to fp32 is an integer whose low 16 bits are
// round(x) in two's complement; one FFMA per value scales and rounds.
__device__ __forceinline__ uint32_t pack_i16(float x0, float x1, float s) {
  const uint32_t a = __float_as_uint(fmaf(x0, s, 12582912.f)), b = __float_as_uint(fmaf(x1, s, 12582912.f));
  return __byte_perm(a, b, 0x5410);
}

// Decode: flipping the sign bit maps n to n + 2^15 in [0, 2^16); under the exponent of 2^23
// that is the fp32 2^23 + 2^15 + n, from which one FADD recovers n exactly.
__device__ __forceinline__ float2 unpack_i16(uint32_t w) {
  const uint32_t f = w ^ 0x80008000u;
  return make_float2(__uint_as_float(__byte_perm(f, 0x4B000000u, 0x7610)) - 8421376.f,
                     __uint_as_float(__byte_perm(f, 0x4B000000u, 0x7632)) - 8421376.f);
}


// Softmax pieces on 64 columns of one row's S in TMEM. MASK: only columns in
// [lo, hi) (relative to the chunk) count; the others act as -inf.
template <bool MASK>
__device__ __forceinline__ float chunk_max(uint32_t taddr, int lo, int hi) {
  uint32_t v[64];
  tmem_ld32(taddr, v);
  tmem_ld32(taddr + 32, v + 32);
  tmem_wait_ld();
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < 64; ++c) {
    const float x = __uint_as_float(v[c]);
    if (!MASK || (c >= lo && c < hi)) m4[c & 3] = fmaxf(m4[c & 3], x);
  }
  return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
}

// p = 2^(s*sl2 - mref) rounded to bf16, stored as 32 bf16 pairs at `paddr`;
// returns the sum of the rounded values (what the P V product multiplies).
template <bool MASK>
__device__ __forceinline__ float chunk_exp(uint32_t saddr, uint32_t paddr, int lo, int hi, float sl2, float mref) {
  uint32_t v[64];
  tmem_ld32(saddr, v);
  tmem_ld32(saddr + 32, v + 32);
  tmem_wait_ld();
  uint32_t pk[32];
  float rs[4] = {0.f, 0.f, 0.f, 0.f};
  if (mref > -INFINITY) {
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
      float p0 = ex2_approx(fmaf(__uint_as_float(v[c]), sl2, -mref));
      float p1 = ex2_approx(fmaf(__uint_as_float(v[c + 1]), sl2, -mref));
      if (MASK) {
        if (c < lo || c >= hi) p0 = 0.f;
        if (c + 1 < lo || c + 1 >= hi) p1 = 0.f;
      }
      const uint32_t w = pack_bf16(p0, p1);
      pk[c / 2] = w;
      rs[(c >> 1) & 1] += __uint_as_float(w << 16);
      rs[2 + ((c >> 1) & 1)] += __uint_as_float(w & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int c = 0; c < 32; ++c) pk[c] = 0u;       // no allowed key yet in this row
  }
  tmem_st32(paddr, pk);
  return (rs[0] + rs[1]) + (rs[2] + rs[3]);
}

// ------------------------------------------------------------------ kernel
constexpr int kMaxSplit = 8;              // cluster size limit (portable)
// one split's partial row as sent to its owner: O as 128 16-bit integers, round(O 2^(14-e)) with
// e per 64-column half such that its max |O| lies in [2^(e-1), 2^e), then the row's max and
// sum and the two halves' 2^(e-14) as fp32 (16-byte units)
constexpr int kRowB = 2 * DH + 16;
static_assert((2 * BM + kMaxSplit) * kRowB + BM * kMaxSplit * 4 <= static_cast<int>(STAGES * kStage),
              "merge buffers fit in the ring");

// grid (S, row tiles, B*Hkv), cluster (S, 1, 1): the S CTAs of one row tile split
// the prefix; cluster rank 0 also takes the own-block (candidate) keys.
__global__ void __launch_bounds__(kThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
          const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_kc,
          const __grid_constant__ CUtensorMap tmap_vc, AttnParams p) {
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
  int P = p.prefix_len[b];
  // a prefix longer than the cache would read another sequence's (or head's) keys
  if (!in_range(P, (p.block_table != nullptr ? 128LL * p.pages_per_seq : p.P_max) + 1, p.hdr, 27)) P = 0;
  // split 0 also takes the own-block tiles, so its share of the prefix is shorter
  const int k0 = split == 0 ? 0 : p.chunk0 + (split - 1) * p.chunk;
  const int k1 = min(P, k0 + (split == 0 ? p.chunk0 : p.chunk));
  const int nP = k1 > k0 ? (k1 - k0 + BN - 1) / BN : 0;
  // candidate slots of this row tile: from the start of its first token's block to its last token
  const int t_first = r0 / G;
  const int t_last = min(NT - 1, (r0 + BM - 1) / G);
  const int s_base = (t_first / p.Dmax) * p.Dmax;
  const int nC = (split == 0 && t_first < NT) ? (t_last + 1 - s_base + BN - 1) / BN : 0;
  const int nT = nC + nP;
  // rows of this tile that exist (rv) and those merged by this CTA: [rb, rb + nr)
  const int rv = min(BM, rows_total - r0);
  const int rpc = (rv + S - 1) / S;
  const int rb = split * rpc, nr = max(0, min(rv, rb + rpc) - rb);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // skip_absent 2: blk_len was complete when this grid launched, so nothing waits for the
  // kernel before this one except the grid's last CTA, before it ends (the grid then still
  // completes after it)
  const bool last_cta = blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1;
  if (p.skip_absent) {
    // a tile none of whose rows belongs to a present token is skipped; the S CTAs of a
    // cluster hold the same rows, so they all leave here together, before any barrier
    if (p.skip_absent == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
    int any = 0;
    for (int i = tid; i < rv; i += kThreads) {
      const int tt = (r0 + i) / G;
      any |= (tt % p.Dmax) < __ldcg(p.blk_len + b * p.NB + tt / p.Dmax) ? 1 : 0;
    }
    if (!__syncthreads_or(any)) {
      if (p.skip_absent == 2 && last_cta && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      return;
    }
  }
  if (warp == 4 && lane == 0) {
    // the descriptors are fetched on first use: start those fetches before the first copy
    prefetch_tmap(&tmap_q);
    if (nP > 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
    }
    if (nC > 0) {
      prefetch_tmap(&tmap_kc);
      prefetch_tmap(&tmap_vc);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars.full_k[s], 1);
      mbar_init(&bars.full_v[s], 1);
      mbar_init(&bars.empty_k[s], 1);
      mbar_init(&bars.empty_v[s], 1);
    }
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.recv_full, 1);
    for (int i = 0; i < SBUF; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], BM);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&bars.pv_done[i], 1);
    bars.failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  float m = -INFINITY, l = 0.f;            // softmax rows: reference max (log2 units) and sum

  if (warp < 4) {
    // ---------------------------------------------------------- softmax rows
    // this thread's packed row: token t, allowed own-block slots [c_lo, t]
    const int r = r0 + tid;
    const bool row_ok = r < rows_total;
    const int t = row_ok ? r / G : 0;
    const int c_lo = (t / p.Dmax) * p.Dmax;
    const float sl2 = p.scale_log2;
    for (int j = 0; j < nT; ++j) {
      const int sb = j % SBUF;
      mbar_wait(bars, &bars.s_full[sb], (j / SBUF) & 1, p.hdr, 10);
      tc_fence_after();
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
      const bool full = v_lo <= 0 && v_hi >= BN;
      const uint32_t sc = tmem + TM_S + sb * BN + lane_off;
      // pass 1: row max over the allowed columns
      float mx = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < BN / 64; ++h)
        mx = fmaxf(mx, full ? chunk_max<false>(sc + h * 64, 0, 0) : chunk_max<true>(sc + h * 64, v_lo - h * 64, v_hi - h * 64));
      // reference max only moves when the row max grows by more than 2^8
      const float m_new = fmaxf(m, mx * sl2);
      const bool need = m_new > m + 8.f;
      const float mref = need ? m_new : m;
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      // pass 2: P = 2^(s*scale - mref) as bf16 pairs into the first BN/2 columns of the
      // same buffer (64 columns of S are read before their 32 columns of P are written, and
      // the columns written hold S already read), and its row sum
      float rs = 0.f;
#pragma unroll 1
      for (int h = 0; h < BN / 64; ++h)
        rs += full ? chunk_exp<false>(sc + h * 64, sc + h * 32, 0, 0, sl2, mref)
                   : chunk_exp<true>(sc + h * 64, sc + h * 32, v_lo - h * 64, v_hi - h * 64, sl2, mref);
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O holds the sum up to tile j-1: wait for its last MMA, then rescale
        mbar_wait(bars, &bars.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.hdr, 11);
        tc_fence_after();
#pragma unroll 1
        for (int q = 0; q < DH / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tmem + TM_O + lane_off + q * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tmem + TM_O + lane_off + q * 32, o);
        }
      }
      l = l * alpha + rs;
      m = mref;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars.p_full[sb]);
    }
    if (nT > 0) {
      mbar_wait(bars, &bars.pv_done[(nT - 1) & 1], ((nT - 1) >> 1) & 1, p.hdr, 13);
      tc_fence_after();
    }
  } else if (warp == 4 || warp == 6) {
    // ---------------------------------------------------------- TMA producers
    // warp 4 loads Q and the K tiles, warp 6 the V tiles: a K slot is free once the
    // S = Q K^T product of its tile has completed, a V slot only after P V, so the K of
    // a later tile is not held back behind the V of an earlier one
    const bool kside = warp == 4;
    if (lane == 0 && nT > 0) {
      if (kside) {
        mbar_expect_tx(&bars.q_full, 2 * kHalf);
        const int qz = b * NT + t_first;                   // rows past the sequence are masked or zero
        tma_load_4d(sbase + OFF_Q, &tmap_q, 0, 0, kvh, qz, &bars.q_full);
        tma_load_4d(sbase + OFF_Q + kHalf, &tmap_q, 64, 0, kvh, qz, &bars.q_full);
      }
      const int y0 = p.block_table != nullptr ? 0 : (b * p.Hkv + kvh) * static_cast<int>(p.P_max) + k0;
      const CUtensorMap* cand_map = kside ? &tmap_kc : &tmap_vc;
      const CUtensorMap* pref_map = kside ? &tmap_k : &tmap_v;
      for (int j = 0; j < nT; ++j) {
        const int s = j % STAGES;
        uint64_t* empty = kside ? &bars.empty_k[s] : &bars.empty_v[s];
        uint64_t* full = kside ? &bars.full_k[s] : &bars.full_v[s];
        if (j >= STAGES) mbar_wait(bars, empty, ((j / STAGES) - 1) & 1, p.hdr, kside ? 20 : 21);
        if (bars.failed) break;
        const uint32_t dst = sbase + OFF_RING + s * kStage + (kside ? 0u : 2 * kHalf);
        mbar_expect_tx(full, 2 * kHalf);
        if (j < nC) {
          const int z = b * NT + s_base + j * BN;          // candidate slot (rows past NT are masked)
          tma_load_3d(dst, cand_map, 0, kvh, z, full);
          tma_load_3d(dst + kHalf, cand_map, 64, kvh, z, full);
        } else {
          int y = y0 + (j - nC) * BN;
          if (p.block_table != nullptr) {
            // paged cache: this tile of 128 keys is one page; rows (page, kv head, 0..127)
            int pg = __ldg(p.block_table + static_cast<int64_t>(b) * p.pages_per_seq + (k0 + (j - nC) * BN) / BN);
            if (pg < 0 || pg >= p.num_pages) {
              record_error(p.hdr, SSD_ERR_DEVICE, 26);
              pg = 0;
            }
            y = (pg * p.Hkv + kvh) * BN;
          }
          tma_load_2d(dst, pref_map, 0, y, full);
          tma_load_2d(dst + kHalf, pref_map, 64, y, full);
        }
      }
    }
    __syncwarp();                                   // warp 6 joins the merge converged
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nT > 0) {
      constexpr uint32_t idS = idesc_bf16(false, BN), idPV = idesc_bf16(true, DH);
      // S[jj % SBUF] = Q K_jj^T : M128 N128, eight K16 steps over the head dim; its K slot is
      // free once these products complete
      auto issue_S = [&](int jj) {
        const int s = jj % STAGES;
        mbar_wait(bars, &bars.full_k[s], (jj / STAGES) & 1, p.hdr, 31);
        tc_fence_after();
        const uint32_t kb = sbase + OFF_RING + s * kStage;
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const uint64_t a = sw128_desc(sbase + OFF_Q + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(kb + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
          mma_bf16(tmem + TM_S + (jj % SBUF) * BN, a, bd, idS, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[jj % SBUF]);
        mma_commit(&bars.empty_k[s]);
      };
      mbar_wait(bars, &bars.q_full, 0, p.hdr, 30);
      for (int jj = 0; jj < SBUF && jj < nT; ++jj) issue_S(jj);
      for (int j = 0; j < nT; ++j) {
        // O += P_j V_j : M128 N128 (head dim), eight K16 steps over the tile's keys, P from TMEM
        const int s = j % STAGES;
        mbar_wait(bars, &bars.p_full[j % SBUF], (j / SBUF) & 1, p.hdr, 34);
        mbar_wait(bars, &bars.full_v[s], (j / STAGES) & 1, p.hdr, 35);
        tc_fence_after();
        const uint32_t vb = sbase + OFF_RING + s * kStage + 2 * kHalf;
        const uint32_t pa = tmem + TM_S + (j % SBUF) * BN;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t bd = sw128_desc(vb + ks * 16 * 128, kHalf, 1024);
          mma_bf16_ts(tmem + TM_O, pa + ks * 8, bd, idPV, (j > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(&bars.pv_done[j & 1]);
        mma_commit(&bars.empty_v[s]);
        // S of tile j+SBUF into the buffer that holds P_j: the products of one thread run in
        // the order issued, so the P V product above has read P_j before it is overwritten
        if (j + SBUF < nT) issue_S(j + SBUF);
      }
    }
  }

  // ---- merge the S splits of every row in the CTA that owns it
  // Each row's partial O is staged in this CTA's idle ring as 16-bit integers, each 64-column
  // half scaled by its own power of two (so that its max |O| maps into [2^13, 2^14)), with
  // the row's max, sum and the two inverse scales; warps 0-3 stage columns 0-63 and warps 6-9
  // (which share the TMEM lane quarters) columns 64-127. After a cluster barrier (every ring
  // is idle) S-1 threads each send one other CTA the rows it owns with one bulk copy,
  // completing on that CTA's mbarrier. Every owner thread then weights and sums the S copies
  // (its own split's rows where they were staged) and writes the rows of tokens that exist.
  // (Owners reading the peers' staged rows in place with distributed shared memory loads,
  // with a second cluster barrier before exit, made the step 2 us slower.)
  // Ring layout (bytes): staged rows [BM][kRowB], received rows [sender split][rpc][kRowB].
  uint8_t* stage = smem + OFF_RING;
  uint8_t* recv = stage + BM * kRowB;
  auto part = [&](int c, int i) -> const uint8_t* {
    return c == split ? stage + (rb + i) * kRowB : recv + (c * rpc + i) * kRowB;
  };
  if (warp < 4 || (warp >= 6 && warp < 10)) {
    const int half = warp < 4 ? 0 : 1;
    const int row = (warp & 3) * 32 + lane;          // this warp's TMEM lane quarter
    const uint32_t oa = tmem + TM_O + (static_cast<uint32_t>((warp & 3) * 32) << 16) + half * 64;
    // warps 6-9 read O once warps 0-3 have seen the last P V product complete (a parity
    // wait on pv_done is only valid for a waiter at most one phase behind, as those are)
    tc_fence_before();
    asm volatile("bar.sync 1, 256;" ::: "memory");
    tc_fence_after();
    // max |O| of this half row, then round(O 2^(14-e)) as 16-bit pairs
    uint32_t o[64];
    if (nT > 0) {
      tmem_ld32(oa, o);
      tmem_ld32(oa + 32, o + 32);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 64; ++e) o[e] = 0u;
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 64; ++e) amax = fmaxf(amax, fabsf(__uint_as_float(o[e])));
    // amax in [2^k, 2^(k+1)): e = k + 1; halves below 2^-100 keep e = 0 (they round to zero)
    const int k = (amax >= 0x1p-100f) ? static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127 : -1;
    const int ex = min(k, 125) + 1;
    const float scale = __uint_as_float(static_cast<uint32_t>(127 + 14 - ex) << 23);
    const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - 14 + ex) << 23);
    uint4* dst = reinterpret_cast<uint4*>(stage + row * kRowB + half * DH);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pk[e] = pack_i16(__uint_as_float(o[8 * u + 2 * e]), __uint_as_float(o[8 * u + 2 * e + 1]), scale);
      dst[u] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    float* tail = reinterpret_cast<float*>(stage + row * kRowB + 2 * DH);
    if (half == 0) {
      tail[0] = m;
      tail[1] = l;
    }
    tail[2 + half] = inv_scale;
    fence_async_smem();                              // the bulk copies read what the threads wrote
  }
  if (tid == 0) mbar_expect_tx(&bars.recv_full, static_cast<uint32_t>((S - 1) * nr * kRowB));
  tc_fence_before();
  __syncwarp();
  cluster_sync();                                   // every CTA is past its main loop: the rings are idle
  tc_fence_after();
  if (tid < S - 1) {
    // rows [c*rpc, c*rpc + n_c) go to cluster rank c, into its slot for this split; each
    // rank starts with a different destination, so that no CTA receives from all at once
    const int c = (split + 1 + tid) % S;
    const int n_c = min(rv, (c + 1) * rpc) - c * rpc;
    if (n_c > 0) {
      const uint32_t dst = map_peer(smem_u32(recv + split * rpc * kRowB), static_cast<uint32_t>(c));
      const uint32_t bar = map_peer(smem_u32(&bars.recv_full), static_cast<uint32_t>(c));
      bulk_copy_to_peer(dst, smem_u32(stage + c * rpc * kRowB), static_cast<uint32_t>(n_c * kRowB), bar);
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  if (warp == 4) {
    // which owned rows belong to tokens that exist: blk_len comes from the retrieval, which
    // precedes this kernel in the stream (with all_rows every slot's row is written)
    if (!p.all_rows && p.skip_absent != 2) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = lane; i < nr; i += 32) {
      const int gr = r0 + rb + i;
      const int tt = gr / G;
      bars.exists[i] = p.all_rows ? 1 : ((tt % p.Dmax) < __ldcg(p.blk_len + b * p.NB + tt / p.Dmax) ? 1 : 0);
    }
  }
  __syncthreads();
  // one thread per (owned row, 16-column group): every split's max, sum, scale and 32 bytes
  // of the row loaded together, the weights 2^(m_c - M) / sum_c l_c 2^(m_c - M) computed here
  for (int it = tid; it < nr * (DH / 16); it += kThreads) {
    const int i = it / (DH / 16), cg = it % (DH / 16);
    if (!bars.exists[i]) continue;
    if (!mbar_wait(bars, &bars.recv_full, 0, p.hdr, 40)) continue;
    float4 tl[kMaxSplit];
    uint4 h[kMaxSplit][2];
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) {
      tl[c] = make_float4(-INFINITY, 0.f, 0.f, 0.f);
      if (c < S) {
        const uint8_t* pr = part(c, i);
        tl[c] = *reinterpret_cast<const float4*>(pr + 2 * DH);
        const uint4* src = reinterpret_cast<const uint4*>(pr + cg * 32);
        h[c][0] = src[0];
        h[c][1] = src[1];
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) M = fmaxf(M, tl[c].x);
    float fw[kMaxSplit], L = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) {
      fw[c] = tl[c].x > -INFINITY ? ex2_approx(tl[c].x - M) : 0.f;
      L = fmaf(tl[c].y, fw[c], L);
    }
    // a row with no allowed key is not a present token: nothing written
    if (bars.failed || !(L > 0.f)) continue;
    const float inv = __frcp_rn(L);
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c) {
      if (c < S) {
        const float f = fw[c] * inv * (cg < 4 ? tl[c].z : tl[c].w);
        const uint32_t w[8] = {h[c][0].x, h[c][0].y, h[c][0].z, h[c][0].w, h[c][1].x, h[c][1].y, h[c][1].z, h[c][1].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 v = unpack_i16(w[e]);
          acc[2 * e] = fmaf(f, v.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(f, v.y, acc[2 * e + 1]);
        }
      }
    }
    const int gr = r0 + rb + i;
    const int tt = gr / G, hh = kvh * G + (gr - tt * G);
    const int64_t o_off = ((static_cast<int64_t>(b) * NT + tt) * p.Hq + hh) * DH + cg * 16;
    if (p.out_f32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o_off);
#pragma unroll
      for (int u = 0; u < 4; ++u) o[u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
    } else {
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o_off);
      o[0] = make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                        pack_bf16(acc[6], acc[7]));
      o[1] = make_uint4(pack_bf16(acc[8], acc[9]), pack_bf16(acc[10], acc[11]), pack_bf16(acc[12], acc[13]),
                        pack_bf16(acc[14], acc[15]));
    }
  }
  // this CTA's outgoing copies have finished reading its staged rows before it exits
  if (tid < S - 1) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");

  // teardown: every role is done with TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  // with all_rows (or skip_absent 2) nothing above waited for the kernel before this one: one
  // thread waits for it here, after the rows are written, so that this grid still completes
  // after it
  if ((p.all_rows || (p.skip_absent == 2 && last_cta)) && tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ host
static bool make_kv_map(CUtensorMap* map, const void* base, uint64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(DH), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(DH) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BN)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [B*NT][Hq][dh] as a 4-D tensor (dh, head in group, kv head, token): a box of
// 128/G tokens of one kv head's G heads lands as the 128 packed rows of a row tile
static bool make_q_map(CUtensorMap* map, const void* base, uint64_t tokens, int G, int Hkv) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(DH), static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(Hkv),
                              tokens};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(DH) * 2, static_cast<cuuint64_t>(G) * DH * 2,
                                 static_cast<cuuint64_t>(G) * Hkv * DH * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), 1, static_cast<cuuint32_t>(BM / G)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// candidate K or V [B*NT][Hkv][dh] as a 3-D tensor (dh, kv head, slot): a box of
// BN slots of one kv head lands as a [BN][64] tile like a prefix tile
static bool make_cand_map(CUtensorMap* map, const void* base, uint64_t slots, int Hkv) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(DH), static_cast<cuuint64_t>(Hkv), slots};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(DH) * 2, static_cast<cuuint64_t>(Hkv) * DH * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(BN)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How many clusters of S CTAs can be resident at once (0 if the query fails).
static int max_active_clusters(int S) {
  static int cache[kMaxSplit + 1][kMaxDevices];
  static bool done[kMaxSplit + 1][kMaxDevices];
  static std::mutex mu;
  const int dev = current_device();
  if (dev < 0) return 0;
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

// Splits (cluster size <= 8): minimise (waves of clusters) x (tiles per split + fixed
// cost). Split 0 also takes the own-block tiles of its row tile (at most nc of them),
// so it gets nc fewer prefix tiles than the others.
static void choose_split(const ssd_attn_args* a, int mtiles, int* S_out, int* chunk_out, int* chunk0_out) {
  const long long groups = static_cast<long long>(a->B) * a->Hkv * mtiles;   // clusters in the grid
  const long long nkt = a->P_max > 0 ? (a->P_max + BN - 1) / BN : 1;
  const int G = a->Hq / a->Hkv;
  // a row tile spans BM/G tokens; with the start of the first one's block, at most this many slots
  const long long nc = (BM / G + a->Dmax - 1 + BN - 1) / BN;
  long long best_cost = -1;
  int best_S = 1;
  for (int S = 1; S <= kMaxSplit && S <= nkt; ++S) {
    int active = max_active_clusters(S);
    if (active <= 0) continue;
    if (a->max_ctas > 0) {
      // a grid of at most max_ctas CTAs (whole clusters, at least one per row tile)
      if (S > 1 && groups * S > a->max_ctas) continue;
      active = static_cast<int>(std::min<long long>(active, std::max<long long>(1, a->max_ctas / S)));
    }
    const long long tiles = (nkt + 2 * nc + S - 1) / S;
    const long long waves = (groups + active - 1) / active;
    const long long cost = waves * (tiles + 2) * 16 + S;   // +2 tiles: prologue and merge
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_S = S;
    }
  }
  // a masked candidate tile costs about two prefix tiles (per-element masks in both passes)
  const long long tiles = (nkt + 2 * nc + best_S - 1) / best_S;
  *S_out = best_S;
  *chunk_out = static_cast<int>(tiles * BN);
  *chunk0_out = static_cast<int>((tiles > 2 * nc ? tiles - 2 * nc : 0) * BN);
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
  if (a->block_table == nullptr && static_cast<long long>(a->B) * a->Hkv * a->P_max >= (1LL << 31)) return false;
  if (static_cast<long long>(a->B) * a->NB * a->Dmax >= (1LL << 31)) return false;
  if (a->B * a->Hkv > 65535) return false;
  // Q rows arrive by TMA as whole tokens: G must divide the 128 rows of a tile
  const int G = a->Hq / a->Hkv;
  if (G < 1 || G > 64 || (tc::BM % G) != 0) return false;
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
  static std::once_flag attr_once[kMaxDevices];
  static cudaError_t attr_err[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return SSD_ERR_CUDA;
  std::call_once(attr_once[dev], [dev] {
    attr_err[dev] = cudaFuncSetAttribute(tc::k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tc::kSmemBytes));
  });
  if (attr_err[dev] != cudaSuccess) return SSD_ERR_CUDA;
  int S = 1, chunk = tc::BN, chunk0 = tc::BN;
  tc::choose_split(a, mtiles, &S, &chunk, &chunk0);
  CUtensorMap mq, mk, mv, mkc, mvc;
  // K/V rows of the 2-D maps: [B][Hkv][P_max] contiguous, or [num_pages][Hkv][128] pages
  const uint64_t rows = a->block_table != nullptr ? static_cast<uint64_t>(a->num_pages) * a->Hkv * tc::BN
                                                  : static_cast<uint64_t>(a->B) * a->Hkv * a->P_max;
  const uint64_t slots = static_cast<uint64_t>(a->B) * NT;
  if (!tc::make_q_map(&mq, a->q, slots, G, a->Hkv) || !tc::make_kv_map(&mk, a->k_cache, rows) || !tc::make_kv_map(&mv, a->v_cache, rows) ||
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
  p.chunk0 = chunk0;
  p.out_f32 = (a->out_dtype == SSD_F32) ? 1 : 0;
  p.block_table = a->block_table;
  p.pages_per_seq = a->pages_per_seq;
  p.num_pages = a->num_pages;
  p.skip_absent = a->skip_absent;
  p.all_rows = a->all_rows;
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
    if (cudaLaunchKernelEx(&cfg, tc::k_attn_tc, mq, mk, mv, mkc, mvc, p) != cudaSuccess) return SSD_ERR_CUDA;
  }
  count_launch(1);
  return check_launch();
}

}  // namespace ssd
