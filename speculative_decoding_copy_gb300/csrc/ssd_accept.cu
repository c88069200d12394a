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
//   k_vocab_stats   every warp streams whole pieces of 2048 entries of the rows
//                   some token needs (16-byte loads, all in flight together) and
//                   reduces each to max, argmax (greedy only; lowest index on
//                   ties) and sum of 2^((l - max) log2 e) with warp shuffles; in
//                   the early mode it streams every row a block length can reach
//                   without waiting for the kernel before it (it only stores after
//                   that wait), and only its last CTA, which takes no pieces, waits
//                   before letting the next kernel launch;
//   k_accept_finish_wide / k_accept_finish_batch  per sequence (one cluster each):
//                   merges every needed row's pieces, runs the acceptance test
//                   of every candidate token and picks the longest accepted block,
//                   and in sample mode draws the final token from the integer
//                   weights of the stop row (chunk sums exchanged through
//                   distributed shared memory, then the chunk, the lane and the
//                   entry that hold the threshold);
//   k_probs_out     optional diagnostic copy of p for every needed row.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "ssd_accept.cuh"

namespace ssd {

constexpr int kVocabThreads = 256;
constexpr int kMaxRows = 1024;          // 1 + NB*Dmax + K
constexpr int kMaxSlots = 1024;         // NB*Dmax
constexpr int kSampleChunk = 512;       // stop-row entries per warp of the final draw
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

// (m, s) += (m2, s2) with one exponential and no branch: the side with the larger max keeps
// its sum as is, the other is scaled by 2^((min - max) log2 e) (0 when the smaller max is
// -inf). Both lanes of a shuffle pair form the same two terms, so they agree bit for bit.
__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2) {
  const float hi = fmaxf(m, m2), lo = fminf(m, m2);
  const float e = lo > -INFINITY ? ex2_approx((lo - hi) * kLog2e) : 0.f;
  s = m2 > m ? fmaf(s, e, s2) : fmaf(s2, e, s);
  m = hi;
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
// k_vocab_stats: every warp streams whole pieces of 2048 entries of the rows
// some token needs (8 KB of fp32 or 4 KB of bf16: 16 or 8 16-byte loads per
// lane, all in flight together) and reduces each piece alone with warp
// shuffles; two CTAs of 8 warps per SM (one of 16 warps under max_ctas) keep up to
// 128 KB of loads in flight per SM.
constexpr int kPieceElems = 2048;
template <bool BF16>
struct Piece {
  static constexpr int kEPV = BF16 ? 8 : 4;                 // entries per 16-byte vector
  static constexpr int kVec = kPieceElems / kEPV / 32;     // 16-byte loads per lane
};

// element e (0..EPV-1) of a 16-byte vector
template <bool BF16>
__device__ __forceinline__ float vec_elem(const uint4& u, int e) {
  const uint32_t w = e < (BF16 ? 2 : 1) ? u.x : e < (BF16 ? 4 : 2) ? u.y : e < (BF16 ? 6 : 3) ? u.z : u.w;
  if (BF16) return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  return __uint_as_float(w);
}

template <bool BF16, bool AMAX, bool FULL>
__device__ __forceinline__ RowStat reduce_vecs(const uint4 (&v)[Piece<BF16>::kVec], int n, int e0, int probs);

// One warp's statistics of the piece of n elements starting at element e0 of `row`:
// max, sum of 2^((x - max) log2 e) (not for probabilities) and, with AMAX, the argmax
// (lowest index on ties). VEC: the row is 16-byte aligned with a whole number of
// vectors, so every lane reads 16-byte vectors; missing elements count as -inf.
// FULL: a whole piece (n = kPieceElems), no bounds checks.
template <bool BF16, bool AMAX, bool VEC, bool FULL>
__device__ __forceinline__ RowStat reduce_piece(const void* row, int n, int e0, int probs) {
  constexpr int EPV = Piece<BF16>::kEPV;
  constexpr int kPieceVec = Piece<BF16>::kVec;
  const int lane = threadIdx.x & 31;
  uint4 v[kPieceVec];
  // lane's elements: vector j covers [e0 + (j*32 + lane)*EPV, +EPV)
  if (VEC) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + static_cast<int64_t>(e0) * (BF16 ? 2 : 4));
    const int nv = n / EPV;                 // whole vectors (the row length is a multiple of EPV)
#pragma unroll
    for (int j = 0; j < kPieceVec; ++j) {
      const int vi = j * 32 + lane;
      // streaming loads (evict first): the logits are read once, and the piece statistics
      // this grid writes should stay in L2 for the finish kernel while the rows stream by
      v[j] = (FULL || vi < nv) ? __ldcs(src + vi) : make_uint4(0, 0, 0, 0);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPieceVec; ++j) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const int i = (j * 32 + lane) * EPV + e;
        if (i < n) {
          if (BF16) {
            const uint32_t hbits = __ldg(static_cast<const uint16_t*>(row) + e0 + i);
            w[e >> 1] |= (e & 1) ? (hbits << 16) : hbits;
          } else {
            w[e] = __float_as_uint(__ldg(static_cast<const float*>(row) + e0 + i));
          }
        }
      }
      v[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  return reduce_vecs<BF16, AMAX, FULL>(v, n, e0, probs);
}

// The reduction of reduce_piece on a piece already in registers: lane's vector j holds
// elements [e0 + (j*32 + lane)*EPV, +EPV), those at or past n count as -inf.
template <bool BF16, bool AMAX, bool FULL>
__device__ __forceinline__ RowStat reduce_vecs(const uint4 (&v)[Piece<BF16>::kVec], int n, int e0, int probs) {
  constexpr int EPV = Piece<BF16>::kEPV;
  constexpr int kPieceVec = Piece<BF16>::kVec;
  const int lane = threadIdx.x & 31;
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float av = -INFINITY;
  int ai = 0x7fffffff;
#pragma unroll
  for (int j = 0; j < kPieceVec; ++j) {
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const int i = (j * 32 + lane) * EPV + e;
      const float x = (FULL || i < n) ? vec_elem<BF16>(v[j], e) : -INFINITY;
      if (AMAX) {
        if (x > av) {                       // indices increase along the lane: strict > keeps the lowest
          av = x;
          ai = e0 + i;
        }
      } else {
        m4[e & 3] = fmaxf(m4[e & 3], x);
      }
    }
  }
  float M = AMAX ? av : fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (AMAX) {
      const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
      amax_merge(av, ai, v2, i2);
    }
  }
  float S = 0.f;
  if (!probs && M > -INFINITY) {
    const float c = -M * kLog2e;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kPieceVec; ++j)
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        if (FULL || (j * 32 + lane) * EPV + e < n) s4[e & 3] += ex2_approx(fmaf(vec_elem<BF16>(v[j], e), kLog2e, c));
    S = warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3]));
  }
  return RowStat{M, S, av, ai};
}

// AMAX = false (sample mode, where no decision reads the argmax): max and sum only, half the
// shuffles
template <bool AMAX>
__device__ __forceinline__ RowStat warp_merge_stat(float M, float S, float av, int ai) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
    stat_merge(M, S, m2, s2);
    if (AMAX) {
      const float v2 = __shfl_xor_sync(0xffffffffu, av, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, o);
      amax_merge(av, ai, v2, i2);
    }
  }
  return RowStat{M, S, av, ai};
}

// next task (sequence, row, piece) at or after t, in steps of `step`, whose row some
// token needs (in the early mode every row a block length can reach), or ntask; tasks
// are numbered ((b * NRD) + r) * nch + c
__device__ __forceinline__ int next_task(const AcceptParams& p, int t, int step, int ntask) {
  if (p.early) {
    // every row but the chain block's rows at positions K and beyond, which no block
    // length can reach (the chain block holds at most K tokens)
    const int c0 = p.chain_blk >= 0 ? 1 + p.chain_blk * p.Dmax + p.K : 0;
    const int c1 = p.chain_blk >= 0 ? 1 + (p.chain_blk + 1) * p.Dmax : 0;
    for (; t < ntask; t += step) {
      const int r = (t / p.nch) % p.NRD;
      if (r < c0 || r >= c1) break;
    }
    return t < ntask ? t : ntask;
  }
  for (; t < ntask; t += step) {
    const int br = t / p.nch;
    const int b = br / p.NRD, r = br - b * p.NRD;
    if (row_needed(p, b, r)) break;
  }
  return t;
}

// Every warp of the grid takes the tasks gw, gw + (warps in the grid), ...
// WARPS = 8: two CTAs per SM (the whole-GPU grid); WARPS = 16: one CTA per SM (a grid
// capped to part of the GPU, so that every CTA holds an SM of its own)
template <bool BF16, bool AMAX, int WARPS>
__global__ void __launch_bounds__(32 * WARPS, 16 / WARPS)
k_vocab_stats(AcceptParams p) {
  // blk_len comes from the retrieval; once it is in, the next kernel of the stream may
  // start (its prologue reads the retrieval's outputs, never this kernel's). The early
  // mode reads no blk_len: every CTA but the last lets the next kernel start at once;
  // the last CTA takes no pieces: it waits for the preceding kernel, lets the next one
  // start and leaves. So the next kernel starts only once that kernel (and what it
  // waited for) has completed, and this grid completes only after it: the next kernel's
  // wait then covers them all. (With pieces of its own as well, the waiting CTA, which
  // starts its pieces only after the retrieval, ended about 5 us after the others.)
  // The workspace may still be read by the kernel before this one (the finish kernel of
  // an earlier call on the same workspace, which lets this grid launch at its start), so
  // no CTA writes it before griddepcontrol.wait: in the early mode each warp keeps up to
  // 32 piece results in its lanes and waits only before its first store.
  const bool waiter = p.early && blockIdx.x == gridDim.x - 1;
  bool waited = !p.early || waiter;
  if (waited) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (waiter) return;
  constexpr int es = BF16 ? 2 : 4;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int TW = (gridDim.x - (p.early ? 1 : 0)) * WARPS;    // the early mode's last CTA takes none
  const int ntask = p.nch * p.NRD * p.B;
  const int per = kPieceElems;
  const bool vec_rows = ((p.V * es) & 15) == 0;
  RowStat held{};                     // lane i: the i-th result of this warp, not yet stored
  int64_t held_at = -1;
  int nheld = 0;
  for (int t = next_task(p, gw, TW, ntask); t < ntask; t = next_task(p, t + TW, TW, ntask)) {
    const int br = t / p.nch, c = t - br * p.nch;
    const int b = br / p.NRD, r = br - b * p.NRD;
    const void* row = row_ptr(p, b, r);
    const int e0 = c * per;
    const int n = static_cast<int>(min(static_cast<int64_t>(per), p.V - e0));
    RowStat st;
    if (!vec_rows || !aligned_dev(row, 16)) st = reduce_piece<BF16, AMAX, false, false>(row, n, e0, p.probs);
    else if (n == per) st = reduce_piece<BF16, AMAX, true, true>(row, n, e0, p.probs);
    else st = reduce_piece<BF16, AMAX, true, false>(row, n, e0, p.probs);
    const int64_t at = static_cast<int64_t>(br) * p.nch + c;
    if (!waited && nheld < 32) {      // every lane holds the same st after the warp reduction
      if (lane == nheld) {
        held = st;
        held_at = at;
      }
      ++nheld;
      continue;
    }
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
      if (held_at >= 0) p.part[held_at] = held;
      held_at = -1;
    }
    if (lane == 0) p.part[at] = st;
  }
  if (!waited && nheld > 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (held_at >= 0) p.part[held_at] = held;
  }
}

// ------------------------------------------------------------------ finish
// k_accept_finish_batch: one cluster of C CTAs (C = 1, 2 or 4; chosen so that the
// clusters of the whole batch fit on the GPU at once) per sequence does the rest
// of the step after the row pass: merging every needed row's piece statistics
// (every CTA, one row per warp), the acceptance tests and the choice of block
// (each CTA takes the same decisions from the same data; rank 0 writes them), and
// in sample mode the final draw from the stop row: CTA r owns a contiguous range
// of 512-entry chunks, its warps loop over them summing the exact integer weights
// per chunk, the CTA totals go to every rank through distributed shared memory,
// and the CTA holding the threshold finds the chunk, then the lane, then the
// entry. What needs only the retrieval's outputs and the inputs (token slots,
// their logits and uniforms) is loaded before griddepcontrol.wait, while the row
// pass still runs.
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kSlotsPer = kMaxSlots / kFinThreads;
constexpr int kMaxSampleChunks = 512;       // chunks of a stop row (V <= 262144)
constexpr int kLaneEntries = kSampleChunk / 32;             // contiguous entries per lane per chunk
constexpr int kChunkVec = kLaneEntries / 4;                  // float4 per lane per chunk

struct __align__(16) FinishSmem {
  RowStat st[kMaxRows];                     // merged rows
  long long csum[kMaxSampleChunks][2];      // residual and bonus weight sums of this CTA's chunks
  long long ctasum[4][2];                   // ... of every rank's chunks (clusters of up to 4)
  StopInfo si;                              // the stop row
  int tok_s[kMaxSlots];                     // candidate tokens
  int len_s[256];
  int acc_s[256];
  unsigned char ok_s[kMaxSlots];
  int sel[4];
  int c_star, use_bonus;
  long long t_rem;
};

__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster; orders shared-memory accesses across the cluster
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t cl_map(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}

// row_needed with the (clamped) block lengths in shared memory
__device__ __forceinline__ bool row_needed_s(const AcceptParams& p, const int* len_s, int r) {
  if (r == 0) return true;
  if (r < p.NR) {
    const int sl = r - 1, k = sl / p.Dmax;
    return sl - k * p.Dmax < len_s[k];
  }
  return p.chain_blk >= 0 && (r - p.NR) < len_s[p.chain_blk];
}

// Statistics of the needed rows of sequence b merged from their pieces into st[], every
// warp taking rows warp, warp + nw, ... with the loads of all its rows issued before any
// merge (one round trip to L2 for up to kRowsPerWarp rows of up to 32 kLoadsPerRow pieces);
// rows and pieces beyond that loop.
template <int kRowsPerWarp, int kLoadsPerRow, bool AMAX>
__device__ __forceinline__ void merge_needed_rows(const AcceptParams& p, int b, const int* len_s, RowStat* st,
                                                  int warp, int nw) {
  const int lane = threadIdx.x & 31;
  for (int r0 = warp; r0 < p.NRD; r0 += kRowsPerWarp * nw) {
    float M[kRowsPerWarp], S[kRowsPerWarp], av[kRowsPerWarp];
    int ai[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      M[q] = -INFINITY;
      S[q] = 0.f;
      av[q] = -INFINITY;
      ai[q] = 0x7fffffff;
    }
    for (int c0 = 0; c0 < p.nch; c0 += 32 * kLoadsPerRow) {
      float4 v[kRowsPerWarp][kLoadsPerRow];
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q) {
        const int r = r0 + q * nw;
        const bool need = r < p.NRD && row_needed_s(p, len_s, r);
        const RowStat* src = p.part + (static_cast<int64_t>(b) * p.NRD + (need ? r : 0)) * p.nch;
#pragma unroll
        for (int h = 0; h < kLoadsPerRow; ++h) {
          const int c = c0 + h * 32 + lane;
          v[q][h] = (need && c < p.nch) ? __ldcg(reinterpret_cast<const float4*>(src + c))
                                        : make_float4(-INFINITY, 0.f, -INFINITY, __int_as_float(0x7fffffff));
        }
      }
#pragma unroll
      for (int q = 0; q < kRowsPerWarp; ++q)
#pragma unroll
        for (int h = 0; h < kLoadsPerRow; ++h) {
          stat_merge(M[q], S[q], v[q][h].x, v[q][h].y);
          if (AMAX) amax_merge(av[q], ai[q], v[q][h].z, __float_as_int(v[q][h].w));
        }
    }
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
      const int r = r0 + q * nw;
      const RowStat x = warp_merge_stat<AMAX>(M[q], S[q], av[q], ai[q]);
      if (lane == 0 && r < p.NRD && row_needed_s(p, len_s, r)) st[r] = x;
    }
  }
}

// The weights of the final draw with the row statistics folded in once. p is formed
// exactly as prob_of forms it (2^(v log2 e - m log2 e) * (1/Z)), with the power of two
// 2^20 folded into 1/Z, which scales the rounded product exactly. P = floor(p 2^40) is
// then built in fp32 as hi 2^20 + lo with hi = floor(y), lo = floor((y - hi) 2^20) for
// y = p 2^20: each floor is the low bits of y + 2^23 added with rounding toward zero,
// and every step is exact for 0 <= y < 2^23 (p < 8; a probability is at most 1).
struct DrawRow {
  float c;      // -m log2 e
  float inv20;  // (1/Z rounded to nearest) * 2^20
  int probs;
};
__device__ __forceinline__ DrawRow draw_row(const RowStat& st, int probs) {
  return DrawRow{-st.m * kLog2e, __frcp_rn(st.s) * 1048576.0f, probs};
}
struct Split {
  uint32_t hi, lo;      // P = hi 2^20 + lo
};
__device__ __forceinline__ Split weight_split(float v, const DrawRow& r) {
  float y = r.probs ? v * 1048576.0f : ex2_approx(fmaf(v, kLog2e, r.c)) * r.inv20;
  y = fminf(fmaxf(y, 0.f), 8388607.0f);
  const float t1 = __fadd_rz(y, 8388608.0f);           // 2^23 + floor(y)
  const float f = y + (8388608.0f - t1);               // y - floor(y)
  const float t2 = __fadd_rz(f * 1048576.0f, 8388608.0f);
  return Split{__float_as_uint(t1) - 0x4B000000u, __float_as_uint(t2) - 0x4B000000u};
}
__device__ __forceinline__ long long split64(const Split& w) {
  return (static_cast<long long>(w.hi) << 20) + static_cast<long long>(w.lo);
}
// the weight the draw uses at entry i: P (bonus) or the residual max(0, P - Q), with Q
// one-hot at excl for a copy block or from the draft row for the chain block
__device__ __forceinline__ long long draw_weight(float pv, const DrawRow& pr, bool has_q, float qv,
                                                 const DrawRow& qr, int excl, int ub, int64_t i) {
  const long long P = split64(weight_split(pv, pr));
  if (ub) return P;
  const long long Q = has_q ? split64(weight_split(qv, qr)) : ((i == excl) ? kOneWeight : 0LL);
  return P > Q ? P - Q : 0LL;
}

__device__ __forceinline__ float f4(const float4& v, int e) { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }

// Sums over one lane's run of a chunk (kChunkVec float4 of the target row `a`, and of the draft
// row `q` when HAS_Q): sp = the bonus weights P, sw = the residual max(0, P - Q) with HAS_Q,
// else P. Each weight is formed once. P and Q are kept as (hi, lo) = value hi 2^20 + lo with
// lo < 2^20, so P - Q = (hi_P - hi_Q) 2^20 + (lo_P - lo_Q) with the low difference inside
// (-2^20, 2^20): it is positive exactly when the high difference is, or when that is zero and
// the low one is positive. Sums of kLaneEntries entries fit the 32-bit parts.
template <bool HAS_Q>
__device__ __forceinline__ void lane_weight_sums(const float4 (&a)[kChunkVec], const float4 (&q)[kChunkVec],
                                                 const DrawRow& pr, const DrawRow& qr, long long& sp, long long& sw) {
  uint32_t phi = 0, plo = 0;
  int32_t whi = 0, wlo = 0;
#pragma unroll
  for (int j = 0; j < kChunkVec; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const Split P = weight_split(f4(a[j], e), pr);
      phi += P.hi;
      plo += P.lo;
      if (HAS_Q) {
        const Split Q = weight_split(f4(q[j], e), qr);
        const int32_t dh = static_cast<int32_t>(P.hi) - static_cast<int32_t>(Q.hi);
        const int32_t dl = static_cast<int32_t>(P.lo) - static_cast<int32_t>(Q.lo);
        if (dh > 0 || (dh == 0 && dl > 0)) {
          whi += dh;
          wlo += dl;
        }
      }
    }
  sp = (static_cast<long long>(phi) << 20) + static_cast<long long>(plo);
  sw = HAS_Q ? (static_cast<long long>(whi) << 20) + static_cast<long long>(wlo) : sp;
}

// this lane's entries [lo + lane*kLaneEntries, + kLaneEntries) of a row as kChunkVec float4
// (entry k of the run is component k%4 of v[k/4]); entries past the row end are -inf
__device__ __forceinline__ void load_lane_run(const AcceptParams& p, const void* row, int64_t lo, float4* v) {
  const int lane = threadIdx.x & 31;
  const int64_t l0 = lo + static_cast<int64_t>(lane) * kLaneEntries;
  if (!p.bf16 && l0 + kLaneEntries <= p.V && ((p.V * 4) & 15) == 0 && aligned_dev(row, 16)) {
    const float4* r4 = reinterpret_cast<const float4*>(static_cast<const float*>(row) + l0);
#pragma unroll
    for (int j = 0; j < kChunkVec; ++j) v[j] = __ldg(r4 + j);
  } else if (p.bf16 && l0 + kLaneEntries <= p.V && ((p.V * 2) & 15) == 0 && aligned_dev(row, 16)) {
    const uint4* r2 = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(row) + l0);
#pragma unroll
    for (int j = 0; j < kChunkVec / 2; ++j) {
      const uint4 w = __ldg(r2 + j);
      v[2 * j] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                             __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
      v[2 * j + 1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                                 __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
    }
  } else {
#pragma unroll
    for (int j = 0; j < kChunkVec; ++j) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t i = l0 + j * 4 + e;
        x[e] = i < p.V ? load_val(row, i, p.bf16) : -INFINITY;
      }
      v[j] = make_float4(x[0], x[1], x[2], x[3]);
    }
  }
}

__global__ void __launch_bounds__(kFinThreads, 1)
k_accept_finish_batch(AcceptParams p) {
  __shared__ FinishSmem sm;
  const uint32_t rank = cl_rank();
  const int C = static_cast<int>(gridDim.x);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nslots = p.NB * p.Dmax;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    // this CTA has started this sequence (its peers wait for that before writing to it)
    if (C > 1) asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
    // ---- 1. per token slot: token, block length, uniform and the logits the test needs;
    //         none of it comes from the row pass, so it is loaded before griddepcontrol.wait.
    //         Every CTA of the cluster takes the same decisions from the same data.
    int x_[kSlotsPer], row_[kSlotsPer];
    bool live_[kSlotsPer];
    float lp_[kSlotsPer], lq_[kSlotsPer], u_[kSlotsPer];
#pragma unroll
    for (int k = 0; k < kSlotsPer; ++k) {
      live_[k] = false;
      x_[k] = 0;
      row_[k] = 0;
      lp_[k] = 0.f;
      lq_[k] = 0.f;
      u_[k] = 0.f;
      const int sl = tid + k * kFinThreads;
      if (sl < nslots) {
        const int blk = sl / p.Dmax, d = sl % p.Dmax;
        sm.tok_s[sl] = p.blk_tok[static_cast<int64_t>(b) * nslots + sl];
        const int raw = p.blk_len[b * p.NB + blk];
        const int cap = (blk == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
        const int L = min(max(raw, 0), cap);
        if (d < L) {
          const int x = sm.tok_s[sl];
          if (x < 0 || x >= p.V) {
            if (rank == 0) record_error(p.hdr, SSD_ERR_DEVICE, 100);
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
    for (int k = tid; k < p.NB; k += kFinThreads) {
      const int raw = p.blk_len[b * p.NB + k];
      const int cap = (k == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
      const int L = min(max(raw, 0), cap);
      if (rank == 0 && L != raw) record_error(p.hdr, SSD_ERR_DEVICE, 101);
      sm.len_s[k] = L;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the piece statistics are complete

    // ---- 2. every needed row merged from its pieces (rank 0 keeps the merged rows for the
    //         diagnostic copy of p)
    if (p.sample) merge_needed_rows<4, 2, false>(p, b, sm.len_s, sm.st, warp, kFinWarps);
    else merge_needed_rows<4, 2, true>(p, b, sm.len_s, sm.st, warp, kFinWarps);
    __syncthreads();
    if (rank == 0)
      for (int r = tid; r < p.NRD; r += blockDim.x)
        if (row_needed_s(p, sm.len_s, r)) p.stat[static_cast<int64_t>(b) * p.NRD + r] = sm.st[r];

    // ---- 3. acceptance, leading runs, longest block, stop row (outputs by rank 0)
#pragma unroll
    for (int k = 0; k < kSlotsPer; ++k) {
      const int sl = tid + k * kFinThreads;
      if (sl >= nslots) continue;
      bool ok = false;
      if (live_[k]) {
        const int blk = sl / p.Dmax, d = sl % p.Dmax;
        if (!p.sample) {
          ok = (x_[k] == sm.st[row_[k]].amax_i);
        } else {
          const float px = prob_of(lp_[k], sm.st[row_[k]], p.probs);
          const float qx = (blk == p.chain_blk) ? prob_of(lq_[k], sm.st[p.NR + d], p.probs) : 1.f;
          ok = __dmul_rn(static_cast<double>(u_[k]), static_cast<double>(qx)) < static_cast<double>(px);
        }
      }
      sm.ok_s[sl] = ok ? 1 : 0;
    }
    __syncthreads();
    // leading accepted run of every block: one warp per block, the first rejection by ballot
    for (int k = warp; k < p.NB; k += kFinWarps) {
      const int L = sm.len_s[k];
      int a = L;
      for (int d0 = 0; d0 < L; d0 += 32) {
        const int d = d0 + lane;
        const unsigned rej = __ballot_sync(0xffffffffu, d < L && !sm.ok_s[k * p.Dmax + d]);
        if (rej != 0u) {
          a = d0 + __ffs(rej) - 1;
          break;
        }
      }
      if (lane == 0) {
        sm.acc_s[k] = a;
        if (rank == 0) p.acc_len[b * p.NB + k] = a;
      }
    }
    __syncthreads();
    if (tid == 0) {
      // longest accepted run, lowest block index on ties
      int best = -1, ba = -1;
      for (int k = 0; k < p.NB; ++k) {
        if (sm.len_s[k] > 0 && sm.acc_s[k] > ba) {
          ba = sm.acc_s[k];
          best = k;
        }
      }
      const int a = best >= 0 ? ba : 0;
      const int L = best >= 0 ? sm.len_s[best] : 0;
      const int stop = a == 0 ? 0 : 1 + best * p.Dmax + a - 1;
      sm.sel[0] = best;
      sm.sel[1] = a;
      sm.sel[3] = sm.st[stop].amax_i;
      if (rank == 0) {
        p.best_blk[b] = best;
        p.n_out[b] = a + 1;
      }
      StopInfo si;
      si.row = stop;
      si.ps = sm.st[stop];
      si.a = a;
      si.drf_row = -1;
      si.excl = -1;
      si.bonus = (a >= L) ? 1 : 0;
      si.pad[0] = si.pad[1] = si.pad[2] = 0;
      si.qs = si.ps;
      if (a < L) {
        if (best == p.chain_blk) {
          si.drf_row = a;
          si.qs = sm.st[p.NR + a];
        } else {
          si.excl = sm.tok_s[best * p.Dmax + a];
        }
      }
      sm.si = si;
    }
    __syncthreads();
    if (rank == 0) {
      // emitted tokens (the draw below fills the final one in sample mode)
      const int best = sm.sel[0], a = sm.sel[1];
      for (int i = tid; i <= p.Dmax; i += kFinThreads) {
        int v = -1;
        if (i < a) v = sm.tok_s[best * p.Dmax + i];
        else if (i == a && !p.sample) v = sm.sel[3];
        p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + i] = v;
      }
    }
    if (!p.sample) {
      if (C > 1) asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
      __syncthreads();                    // shared state is reused by the next sequence
      continue;
    }

    // ---- 4. the bonus weights P and residual weights W of every chunk of this CTA's
    //         range [c0, c1): warp w takes chunks c0 + w, c0 + w + 32, ...; lane l sums
    //         entries [16 l, 16 l + 16) of a chunk
    const StopInfo si = sm.si;
    const void* prow = row_ptr(p, b, si.row);
    const bool has_q = si.drf_row >= 0;
    const void* qrow = has_q ? row_ptr(p, b, p.NR + si.drf_row) : prow;
    const DrawRow pr = draw_row(si.ps, p.probs), qr = draw_row(si.qs, p.probs);
    const int nper = (p.nchs + C - 1) / C;
    const int c0 = min(p.nchs, static_cast<int>(rank) * nper), c1 = min(p.nchs, c0 + nper);
    // this lane's weights W (residual or bonus) and P of chunk cc, summed, from its entries
    // a (target row) and q (draft row, when there is one)
    auto lane_load = [&](int cc, float4 (&a)[kChunkVec], float4 (&q)[kChunkVec]) {
      const int64_t lo = static_cast<int64_t>(cc) * kSampleChunk;
      load_lane_run(p, prow, lo, a);
      if (has_q && !si.bonus) load_lane_run(p, qrow, lo, q);
    };
    auto lane_sums = [&](int cc, const float4 (&a)[kChunkVec], const float4 (&q)[kChunkVec], long long& sw,
                         long long& sp) {
      if (has_q && !si.bonus) {
        lane_weight_sums<true>(a, q, pr, qr, sp, sw);
        return;
      }
      lane_weight_sums<false>(a, q, pr, qr, sp, sw);
      if (!si.bonus) {
        // a rejected copy token: W = P everywhere but there, where Q = 2^40
        const int64_t l0 = static_cast<int64_t>(cc) * kSampleChunk + static_cast<int64_t>(lane) * kLaneEntries;
        const int64_t xl = static_cast<int64_t>(si.excl) - l0;
        if (xl >= 0 && xl < kLaneEntries) {
          float pe = 0.f;
#pragma unroll
          for (int j = 0; j < kChunkVec; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (4 * j + e == xl) pe = f4(a[j], e);
          const long long Pe = split64(weight_split(pe, pr));
          sw = sp - Pe + (Pe > kOneWeight ? Pe - kOneWeight : 0LL);
        }
      }
    };
    for (int cc = c0 + warp; cc < c1; cc += kFinWarps) {
      long long sw, sp;
      float4 a[kChunkVec], q[kChunkVec];
      lane_load(cc, a, q);
      lane_sums(cc, a, q, sw, sp);
      sw = warp_sum(sw);
      sp = warp_sum(sp);
      if (lane == 0) {
        sm.csum[cc - c0][0] = sw;
        sm.csum[cc - c0][1] = sp;
      }
    }
    __syncthreads();
    // this CTA's totals go to every rank (after every peer has started this sequence)
    if (C > 1) asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
    if (warp == 0) {
      long long tw = 0, tp = 0;
      for (int i = lane; i < c1 - c0; i += 32) {
        tw += sm.csum[i][0];
        tp += sm.csum[i][1];
      }
      tw = warp_sum(tw);
      tp = warp_sum(tp);
      if (C == 1) {
        if (lane == 0) {
          sm.ctasum[0][0] = tw;
          sm.ctasum[0][1] = tp;
        }
      } else if (lane < C) {
        const uint32_t dst = cl_map(&sm.ctasum[rank][0], static_cast<uint32_t>(lane));
        asm volatile("st.shared::cluster.v2.b64 [%0], {%1, %2};" ::"r"(dst), "l"(tw), "l"(tp) : "memory");
      }
    }
    if (C > 1) cl_sync();
    else __syncthreads();

    // ---- 5. (warp 0) S, the threshold T = floor(U S / 2^24), the CTA and then the chunk
    //         that hold it
    if (warp == 0) {
      const long long cw = lane < C ? sm.ctasum[lane][0] : 0, cp = lane < C ? sm.ctasum[lane][1] : 0;
      long long iw = cw, ip = cp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long yw = __shfl_up_sync(0xffffffffu, iw, o);
        const long long yp = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
          iw += yw;
          ip += yp;
        }
      }
      const long long SW = __shfl_sync(0xffffffffu, iw, 31), SP = __shfl_sync(0xffffffffu, ip, 31);
      const int ub = (si.bonus || SW == 0) ? 1 : 0;
      const unsigned long long S = static_cast<unsigned long long>(ub ? SP : SW);
      const float u = fminf(fmaxf(p.u_fin[b], 0.f), 0.99999994f);               // contract: u in [0, 1)
      const unsigned long long U = static_cast<unsigned long long>(u * 16777216.0f);   // floor(u 2^24), exact
      const long long T = static_cast<long long>((__umul64hi(U, S) << 40) | ((U * S) >> 24));
      const long long mc = ub ? cp : cw, ec = (ub ? ip : iw) - mc;
      const unsigned hitc = __ballot_sync(0xffffffffu, mc > 0 && ec <= T && T < ec + mc);
      int oc = -1;
      long long t2 = 0;
      if (hitc != 0u && static_cast<int>(rank) == __ffs(hitc) - 1) {
        // this CTA: the chunk, lane l scanning local chunks [16 l, 16 l + 16)
        const long long t1 = T - __shfl_sync(0xffffffffu, ec, __ffs(hitc) - 1);
        const int n = c1 - c0;
        constexpr int kPerLane = kMaxSampleChunks / 32;
        long long mine = 0;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
          const int i = lane * kPerLane + k;
          if (i < n) mine += sm.csum[i][ub];
        }
        long long incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const long long ex = incl - mine;
        const unsigned hitl = __ballot_sync(0xffffffffu, mine > 0 && ex <= t1 && t1 < incl);
        if (hitl != 0u && lane == __ffs(hitl) - 1) {
          long long acc = ex;
          for (int k = 0; k < kPerLane; ++k) {
            const int i = lane * kPerLane + k;
            if (i >= n) break;
            const long long w = sm.csum[i][ub];
            if (w > 0 && t1 < acc + w) {
              oc = i;
              t2 = t1 - acc;
              break;
            }
            acc += w;
          }
        }
        const unsigned got = __ballot_sync(0xffffffffu, oc >= 0);
        if (got != 0u) {
          const int src = __ffs(got) - 1;
          oc = __shfl_sync(0xffffffffu, oc, src);
          t2 = __shfl_sync(0xffffffffu, t2, src);
        }
      }
      if (lane == 0) {
        sm.c_star = oc;
        sm.t_rem = t2;
        sm.use_bonus = ub;
      }
    }
    __syncthreads();

    // ---- 6. (warp 0 of the CTA that holds it) the lane by one scan of the chunk's lane
    //         sums, then that lane walks its 16 entries
    if (warp == 0 && sm.c_star >= 0) {
      const int ub = sm.use_bonus;
      const long long Tr = sm.t_rem;
      const int cc = c0 + sm.c_star;
      long long mine;
      {
        long long sw, sp;
        float4 a[kChunkVec], q[kChunkVec];
        lane_load(cc, a, q);
        lane_sums(cc, a, q, sw, sp);
        mine = ub ? sp : sw;
      }
      long long incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const long long ex = incl - mine;
      const unsigned hit = __ballot_sync(0xffffffffu, mine > 0 && ex <= Tr && Tr < incl);
      if (hit != 0u && lane == __ffs(hit) - 1) {
        const int64_t l0 = static_cast<int64_t>(cc) * kSampleChunk + static_cast<int64_t>(lane) * kLaneEntries;
        float4 a[kChunkVec], q[kChunkVec];
        lane_load(cc, a, q);                  // again (cached): fewer live registers across the scan
        // the first entry whose prefix sum exceeds the threshold (unrolled: the entries
        // stay in registers)
        long long acc = ex;
        int k_hit = -1;
#pragma unroll
        for (int k = 0; k < kLaneEntries; ++k) {
          acc += draw_weight(f4(a[k / 4], k % 4), pr, has_q, has_q ? f4(q[k / 4], k % 4) : 0.f, qr, si.excl, ub,
                             l0 + k);
          if (k_hit < 0 && acc > Tr) k_hit = k;
        }
        if (k_hit < 0) k_hit = kLaneEntries - 1;
        p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + si.a] = static_cast<int>(l0 + k_hit);
      }
    }
    __syncthreads();
  }
  // no peer writes to this CTA after the last cluster barrier of its sequences
}

// ------------------------------------------------------------------ finish, one warp per chunk
// k_accept_finish_wide: for batches whose clusters of eight (or sixteen) 1024-thread CTAs
// all fit on the GPU at once (B x 8 <= SMs): the same steps with one warp per 512-entry
// chunk of the stop row, each warp staging its chunk in shared memory for the final walk
// and keeping its lanes' sums there, so that the draw needs no second pass over the row.
constexpr int kWideCTAs = 8;                 // cluster size when the stop row has at most 256 chunks
constexpr int kWideMaxCTAs = 16;             // ... and up to 512 chunks (a non-portable cluster size)
constexpr int kWideThreads = 1024;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideSlotsPer = kMaxSlots / kWideThreads;
constexpr size_t kWideDynSmem = 2ull * kWideWarps * kSampleChunk * sizeof(float);

struct __align__(16) WideSmem {
  RowStat st[kMaxRows];                     // merged rows (rank 0 receives them)
  long long wsum[kWideWarps][2];             // residual and bonus weight sums of this CTA's chunks
  long long lsum[kWideWarps][32][2];         // ... of every lane's entries
  long long ctasum[kWideMaxCTAs][2];         // ... of every rank's chunks
  StopInfo si;                              // the stop row (rank 0 sends it to every rank)
  int tok_s[kMaxSlots];                     // candidate tokens (rank 0)
  int len_s[256];
  int acc_s[256];
  unsigned char ok_s[kMaxSlots];
  long long red_w[kWideWarps], red_p[kWideWarps];
  int sel[4];
  int c_star, use_bonus;
  long long t_rem;
};

__global__ void __launch_bounds__(kWideThreads, 1)
k_accept_finish_wide(AcceptParams p) {
  __shared__ WideSmem sm;
  extern __shared__ float4 wide_chunk[];             // [2][kWideWarps][kSampleChunk] fp32 chunks of p and q
  const uint32_t rank = cl_rank();
  const int C = static_cast<int>(gridDim.x);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nslots = p.NB * p.Dmax;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    // this CTA has started this sequence (its peers wait for that before writing to it)
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
    // ---- 1. per token slot: token, block length, uniform and the logits the test needs;
    //         none of it comes from the row pass, so it is loaded before griddepcontrol.wait.
    //         Every CTA of the cluster takes the same decisions from the same data.
    int x_[kWideSlotsPer], row_[kWideSlotsPer];
    bool live_[kWideSlotsPer];
    float lp_[kWideSlotsPer], lq_[kWideSlotsPer], u_[kWideSlotsPer];
#pragma unroll
    for (int k = 0; k < kWideSlotsPer; ++k) {
      live_[k] = false;
      x_[k] = 0;
      row_[k] = 0;
      lp_[k] = 0.f;
      lq_[k] = 0.f;
      u_[k] = 0.f;
      const int sl = tid + k * kWideThreads;
      if (sl < nslots) {
        const int blk = sl / p.Dmax, d = sl % p.Dmax;
        sm.tok_s[sl] = p.blk_tok[static_cast<int64_t>(b) * nslots + sl];
        const int raw = p.blk_len[b * p.NB + blk];
        const int cap = (blk == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
        const int L = min(max(raw, 0), cap);
        if (d < L) {
          const int x = sm.tok_s[sl];
          if (x < 0 || x >= p.V) {
            if (rank == 0) record_error(p.hdr, SSD_ERR_DEVICE, 100);
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
    for (int k = tid; k < p.NB; k += kWideThreads) {
      const int raw = p.blk_len[b * p.NB + k];
      const int cap = (k == p.chain_blk) ? min(p.Dmax, p.K) : p.Dmax;
      const int L = min(max(raw, 0), cap);
      if (rank == 0 && L != raw) record_error(p.hdr, SSD_ERR_DEVICE, 101);
      sm.len_s[k] = L;
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the piece statistics are complete

    // ---- 2. every needed row merged from its pieces (rank 0 keeps the merged rows for the
    //         diagnostic copy of p)
    if (p.sample) merge_needed_rows<3, 2, false>(p, b, sm.len_s, sm.st, warp, kWideWarps);
    else merge_needed_rows<3, 2, true>(p, b, sm.len_s, sm.st, warp, kWideWarps);
    __syncthreads();
    if (rank == 0)
      for (int r = tid; r < p.NRD; r += blockDim.x)
        if (row_needed_s(p, sm.len_s, r)) p.stat[static_cast<int64_t>(b) * p.NRD + r] = sm.st[r];

    // ---- 3. acceptance, leading runs, longest block, stop row (outputs by rank 0)
#pragma unroll
    for (int k = 0; k < kWideSlotsPer; ++k) {
      const int sl = tid + k * kWideThreads;
      if (sl >= nslots) continue;
      bool ok = false;
      if (live_[k]) {
        const int blk = sl / p.Dmax, d = sl % p.Dmax;
        if (!p.sample) {
          ok = (x_[k] == sm.st[row_[k]].amax_i);
        } else {
          const float px = prob_of(lp_[k], sm.st[row_[k]], p.probs);
          const float qx = (blk == p.chain_blk) ? prob_of(lq_[k], sm.st[p.NR + d], p.probs) : 1.f;
          ok = __dmul_rn(static_cast<double>(u_[k]), static_cast<double>(qx)) < static_cast<double>(px);
        }
      }
      sm.ok_s[sl] = ok ? 1 : 0;
    }
    __syncthreads();
    // leading accepted run of every block: one warp per block, the first rejection by ballot
    for (int k = warp; k < p.NB; k += kWideWarps) {
      const int L = sm.len_s[k];
      int a = L;
      for (int d0 = 0; d0 < L; d0 += 32) {
        const int d = d0 + lane;
        const unsigned rej = __ballot_sync(0xffffffffu, d < L && !sm.ok_s[k * p.Dmax + d]);
        if (rej != 0u) {
          a = d0 + __ffs(rej) - 1;
          break;
        }
      }
      if (lane == 0) {
        sm.acc_s[k] = a;
        if (rank == 0) p.acc_len[b * p.NB + k] = a;
      }
    }
    __syncthreads();
    if (tid == 0) {
      // longest accepted run, lowest block index on ties
      int best = -1, ba = -1;
      for (int k = 0; k < p.NB; ++k) {
        if (sm.len_s[k] > 0 && sm.acc_s[k] > ba) {
          ba = sm.acc_s[k];
          best = k;
        }
      }
      const int a = best >= 0 ? ba : 0;
      const int L = best >= 0 ? sm.len_s[best] : 0;
      const int stop = a == 0 ? 0 : 1 + best * p.Dmax + a - 1;
      sm.sel[0] = best;
      sm.sel[1] = a;
      sm.sel[3] = sm.st[stop].amax_i;
      if (rank == 0) {
        p.best_blk[b] = best;
        p.n_out[b] = a + 1;
      }
      StopInfo si;
      si.row = stop;
      si.ps = sm.st[stop];
      si.a = a;
      si.drf_row = -1;
      si.excl = -1;
      si.bonus = (a >= L) ? 1 : 0;
      si.pad[0] = si.pad[1] = si.pad[2] = 0;
      si.qs = si.ps;
      if (a < L) {
        if (best == p.chain_blk) {
          si.drf_row = a;
          si.qs = sm.st[p.NR + a];
        } else {
          si.excl = sm.tok_s[best * p.Dmax + a];
        }
      }
      sm.si = si;
    }
    __syncthreads();
    if (rank == 0) {
      // emitted tokens (the draw below fills the final one in sample mode)
      const int best = sm.sel[0], a = sm.sel[1];
      for (int i = tid; i <= p.Dmax; i += kWideThreads) {
        int v = -1;
        if (i < a) v = sm.tok_s[best * p.Dmax + i];
        else if (i == a && !p.sample) v = sm.sel[3];
        p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + i] = v;
      }
    }
    if (!p.sample) {
      asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
      continue;
    }

    // ---- 4. warp gw stages chunk gw of the stop row in shared memory (lane l: entries
    //         [16 l, 16 l + 16) of the chunk) and sums the bonus weights P and residual
    //         weights W per lane and per warp; the CTA's totals go to every rank
    const StopInfo si = sm.si;
    const void* prow = row_ptr(p, b, si.row);
    const bool has_q = si.drf_row >= 0;
    const void* qrow = has_q ? row_ptr(p, b, p.NR + si.drf_row) : prow;
    const DrawRow pr = draw_row(si.ps, p.probs), qr = draw_row(si.qs, p.probs);
    const int gw = static_cast<int>(rank) * kWideWarps + warp;
    const int64_t lo = static_cast<int64_t>(gw) * kSampleChunk;
    const int64_t l0 = lo + static_cast<int64_t>(lane) * kLaneEntries;   // this lane's first entry
    float* pf = reinterpret_cast<float*>(wide_chunk + warp * (kSampleChunk / 4)) + lane * kLaneEntries;
    float* qf = reinterpret_cast<float*>(wide_chunk + (kWideWarps + warp) * (kSampleChunk / 4)) + lane * kLaneEntries;
    {
      long long sw = 0, sp = 0;
      if (gw < p.nchs) {
        float4 a[kChunkVec];
        load_lane_run(p, prow, lo, a);
#pragma unroll
        for (int j = 0; j < kChunkVec; ++j) reinterpret_cast<float4*>(pf)[j] = a[j];
        if (has_q && !si.bonus) {
          float4 q[kChunkVec];
          load_lane_run(p, qrow, lo, q);
#pragma unroll
          for (int j = 0; j < kChunkVec; ++j) reinterpret_cast<float4*>(qf)[j] = q[j];
          lane_weight_sums<true>(a, q, pr, qr, sp, sw);
        } else {
          lane_weight_sums<false>(a, a, pr, qr, sp, sw);
        }
        if (!si.bonus && !has_q) {
          // a rejected copy token: W = P everywhere but there, where Q = 2^40
          const int64_t xl = static_cast<int64_t>(si.excl) - l0;
          if (xl >= 0 && xl < kLaneEntries) {
            const long long Pe = split64(weight_split(pf[xl], pr));
            sw = sp - Pe + (Pe > kOneWeight ? Pe - kOneWeight : 0LL);
          }
        }
      }
      sm.lsum[warp][lane][0] = sw;
      sm.lsum[warp][lane][1] = sp;
      sw = warp_sum(sw);
      sp = warp_sum(sp);
      if (lane == 0) {
        sm.wsum[warp][0] = sw;
        sm.wsum[warp][1] = sp;
      }
    }
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");   // every peer has started: its memory may be written
    if (warp == 0) {
      long long tw = sm.wsum[lane][0], tp = sm.wsum[lane][1];
      tw = warp_sum(tw);
      tp = warp_sum(tp);
      if (lane < C) {
        const uint32_t dst = cl_map(&sm.ctasum[rank][0], static_cast<uint32_t>(lane));
        asm volatile("st.shared::cluster.v2.b64 [%0], {%1, %2};" ::"r"(dst), "l"(tw), "l"(tp) : "memory");
      }
    }
    cl_sync();

    // ---- 5. (warp 0) S, the threshold T = floor(U S / 2^24), the CTA and then the warp that hold it
    if (warp == 0) {
      const long long cw = lane < C ? sm.ctasum[lane][0] : 0, cp = lane < C ? sm.ctasum[lane][1] : 0;
      long long iw = cw, ip = cp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long yw = __shfl_up_sync(0xffffffffu, iw, o);
        const long long yp = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) {
          iw += yw;
          ip += yp;
        }
      }
      const long long SW = __shfl_sync(0xffffffffu, iw, 31), SP = __shfl_sync(0xffffffffu, ip, 31);
      const int ub = (si.bonus || SW == 0) ? 1 : 0;
      const unsigned long long S = static_cast<unsigned long long>(ub ? SP : SW);
      const float u = fminf(fmaxf(p.u_fin[b], 0.f), 0.99999994f);               // contract: u in [0, 1)
      const unsigned long long U = static_cast<unsigned long long>(u * 16777216.0f);   // floor(u 2^24), exact
      const long long T = static_cast<long long>((__umul64hi(U, S) << 40) | ((U * S) >> 24));
      const long long mc = ub ? cp : cw, ec = (ub ? ip : iw) - mc;
      const unsigned hitc = __ballot_sync(0xffffffffu, mc > 0 && ec <= T && T < ec + mc);
      int ow = -1;
      long long t2 = 0;
      if (hitc != 0u && static_cast<int>(rank) == __ffs(hitc) - 1) {
        const long long t1 = T - __shfl_sync(0xffffffffu, ec, __ffs(hitc) - 1);
        const long long mw = sm.wsum[lane][ub];
        long long iw2 = mw;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, iw2, o);
          if (lane >= o) iw2 += y;
        }
        const long long ew2 = iw2 - mw;
        const unsigned hitw = __ballot_sync(0xffffffffu, mw > 0 && ew2 <= t1 && t1 < iw2);
        if (hitw != 0u) {
          ow = __ffs(hitw) - 1;
          t2 = t1 - __shfl_sync(0xffffffffu, ew2, ow);
        }
      }
      if (lane == 0) {
        sm.c_star = ow;
        sm.t_rem = t2;
        sm.use_bonus = ub;
      }
    }
    __syncthreads();

    // ---- 6. the warp that holds the threshold: the lane by one scan of its lane sums,
    //         then that lane walks its 16 staged entries
    if (warp == sm.c_star && gw < p.nchs) {
      const int ub = sm.use_bonus;
      const long long Tr = sm.t_rem;
      const long long mine = sm.lsum[warp][lane][ub];
      long long incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const long long ex = incl - mine;
      const unsigned hit = __ballot_sync(0xffffffffu, mine > 0 && ex <= Tr && Tr < incl);
      if (hit != 0u && lane == __ffs(hit) - 1) {
        long long acc = ex;
        int k_hit = kLaneEntries - 1;
        for (int k = 0; k < kLaneEntries; ++k) {
          acc += draw_weight(pf[k], pr, has_q, has_q ? qf[k] : 0.f, qr, si.excl, ub, l0 + k);
          if (acc > Tr) {
            k_hit = k;
            break;
          }
        }
        p.out_tok[static_cast<int64_t>(b) * (p.Dmax + 1) + si.a] = static_cast<int>(l0 + k_hit);
      }
    }
    __syncthreads();
  }
  // no peer writes to this CTA after the last cluster barrier of its sequences
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
  // a stats piece is kPieceElems entries of one row
  L.chunk = kPieceElems;
  L.nch = static_cast<int>((a->V + L.chunk - 1) / L.chunk);
  L.schunk = kSampleChunk;
  L.nchs = static_cast<int>((a->V + kSampleChunk - 1) / kSampleChunk);

  size_t off = sizeof(WsHeader);
  L.part_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * NRD * L.nch * sizeof(RowStat), 256);
  L.stat_off = off;
  off = round_up(off + static_cast<size_t>(a->B) * NRD * sizeof(RowStat), 256);
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
    const long long chunk = kPieceElems;
    if (((a->V + chunk - 1) / chunk) * nrd * a->B >= (1LL << 31) - (1LL << 20)) return SSD_ERR_UNSUPPORTED;
  }
  if (a->chain_blk >= 0 && (a->K < 1 || a->K > a->Dmax)) return SSD_ERR_INVALID;
  if (a->mode == SSD_SAMPLE && (a->V + kSampleChunk - 1) / kSampleChunk > kMaxSampleChunks) return SSD_ERR_UNSUPPORTED;
  if (a->early_rows != 0 && a->early_rows != 1) return SSD_ERR_INVALID;
  if (a->max_ctas < 0) return SSD_ERR_INVALID;
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
  p.early = a->early_rows;
  p.max_ctas = a->max_ctas;
  p.nch = L.nch; p.chunk = L.chunk; p.nchs = L.nchs; p.schunk = L.schunk;
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.part = reinterpret_cast<RowStat*>(base + L.part_off);
  p.stat = reinterpret_cast<RowStat*>(base + L.stat_off);
  return p;
}

// the stats kernel: a grid of as many CTAs as are resident at once, or with max_ctas one
// CTA of 16 warps per SM on at most max_ctas SMs
template <bool BF16, bool AMAX>
static cudaError_t launch_stats(const AcceptParams& p, cudaStream_t s) {
  static std::once_flag once[kMaxDevices];
  static long long cap[kMaxDevices];
  static int sms[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [dev] {
    int n = 152, per = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_vocab_stats<BF16, AMAX, 8>, 256, 0) != cudaSuccess)
      per = 1;
    cap[dev] = static_cast<long long>(n) * (per > 0 ? per : 1);
    sms[dev] = n;
  });
  const long long ntask = static_cast<long long>(p.nch) * p.NRD * p.B;
  // the early mode adds the CTA that only waits (at least one other takes the pieces)
  const int extra = p.early ? 1 : 0;
  if (p.max_ctas > 0) {
    const long long want = (ntask + 15) / 16 + extra;
    long long g = std::min<long long>(want, std::min<long long>(p.max_ctas, sms[dev]));
    if (g < 1 + extra) g = 1 + extra;
    return launch_pdl(k_vocab_stats<BF16, AMAX, 16>, dim3(static_cast<unsigned>(g)), dim3(512), 0, s, p);
  }
  const long long want = (ntask + 7) / 8 + extra;
  long long g = want < cap[dev] ? want : cap[dev];
  if (g < 1 + extra) g = 1 + extra;
  // early mode: clusters of 8 CTAs. A grid launched behind a running kernel
  // (programmatic dependent launch) reaches its SMs about 40 CTAs per microsecond when
  // its CTAs come one by one, in about two thirds of that time as clusters (304 CTAs:
  // 7.6 against 5.9 us), which shortens the Llama-3.1-8B-shaped step; the needed-rows
  // mode of the large batches measured slower as clusters (182 -> 280 us at batch 32)
  const unsigned cl = (p.early && g >= 64) ? 8u : 1u;
  if (cl > 1) g = g / cl * cl;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cl > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_vocab_stats<BF16, AMAX, 8>, p);
}

int accept_launch(const AcceptParams& p, cudaStream_t s) {
  const unsigned by = static_cast<unsigned>(p.B < 65535 ? p.B : 65535);
  cudaError_t e;
  {
    // statistics of every needed row (the argmax only where greedy decisions need it)
    KernelTimer t(SSD_KERNEL_VOCAB_STATS, s);
    const bool amax = !p.sample;
    e = p.bf16 ? (amax ? launch_stats<true, true>(p, s) : launch_stats<true, false>(p, s))
               : (amax ? launch_stats<false, true>(p, s) : launch_stats<false, false>(p, s));
    if (e != cudaSuccess) return SSD_ERR_CUDA;
  }
  {
    // merge, acceptance, choice and final draw. Sample mode with B x 8 <= SMs: a cluster of
    // 8 (16 for stop rows of more than 256 chunks) 1024-thread CTAs per sequence, one warp
    // per chunk (k_accept_finish_wide). Otherwise a cluster of C 512-thread CTAs, C the
    // largest of 4, 2 with the whole batch's clusters resident at once, else 1 (and 1 in
    // greedy mode, which has no draw), warps looping over chunks (k_accept_finish_batch).
    static std::once_flag once[kMaxDevices];
    static int sms[kMaxDevices];
    static cudaError_t attr_err[kMaxDevices];
    const int dev = current_device();
    if (dev < 0) return SSD_ERR_CUDA;
    std::call_once(once[dev], [dev] {
      sms[dev] = 0;
      attr_err[dev] = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (attr_err[dev] == cudaSuccess)
        attr_err[dev] = cudaFuncSetAttribute(k_accept_finish_wide, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kWideDynSmem));
      if (attr_err[dev] == cudaSuccess)
        attr_err[dev] = cudaFuncSetAttribute(k_accept_finish_wide, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (attr_err[dev] != cudaSuccess) return SSD_ERR_CUDA;
    const bool wide = p.sample && 8LL * p.B <= sms[dev];
    unsigned C = 1;
    if (wide) {
      C = p.nchs <= kWideCTAs * kWideWarps ? kWideCTAs : kWideMaxCTAs;
    } else if (p.sample) {
      while (C < 4u && 2LL * C * p.B <= sms[dev]) C *= 2;
    }
    KernelTimer t(SSD_KERNEL_ACCEPT_FINISH, s);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, by, 1);
    cfg.blockDim = dim3(wide ? kWideThreads : kFinThreads);
    cfg.dynamicSmemBytes = wide ? kWideDynSmem : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 2 : 1;
    if (wide) {
      e = cudaLaunchKernelEx(&cfg, k_accept_finish_wide, p);
      if (e != cudaSuccess) return SSD_ERR_CUDA;
    } else {
      e = cudaLaunchKernelEx(&cfg, k_accept_finish_batch, p);
      if (e != cudaSuccess) return SSD_ERR_CUDA;
    }
  }
  int n = 2;
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

static std::mutex g_scratch_mu;
static void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up on the
// first call for that device (the lookup loads the module there if needed).
static int static_scratch(void** out) {
  const int dev = current_device();
  if (dev < 0) return SSD_ERR_CUDA;
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
  // Nothing in the scratch has to start at zero: the row pass writes every partial
  // row statistic and the finish kernel every merged one before either is read. The error header at its start keeps the first device-side error until
  // ssd_read_static_error reads and clears it (the array starts zeroed at load).
  const AcceptParams p = accept_params(a, L, static_cast<char*>(ws));
  return accept_launch(p, static_cast<cudaStream_t>(stream));
}

extern "C" int ssd_read_static_error(void* stream, int32_t* out) {
  if (out == nullptr) return SSD_ERR_INVALID;
  void* ws = nullptr;
  const int rc = static_scratch(&ws);
  if (rc != SSD_OK) return rc;
  // the same read-and-clear as for a caller's workspace: a copy to the host, no allocation
  return ssd_read_device_error(ws, stream, out);
}
