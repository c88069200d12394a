// Internal interface between the acceptance host code and its kernels.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// per (row, chunk) and merged per row: running max, sum of exp(l - max),
// argmax value and index (lowest index on ties)
struct RowStat {
  float m;
  float s;
  float amax_v;
  int amax_i;
};

// what the final draw of one sequence needs
struct StopInfo {
  int row;       // target row of the draw
  int a;         // accepted tokens; the drawn token goes to out_tok[a]
  int drf_row;   // draft row whose q enters the residual, or -1
  int excl;      // one-hot q of a rejected copy token, or -1
  int bonus;     // 1: every token was accepted, draw from p
  int pad[3];
  RowStat ps;    // statistics of the target row
  RowStat qs;    // statistics of the draft row (= ps when there is none)
};

struct AcceptParams {
  const void* tgt;
  const void* drf;
  int64_t V;
  const int32_t* blk_tok;
  const int32_t* blk_len;
  int B, NB, Dmax, K, chain_blk, NR, NRD;
  const float* u_acc;
  const float* u_fin;
  int32_t* acc_len;
  int32_t* best_blk;
  int32_t* n_out;
  int32_t* out_tok;
  float* probs_out;
  int sample, bf16, probs;
  int early;          // row pass reads every row without waiting for the retrieval
  int max_ctas;       // row pass on at most this many SMs (0: the whole GPU)
  int nch, nchs;
  int64_t chunk, schunk;
  WsHeader* hdr;
  RowStat* part;      // [B][NRD][nch]
  RowStat* stat;      // [B][NRD] merged rows (read by the diagnostic copy of p)
};

struct AcceptLayout {
  int NR, NRD, nch, nchs;
  int64_t chunk, schunk;
  size_t part_off, stat_off, total;
};

__device__ __forceinline__ bool aligned_dev(const void* p, unsigned a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

AcceptLayout accept_layout(const ssd_accept_args* a);
int accept_validate(const ssd_accept_args* a);
AcceptParams accept_params(const ssd_accept_args* a, const AcceptLayout& L, char* base);
int accept_launch(const AcceptParams& p, cudaStream_t s);

}  // namespace ssd
