// Internal interface between the attention host code and its kernels.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

struct AttnParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* k_cand;
  const void* v_cand;
  void* out;
  const int32_t* prefix_len;
  const int32_t* blk_len;
  int B, NB, Dmax, Hq, Hkv;
  int64_t P_max;
  float scale_log2;      // softmax scale times log2(e): scores are kept in log2 units
  int out_f32;           // 1: fp32 output whatever the input type
  int S, chunk;          // KV splits and keys per split
  int chunk0;            // keys of split 0 (tensor-core path: it also takes the own-block tiles)
  const int32_t* block_table;   // tensor-core path: paged cache [B][pages_per_seq], or null
  int pages_per_seq;
  int64_t num_pages;
  int skip_absent;       // tensor-core path: skip tiles without a present token (1: after waiting for the
                         // predecessor; 2: blk_len complete at launch, only the last CTA waits, at its end)
  int all_rows;          // write every slot's row; blk_len is never read
  WsHeader* hdr;
  float* ws_ml;          // [rows][S][2]  running max and sum per split
  float* ws_o;           // [rows][S][dh] un-normalised output per split
};

// merge the splits, add the own-block keys, normalise (ssd_attn.cu)
int attn_combine_launch(const AttnParams& p, int dtype, int dh, cudaStream_t s);

// tcgen05 prefix path (ssd_attn_tc.cu)
bool attn_tc_applies(const ssd_attn_args* a);
size_t attn_tc_workspace_size(const ssd_attn_args* a);
int attn_tc_launch(const ssd_attn_args* a, void* ws, cudaStream_t s);

}  // namespace ssd
