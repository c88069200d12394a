// tcgen05 prefix kernel for bf16 verification attention (not enabled yet).
#include "ssd_attn.cuh"

namespace ssd {

bool attn_tc_applies(const ssd_attn_args*) { return false; }
size_t attn_tc_workspace_size(const ssd_attn_args*) { return 0; }
int attn_tc_launch(const ssd_attn_args*, void*, cudaStream_t) { return SSD_ERR_UNSUPPORTED; }

}  // namespace ssd
