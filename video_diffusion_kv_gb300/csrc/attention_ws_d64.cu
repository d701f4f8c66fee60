// attention_ws_d64.cu -- the head_dim 64 instantiations of the fused
// attention kernel (attention_ws.cuh), compiled apart from the head_dim 128
// ones so that the two build in parallel.
#include "attention_ws.cuh"

namespace qvg {

template qvg_status attn_ws<64, 2>(const AttnWsArgs &, int, cudaStream_t);
template qvg_status attn_ws<64, 4>(const AttnWsArgs &, int, cudaStream_t);

}  // namespace qvg
