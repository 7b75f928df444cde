// Causal MHA/GQA attention backward on sm_103a tensor cores (bf16).
#include "attn_common.cuh"
#include "attn_kernels.h"
#include "attn_ptx.cuh"

namespace attn {

cudaError_t tc05_bwd_launch(const Tc05BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace attn
