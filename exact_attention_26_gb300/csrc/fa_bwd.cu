// Backward pass of exact attention for sm_103a (kernels follow).
#include "fa_ptx.cuh"

namespace fa {

int launch_bwd(const BwdParams &, cudaStream_t) { return FA_ERR_UNSUPPORTED; }

}  // namespace fa
