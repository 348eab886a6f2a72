// Placeholder: backward tensor-core path routes to the CUDA-core kernels.
#include "fa_internal.h"
namespace fa {
int launch_bwd_tc(const Problem& p) { return launch_bwd_simt(p) == cudaSuccess ? FA_OK : FA_ERR_CUDA; }
}  // namespace fa
