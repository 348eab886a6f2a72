// Placeholder: forward tensor-core path routes to the CUDA-core kernel.
#include "fa_internal.h"
namespace fa {
int launch_fwd_tc(const Problem& p) { return launch_fwd_simt(p) == cudaSuccess ? FA_OK : FA_ERR_CUDA; }
}  // namespace fa
