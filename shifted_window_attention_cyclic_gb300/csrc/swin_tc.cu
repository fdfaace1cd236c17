// swin_tc.cu -- tcgen05/TMEM kernels of SW-MSA (bf16, head_dim 32).
#include <cuda_runtime.h>

#include "swin_tc.cuh"

namespace swin {

bool tc_supported(const Geo &, int) { return false; }
int tc_fwd_ctas_per_sm(const Geo &) { return 1; }
int tc_bwd_ctas_per_sm(const Geo &) { return 1; }
int launch_fwd_tc(const FwdArgs &, void *) { return SWIN_ERR_UNSUPPORTED; }
int launch_bwd_tc(const BwdArgs &, void *) { return SWIN_ERR_UNSUPPORTED; }

}  // namespace swin
