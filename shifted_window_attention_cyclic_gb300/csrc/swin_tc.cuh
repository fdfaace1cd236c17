// swin_tc.cuh -- entry points of the tcgen05/TMEM kernels (bf16; head_dim 32
// with windows of up to 128 slots, head_dim 128 with windows of any size).
#pragma once
#include "swin_common.cuh"

namespace swin {

// True when the tensor-core kernels take this problem.
bool tc_supported(const Geo &g, int dtype);
int tc_fwd_ctas_per_sm(const Geo &g);
int tc_bwd_ctas_per_sm(const Geo &g);
int launch_fwd_tc(const FwdArgs &a, void *stream);
int launch_bwd_tc(const BwdArgs &a, void *stream);

// Kernels for head_dim 128 and windows of any size (KV-tiled online softmax).
bool large_supported(const Geo &g, int dtype);
int large_max_bias_rows();
int64_t large_fwd_items(const Geo &g);  // (head, image, window, pair of query tiles)
int launch_fwd_large(const FwdArgs &a, void *stream);
int large_bwd_max_bias_rows();
int launch_bwd_large(const BwdArgs &a, void *stream);

}  // namespace swin
