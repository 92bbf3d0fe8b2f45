// Kernel instances of the backward epilogues on bfloat16 operands (the BF16
// backend of "Grouped GEMM + dGLU (SM100)": no scale factors, 16/32-bit
// outputs): 1-CTA 128 x 128 and 128 x 256 tiles and 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_bf16_128_bwd(const Launch& L) { return launch_shape_bwd<IC_BF16, 128, CM_SINGLE>(L); }
cudaError_t launch_bf16_256_bwd(const Launch& L) { return launch_shape_bwd<IC_BF16, 256, CM_SINGLE>(L); }
cudaError_t launch_bf16_pair_bwd(const Launch& L) { return launch_shape_bwd<IC_BF16, 256, CM_PAIR>(L); }
}  // namespace bsgg
