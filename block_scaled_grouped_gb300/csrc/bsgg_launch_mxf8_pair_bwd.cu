// Kernel instances of the backward epilogues: MXFP8 inputs (E4M3 / E5M2 data, UE8M0 scales per 32), 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_mxf8_pair_bwd(const Launch& L) { return launch_shape_bwd<IC_MXF8, 256, CM_PAIR>(L); }
}  // namespace bsgg
