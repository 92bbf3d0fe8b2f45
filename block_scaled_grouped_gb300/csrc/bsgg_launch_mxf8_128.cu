// Kernel instances of the forward epilogues: MXFP8 inputs (E4M3 / E5M2 data, UE8M0 scales per 32), 1-CTA 128 x 128 tiles.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_mxf8_128(const Launch& L) { return launch_shape_fwd<IC_MXF8, 128, CM_SINGLE>(L); }
}  // namespace bsgg
