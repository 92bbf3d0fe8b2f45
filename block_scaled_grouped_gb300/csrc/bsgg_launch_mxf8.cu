// Kernel instances for MXFP8 inputs (E4M3 / E5M2 data, UE8M0 scales per 32).
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_mxf8(const Launch& L) { return launch_family<false>(L); }
}  // namespace bsgg
