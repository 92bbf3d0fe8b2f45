// Kernel instances of the backward epilogues: FP4 inputs with UE8M0 scales (E2M1 data, float8_e8m0fnu scales per 16 or per 32), 256 x 256 tiles on CTA pairs.
#include "bsgg_launch.cuh"

namespace bsgg {
cudaError_t launch_f4e8_pair_bwd(const Launch& L) { return launch_shape_bwd<IC_F4E8, 256, CM_PAIR>(L); }
}  // namespace bsgg
