// Launch sequences for D = 256 (every Dv) of the backward with the score extensions (ALiBi
// slopes, soft cap): the EXT variants of the score-forming kernels, in their own translation unit.
#include "fa_launch.cuh"

namespace fab {
RunFn pick_d256_ext(int Dv) { return pick_ext<256>(Dv); }
}  // namespace fab
