// Launch sequences for D = 128 (every Dv) of the backward with the score extensions (ALiBi
// slopes, soft cap): the EXT variants of the score-forming kernels, in their own translation unit.
#include "fa_launch.cuh"

namespace fab {
RunFn pick_d128_ext(int Dv) { return pick_ext<128>(Dv); }
}  // namespace fab
