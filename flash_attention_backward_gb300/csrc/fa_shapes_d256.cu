// Launch sequences for D = 256 (every Dv), forward and plain backward: their own translation
// unit, so that the library's kernel instantiations compile in parallel.
#include "fa_launch.cuh"

namespace fab {
RunFn pick_d256(int Dv, bool forward) { return pick_plain<256>(Dv, forward); }
}  // namespace fab
