// Launch sequences for D = 64 (every Dv), forward and plain backward: their own translation
// unit, so that the library's kernel instantiations compile in parallel.
#include "fa_launch.cuh"

namespace fab {
RunFn pick_d64(int Dv, bool forward) { return pick_plain<64>(Dv, forward); }
}  // namespace fab
