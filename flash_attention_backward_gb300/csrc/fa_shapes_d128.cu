// Launch sequences for D = 128 (every Dv), forward and plain backward: their own translation
// unit, so that the library's kernel instantiations compile in parallel.
#include "fa_launch.cuh"

namespace fab {
RunFn pick_d128(int Dv, bool forward) { return pick_plain<128>(Dv, forward); }
}  // namespace fab
