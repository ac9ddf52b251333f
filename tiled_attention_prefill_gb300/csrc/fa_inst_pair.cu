// Kernel instances of the paired split-K form (causal launches at D = 64 with one to two
// items per SM).
#include "fa_launch.cuh"

namespace fa {
FA_DECLARE_LAUNCH_PAIR(, 64, false, true)
FA_DECLARE_LAUNCH_PAIR(, 64, true, true)
}  // namespace fa
