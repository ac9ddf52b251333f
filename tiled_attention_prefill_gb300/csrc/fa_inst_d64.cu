// Kernel instances for head dimension 64.
#include "fa_launch.cuh"

namespace fa {
FA_DECLARE_LAUNCH(, 64, false, false)
FA_DECLARE_LAUNCH(, 64, false, true)
FA_DECLARE_LAUNCH(, 64, true, false)
FA_DECLARE_LAUNCH(, 64, true, true)
}  // namespace fa
