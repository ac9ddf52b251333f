// Kernel instances for head dimension 128.
#include "fa_launch.cuh"

namespace fa {
FA_DECLARE_LAUNCH(, 128, false, false)
FA_DECLARE_LAUNCH(, 128, false, true)
FA_DECLARE_LAUNCH(, 128, true, false)
FA_DECLARE_LAUNCH(, 128, true, true)
}  // namespace fa
