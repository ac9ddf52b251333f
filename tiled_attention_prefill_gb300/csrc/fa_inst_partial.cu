// Kernel instances of the split-KV partial form (both head dimensions).
#include "fa_launch.cuh"

namespace fa {
FA_DECLARE_LAUNCH_PARTIAL(, 64, false, false)
FA_DECLARE_LAUNCH_PARTIAL(, 64, false, true)
FA_DECLARE_LAUNCH_PARTIAL(, 64, true, false)
FA_DECLARE_LAUNCH_PARTIAL(, 64, true, true)
FA_DECLARE_LAUNCH_PARTIAL(, 128, false, false)
FA_DECLARE_LAUNCH_PARTIAL(, 128, false, true)
FA_DECLARE_LAUNCH_PARTIAL(, 128, true, false)
FA_DECLARE_LAUNCH_PARTIAL(, 128, true, true)
}  // namespace fa
