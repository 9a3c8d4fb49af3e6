// Kernel variants for tf32 operands: untransposed TMA tiles.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesTF32[] = {SAT_ENTRIES_TMA(kDtTF32)};
const int kNumEntriesTF32 = sizeof(kEntriesTF32) / sizeof(kEntriesTF32[0]);

}  // namespace sat
