// Kernel variants for tf32 operands: plain loads, swapped operands, class views.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesTF32Alt[] = {SAT_ENTRIES_ALT(kDtTF32)};
const int kNumEntriesTF32Alt = sizeof(kEntriesTF32Alt) / sizeof(kEntriesTF32Alt[0]);

}  // namespace sat
