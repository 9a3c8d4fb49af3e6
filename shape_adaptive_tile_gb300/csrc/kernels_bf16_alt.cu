// Kernel variants for bf16 operands: plain loads, swapped operands, class views.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesBF16Alt[] = {SAT_ENTRIES_ALT(kDtBF16)};
const int kNumEntriesBF16Alt = sizeof(kEntriesBF16Alt) / sizeof(kEntriesBF16Alt[0]);

}  // namespace sat
