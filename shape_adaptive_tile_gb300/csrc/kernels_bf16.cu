// Kernel variants for bf16 operands: untransposed TMA tiles.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesBF16[] = {SAT_ENTRIES_TMA(kDtBF16)};
const int kNumEntriesBF16 = sizeof(kEntriesBF16) / sizeof(kEntriesBF16[0]);

}  // namespace sat
