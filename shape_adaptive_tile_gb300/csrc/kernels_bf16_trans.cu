// Kernel variants for bf16 operands: transposed operands.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesBF16Trans[] = {SAT_ENTRIES_TRANS(kDtBF16)};
const int kNumEntriesBF16Trans = sizeof(kEntriesBF16Trans) / sizeof(kEntriesBF16Trans[0]);

}  // namespace sat
