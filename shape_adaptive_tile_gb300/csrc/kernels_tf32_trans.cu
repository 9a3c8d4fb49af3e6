// Kernel variants for tf32 operands: transposed operands.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesTF32Trans[] = {SAT_ENTRIES_TRANS(kDtTF32)};
const int kNumEntriesTF32Trans = sizeof(kEntriesTF32Trans) / sizeof(kEntriesTF32Trans[0]);

}  // namespace sat
