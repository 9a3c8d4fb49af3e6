// Kernel variants for fp16 operands: transposed operands.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesFP16Trans[] = {SAT_ENTRIES_TRANS(kDtFP16)};
const int kNumEntriesFP16Trans = sizeof(kEntriesFP16Trans) / sizeof(kEntriesFP16Trans[0]);

}  // namespace sat
