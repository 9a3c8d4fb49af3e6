// Kernel variants for fp16 operands: untransposed TMA tiles.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesFP16[] = {SAT_ENTRIES_TMA(kDtFP16)};
const int kNumEntriesFP16 = sizeof(kEntriesFP16) / sizeof(kEntriesFP16[0]);

}  // namespace sat
