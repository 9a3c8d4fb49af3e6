// Kernel variants for fp16 operands: plain loads, swapped operands, class views.
#include "launch.cuh"

namespace sat {

const KernelEntry kEntriesFP16Alt[] = {SAT_ENTRIES_ALT(kDtFP16)};
const int kNumEntriesFP16Alt = sizeof(kEntriesFP16Alt) / sizeof(kEntriesFP16Alt[0]);

}  // namespace sat
