// Tensor-core tile path (placeholder until the tcgen05 kernel lands).
#include "../../include/fi.h"
#include "prefill_launch.h"

namespace fi {

int launch_prefill(const PrefillArgs&, cudaStream_t) { return FI_ERR_UNSUPPORTED; }

}  // namespace fi
