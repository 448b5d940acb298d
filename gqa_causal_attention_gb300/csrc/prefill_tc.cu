// Prefill attention on the tcgen05 tensor cores (placeholder until the
// kernel lands: no head dimension is taken yet).
#include "kernels.h"

namespace gqa {

bool prefill_tc_supports(int) { return false; }

cudaError_t launch_prefill_tc(const AttnShape&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gqa
