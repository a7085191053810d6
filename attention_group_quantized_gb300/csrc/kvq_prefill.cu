// kvq_prefill.cu -- causal prefill attention over the group-quantised cache.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

kvq_status launch_prefill(const PrefillArgs&, cudaStream_t) { return KVQ_ERR_UNSUPPORTED; }

}  // namespace kvq
