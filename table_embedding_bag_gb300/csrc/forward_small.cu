// Small-table forward on the tensor cores (placeholder until the tcgen05
// kernel lands: no problem is eligible yet, so every call takes the generic
// gather-pool path).
#include "common.cuh"
#include "internal.h"

namespace tbe {

bool small_table_eligible(const tbe_desc*, int64_t, bool) { return false; }

cudaError_t launch_forward_small(const Launch&, const void*, const void*, const void*, float*,
                                 int*) {
  return cudaErrorNotSupported;
}

}  // namespace tbe
