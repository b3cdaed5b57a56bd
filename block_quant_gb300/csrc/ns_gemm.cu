// Muon Newton-Schulz on tcgen05 tensor cores (placeholder until the GEMM lands).
#include <cuda_runtime.h>

#include "bq_internal.h"

namespace bq {

int muon_ns_workspace(int, const bq_mat*, size_t* bytes) {
  if (bytes) *bytes = 0;
  return set_error(BQ_EDEVICE, "bq_muon_ns: not built");
}

int muon_ns(int, const bq_mat*, int, float, float, float, float, void*, size_t, void*) {
  return set_error(BQ_EDEVICE, "bq_muon_ns: not built");
}

}  // namespace bq
