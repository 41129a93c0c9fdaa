// Chunk attention on the fifth-generation tensor cores: not built yet; every
// chunk-shaped call runs the fp32 kernel meanwhile.
#include "kvq_internal.h"

namespace kvq {

bool chunk_supported(const kvq_cache &, int, int, int) { return false; }

size_t chunk_workspace_bytes(const kvq_cache &, int, int) { return 0; }

int launch_attend_chunk(const kvq_cache &, const void *, int, int, float, void *, int,
                        const int32_t *, int, float *, void *, const KernelCtl &, cudaStream_t) {
  return 0;
}

}  // namespace kvq
