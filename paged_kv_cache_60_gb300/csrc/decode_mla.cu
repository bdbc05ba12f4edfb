// Split-KV decode kernel for the 656-byte FP8 MLA token format (placeholder:
// the kernel is added in the next step; until then the host reports the
// format as unsupported).
#include <cuda_runtime.h>

#include "layout.h"

namespace da {

int mla_ctas_per_part() { return 2; }
bool mla_kernel_available() { return false; }

cudaError_t launch_mla(const MlaParams &, cudaStream_t, bool) { return cudaErrorNotSupported; }

}  // namespace da
