// chunked.cu -- chunked (tensor-core) prefill. Not built yet: the entry
// point reports cudaErrorNotSupported.
#include "kernels.h"

namespace gdn {

size_t chunked_workspace_size(int, int, int, int, int, int) { return 256; }

cudaError_t launch_chunked(const ChunkedArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace gdn
