// fused.cu -- placeholder until the persistent tcgen05 kernel lands.
#include "internal.h"

namespace ssd {

bool fused_supported(const Problem&) { return false; }
size_t fused_workspace_bytes(const Problem&) { return 0; }
cudaError_t launch_fused(const Problem&, void*, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
