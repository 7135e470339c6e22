// Tensor-core (tcgen05) kernels: not built yet.
#include "plx_internal.h"

namespace plx {
bool tc_available() { return false; }
size_t tc_fwd_ws_bytes(int, int, int, int) { return 0; }
size_t tc_bwd_ws_bytes(int, int, int, int) { return 0; }
cudaError_t tc_fwd(const FwdArgs&) { return cudaErrorNotSupported; }
cudaError_t tc_bwd(const BwdArgs&) { return cudaErrorNotSupported; }
}  // namespace plx
