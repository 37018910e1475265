// Placeholder until the tcgen05 swap-AB kernel lands.
#include "internal.h"
namespace wqp {
cudaError_t launch_w8a16_gemm_tc(const GemvArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace wqp
