// Tensor-core decode split kernels for prod keys with 0-bit codes plus QJL signs (every value
// configuration); the kernel itself is in tq_decode_mma.cuh.
#include "tq_decode_mma.cuh"

namespace tq {
namespace mmadec {
template int launch_for_k<0, true>(const SplitArgs&, dim3, int, bool, bool, cudaStream_t);
}  // namespace mmadec
}  // namespace tq
