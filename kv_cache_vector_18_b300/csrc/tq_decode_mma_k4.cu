// Tensor-core decode split kernels for mse keys with 4-bit codes (every value
// configuration); the kernel itself is in tq_decode_mma.cuh.
#include "tq_decode_mma.cuh"

namespace tq {
namespace mmadec {
template int launch_for_k<4, false>(const SplitArgs&, dim3, int, bool, bool, cudaStream_t);
}  // namespace mmadec
}  // namespace tq
