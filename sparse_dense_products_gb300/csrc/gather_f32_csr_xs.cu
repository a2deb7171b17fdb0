// gather_f32_csr_xs.cu -- instantiates the aligned gather (gather_impl.cuh) for
// float values, CSR layout, float operands, with X held in a shared-memory slab.
#include "gather_impl.cuh"

namespace vs {
vs_status launch_gather_f32_csr_xs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  return gather_detail::launch_typed<float, float, false, true>(m, X, Y, w, s);
}
}  // namespace vs
