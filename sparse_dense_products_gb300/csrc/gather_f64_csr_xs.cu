// gather_f64_csr_xs.cu -- instantiates the aligned gather (gather_impl.cuh) for
// double values, CSR layout, double operands, with X held in a shared-memory slab.
#include "gather_impl.cuh"

namespace vs {
vs_status launch_gather_f64_csr_xs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  return gather_detail::launch_typed<double, double, false, true>(m, X, Y, w, s);
}
}  // namespace vs
