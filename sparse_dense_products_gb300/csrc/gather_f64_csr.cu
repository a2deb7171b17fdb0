// gather_f64_csr.cu -- instantiates the aligned gather (gather_impl.cuh) for
// double values, CSR layout, double operands, with X read through L1; hands the product to the
// shared-memory-slab instantiation (gather_f64_csr_xs.cu) when X fits it.
#include "gather_impl.cuh"

namespace vs {
vs_status launch_gather_f64_csr_xs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);

vs_status launch_gather_f64_csr(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  if (gather_detail::slab_fits<double, double, false>(m, X, Y, w)) return launch_gather_f64_csr_xs(m, X, Y, w, s);
  return gather_detail::launch_typed<double, double, false, false>(m, X, Y, w, s);
}
}  // namespace vs
