// gather_mix_csr.cu -- instantiates the aligned gather (gather_impl.cuh) for
// float values, CSR layout, double operands and sums, with X read through L1; hands the product to the
// shared-memory-slab instantiation (gather_mix_csr_xs.cu) when X fits it.
#include "gather_impl.cuh"

namespace vs {
vs_status launch_gather_mix_csr_xs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);

vs_status launch_gather_mix_csr(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  if (gather_detail::slab_fits<double, float, false>(m, X, Y, w)) return launch_gather_mix_csr_xs(m, X, Y, w, s);
  return gather_detail::launch_typed<double, float, false, false>(m, X, Y, w, s);
}
}  // namespace vs
