// gather.cu -- entry of the aligned gather: picks the instantiation for the
// matrix's layout and value type and the operands' type (gather_f32_csr.cu,
// gather_f32_vcs.cu, gather_f64_csr.cu, gather_f64_vcs.cu, gather_mix_csr.cu;
// the kernel itself is in gather_impl.cuh).
#include "vs_internal.h"

namespace vs {

vs_status launch_gather_f32_csr(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);
vs_status launch_gather_f32_vcs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);
vs_status launch_gather_f64_csr(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);
vs_status launch_gather_f64_vcs(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);
vs_status launch_gather_mix_csr(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);

vs_status launch_gather(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  if (w <= 0 || m.n_major == 0) return VS_OK;
  if (m.layout == VS_LAYOUT_VCS)
    return X.f64 ? launch_gather_f64_vcs(m, X, Y, w, s) : launch_gather_f32_vcs(m, X, Y, w, s);
  if (m.dtype == VS_F64) return launch_gather_f64_csr(m, X, Y, w, s);
  return X.f64 ? launch_gather_mix_csr(m, X, Y, w, s) : launch_gather_f32_csr(m, X, Y, w, s);
}

}  // namespace vs
