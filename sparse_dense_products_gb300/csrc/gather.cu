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
  if (m.wide) {
    // each segment gathers its own slices: output rows from its first slice on
    const size_t es = Y.f64 ? 8 : 4;
    for (const Matrix &g : m.segs) {
      DenseView Yg = Y;
      Yg.p = static_cast<char *>(Y.p) + (size_t)g.seg_slice0 * (size_t)Y.ld * es;
      Yg.rows = g.n_major;
      if (Y.scale) Yg.scale = static_cast<const char *>(Y.scale) + (size_t)g.seg_slice0 * es;
      VS_TRY(launch_gather(g, X, Yg, w, s));
    }
    return VS_OK;
  }
  if (m.layout == VS_LAYOUT_VCS)
    return X.f64 ? launch_gather_f64_vcs(m, X, Y, w, s) : launch_gather_f32_vcs(m, X, Y, w, s);
  if (m.dtype == VS_F64) return launch_gather_f64_csr(m, X, Y, w, s);
  return X.f64 ? launch_gather_mix_csr(m, X, Y, w, s) : launch_gather_f32_csr(m, X, Y, w, s);
}

}  // namespace vs
