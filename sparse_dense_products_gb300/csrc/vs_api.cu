// vs_api.cu -- the C ABI of libvs: argument checking, handle lifetime and the
// mapping of the six products onto the two kernel families.
//
// Transpose identity: VCSC(A) holds exactly the arrays of VCSR(A^T), and a
// width-contiguous B@A is (A^T B^T) in row-major terms.  So every product is
// one of two kernels in a "slice frame" -- slices are the stored major axis,
// entries carry the minor index t:
//   aligned    (A@B with major = rows, B@A with major = columns):
//              Y[slice] = sum a * X[t]          (gather.cu)
//   misaligned (A@B with major = columns, B@A with major = rows):
//              Y[t]    += a * X[slice]          (scatter.cu)
// ("Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": the same two binary choices as the host kernels.)
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <new>
#include <string>
#include <utility>

#include "vs_internal.h"

namespace vs {

namespace {
thread_local std::string g_last_error;
std::atomic<int64_t> g_launches{0};
}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
int64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

void set_error(const std::string &msg) { g_last_error = msg; }
const char *last_error() { return g_last_error.c_str(); }

vs_status cuda_status(cudaError_t e, const char *what) {
  set_error(std::string(what) + ": " + cudaGetErrorString(e));
  if (e == cudaErrorMemoryAllocation) return VS_ERR_ALLOC;
  return VS_ERR_CUDA;
}

int64_t Matrix::layout_bytes() const {
  const int64_t pb = wide ? 8 : 4;  // bytes per slice pointer
  int64_t b = pb * (n_major + 1) + (int64_t)sizeof(int32_t) * nnz;
  if (layout == VS_LAYOUT_VCS)
    b += (int64_t)sizeof(float) * R + pb * (R + 1);
  else
    b += (int64_t)dsize() * nnz;
  return b;
}

int64_t Matrix::meta_bytes() const {
  if (wide) {  // each segment's own slice pointers and kernel parameters
    int64_t b = 0;
    for (const Matrix &g : segs) {
      b += (int64_t)sizeof(int32_t) * (g.n_major + 1) + g.meta_bytes();
      if (g.layout == VS_LAYOUT_VCS) b += (int64_t)sizeof(int32_t) * (g.R + 1);
    }
    return b;
  }
  int64_t tt = 0;  // the tiled two-phase arrays
  if (tt_rows > 0) {
    tt = (int64_t)(tt_tiles - 1) * (layout == VS_LAYOUT_VCS ? R : n_major) + (3 * tt_groups + 1) +
         (int64_t)tt_tiles * tt_groups * (kTtOwners + 1) + (layout == VS_LAYOUT_VCS ? R : 0);
    tt *= (int64_t)sizeof(int32_t);
  }
  return (int64_t)sizeof(int4) * 3 * n_blocks + (int64_t)sizeof(int4) * n_long + (int64_t)sizeof(int) +
         (int64_t)sizeof(double) * kMaxBlockWidth * n_shares + (int64_t)sizeof(int32_t) * (tp_chunks + 1) +
         tt;
}

namespace {
// The index arrays of a matrix, freed when the last matrix using them goes.
struct IndexArrays {
  std::vector<void *> p;
  ~IndexArrays() {
    for (void *q : p)
      if (q) cudaFree(q);
  }
};

// The index arrays a matrix owns: its own, and for a wide matrix its 64-bit
// pointers and its segments' (whose idx are views, not owned).
void index_arrays_of(const Matrix &m, std::vector<void *> &out) {
  for (void *q : {(void *)m.ptr, (void *)m.vptr, (void *)m.blocks, (void *)m.longs,
                  (void *)m.tp_bounds, (void *)m.ptr64, (void *)m.vptr64, (void *)m.tt_tab,
                  (void *)m.tt_run_slice, (void *)m.tt_group, (void *)m.tt_own})
    out.push_back(q);
  if (!m.borrowed_idx) out.push_back(m.idx);
  for (const Matrix &g : m.segs) index_arrays_of(g, out);
}

// The per-matrix arrays (values, share partials, failure flag), which are
// never shared; a segment's values are a view.
void free_own_arrays(Matrix &m) {
  for (void *p : {m.partials, (void *)m.err})
    if (p) cudaFree(p);
  if (m.vals && !m.borrowed_vals) cudaFree(m.vals);
  for (Matrix &g : m.segs) free_own_arrays(g);
}
}  // namespace

vs_status share_index_arrays(Matrix &m) {
  if (m.index_owner) return VS_OK;
  IndexArrays *ia = new (std::nothrow) IndexArrays();
  if (!ia) {
    set_error("host allocation failed");
    return VS_ERR_ALLOC;
  }
  index_arrays_of(m, ia->p);
  m.index_owner = std::shared_ptr<void>(ia, [](void *q) { delete static_cast<IndexArrays *>(q); });
  return VS_OK;
}

void free_matrix(Matrix &m) {
  if (m.index_owner) {
    m.index_owner.reset();  // the index arrays go with their last user
  } else {
    std::vector<void *> ix;
    index_arrays_of(m, ix);
    for (void *p : ix)
      if (p) cudaFree(p);
  }
  free_own_arrays(m);
  m.ptr = m.idx = m.vptr = m.tp_bounds = nullptr;
  m.vals = m.partials = nullptr;
  m.blocks = nullptr;
  m.longs = nullptr;
  m.err = nullptr;
  m.ptr64 = m.vptr64 = nullptr;
  m.tt_tab = m.tt_run_slice = m.tt_group = m.tt_own = nullptr;
  m.tt_rows = 0;
  m.segs.clear();
}

namespace {
std::atomic<int> g_stall_launches{0};
}  // namespace

bool take_stall() {
  int n = g_stall_launches.load();
  while (n > 0 && !g_stall_launches.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0;
}

vs_status kernel_occupancy(const void *kernel, int threads, int smem, int *per_sm) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void *, int, int>, int> cache;
  static std::set<std::pair<int, const void *>> raised;
  int dev = 0;
  VS_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(dev, kernel, threads, smem);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *per_sm = it->second;
    return VS_OK;
  }
  if (raised.insert({dev, kernel}).second) {
    int optin = 0;
    VS_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    VS_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin));
  }
  int n = 0;
  VS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, (size_t)smem));
  cache.emplace(key, n);
  *per_sm = n;
  return VS_OK;
}

// Group size of a matrix's gathers (and of its segments'): forced (g > 0) or
// the whole matrix's rule (g = 0).
void set_group_size(Matrix &m, int g) {
  m.g = g ? g : group_size_rule(m.nnz, m.n_major);
  for (Matrix &seg : m.segs) seg.g = m.g;
}

vs_status Scratch::reserve(size_t need, cudaStream_t s) {
  if (need <= bytes) return VS_OK;
  if (p) cudaFreeAsync(p, s);
  p = nullptr;
  bytes = 0;
  cudaError_t e = cudaMallocAsync(&p, need, s);
  if (e != cudaSuccess) {
    p = nullptr;
    return cuda_status(e, "cudaMallocAsync (handle scratch)");
  }
  bytes = need;
  return VS_OK;
}

void Scratch::release() {
  if (p) cudaFree(p);
  p = nullptr;
  bytes = 0;
}

}  // namespace vs

using namespace vs;

namespace {

// The failure flags of every matrix a handle's kernels run over: its layout
// and the attached transpose, or their segments when wide.
void failure_flags(const vs_handle_s &h, std::vector<int *> &out) {
  for (const Matrix *m : {&h.A, (const Matrix *)h.T}) {
    if (!m) continue;
    if (m->wide) {
      for (const Matrix &g : m->segs)
        if (g.err) out.push_back(g.err);
    } else if (m->err) {
      out.push_back(m->err);
    }
  }
}

vs_status invalid(const char *msg) {
  set_error(msg);
  return VS_ERR_INVALID;
}

bool valid_handle(vs_handle h) { return h != nullptr; }

vs_status build_common(vs_layout layout, int64_t n_rows, int64_t n_cols, int64_t nnz,
                       const int32_t *d_row, const int32_t *d_col, const void *d_val,
                       vs_dtype dtype, vs_major major, const vs_build_options *opts,
                       cudaStream_t stream, vs_handle *out) {
  if (!out) return invalid("out handle pointer is NULL");
  *out = nullptr;
  if (n_rows < 0 || n_cols < 0 || nnz < 0) return invalid("negative size");
  if (n_rows >= (int64_t(1) << 31) || n_cols >= (int64_t(1) << 31)) {
    set_error("rows and columns must be below 2^31 (int32 indices)");
    return VS_ERR_UNSUPPORTED;
  }
  const int bits = opts ? opts->pointer_bits : 0;
  if (bits != 0 && bits != 32 && bits != 64) return invalid("pointer_bits must be 0, 32 or 64");
  if (opts && opts->segment_entries < 0) return invalid("negative segment_entries");
  if (opts && (opts->two_phase_tile_rows < -1 || opts->two_phase_tile_rows > kTtRows))
    return invalid("two_phase_tile_rows must lie in -1 .. 2048");
  const bool wide = bits == 64 || (bits == 0 && nnz >= (int64_t(1) << 31));
  if (!wide && nnz >= (int64_t(1) << 31)) {
    set_error("2^31 or more entries need 64-bit slice pointers (pointer_bits 64 or 0)");
    return VS_ERR_UNSUPPORTED;
  }
  if (dtype != VS_F32 && dtype != VS_F64) return invalid("unknown dtype");
  if (major != VS_MAJOR_ROW && major != VS_MAJOR_COL) return invalid("unknown major");
  if (nnz > 0 && (!d_row || !d_col || !d_val)) return invalid("NULL COO pointer");
  vs_handle h = new (std::nothrow) vs_handle_s();
  if (!h) {
    set_error("host allocation failed");
    return VS_ERR_ALLOC;
  }
  cudaGetDevice(&h->device);
  h->A.tt_req_rows = opts ? opts->two_phase_tile_rows : 0;
  vs_status st = wide ? build_wide(h->A, layout, major, dtype, n_rows, n_cols, nnz, d_row, d_col,
                                   d_val, opts ? opts->segment_entries : 0, stream)
                      : build_matrix(h->A, layout, major, dtype, n_rows, n_cols, nnz, d_row, d_col,
                                     d_val, stream);
  if (st == VS_OK) st = prepare_matrix(h->A, stream);
  if (st != VS_OK) {
    std::string msg = last_error();
    cudaStreamSynchronize(stream);
    free_matrix(h->A);
    delete h;
    set_error(msg);
    return st;
  }
  *out = h;
  return VS_OK;
}

int64_t extent_bytes(const vs_dense &d) {
  if (d.rows <= 0 || d.cols <= 0) return 0;
  const int64_t es = d.dtype == VS_F64 ? 8 : 4;
  return ((d.rows - 1) * d.row_stride + (d.cols - 1) * d.col_stride + 1) * es;
}

// Maps (A, B, out, dir) onto the slice frame.  Fills X, Y and w.
vs_status frame(const Matrix &m, const vs_dense &B, const vs_dense &out, vs_direction dir,
                DenseView &X, DenseView &Y, int64_t &w, bool &aligned) {
  if (dir != VS_A_B && dir != VS_B_A) return invalid("unknown direction");
  // operands of the matrix dtype, or float64 operands with a float32 (or
  // VCS) matrix: float values, float64 products and sums
  const bool mixed = B.dtype == VS_F64 && m.dtype == VS_F32;
  if (B.dtype != out.dtype || (B.dtype != m.dtype && !mixed)) {
    set_error("B and out must have the matrix dtype, or float64 with a float32/VCS matrix");
    return VS_ERR_INVALID;
  }
  if (B.rows < 0 || B.cols < 0 || out.rows < 0 || out.cols < 0) return invalid("negative shape");
  if (dir == VS_A_B) {
    w = B.cols;
    if (B.rows != m.n_cols || out.rows != m.n_rows || out.cols != w) {
      set_error("A@B needs B: n_cols x w and out: n_rows x w");
      return VS_ERR_SHAPE;
    }
    if (w > 1 && (B.col_stride != 1 || out.col_stride != 1)) {
      set_error("A@B needs column stride 1 for B and out (row-major)");
      return VS_ERR_LAYOUT;
    }
    if ((B.rows > 1 && B.row_stride < w) || (out.rows > 1 && out.row_stride < w)) {
      set_error("row stride smaller than the width");
      return VS_ERR_LAYOUT;
    }
    X = DenseView{B.ptr, B.rows, B.rows > 1 ? B.row_stride : w};
    Y = DenseView{out.ptr, out.rows, out.rows > 1 ? out.row_stride : w};
  } else {
    w = B.rows;
    if (B.cols != m.n_rows || out.cols != m.n_cols || out.rows != w) {
      set_error("B@A needs B: w x n_rows and out: w x n_cols");
      return VS_ERR_SHAPE;
    }
    if (w > 1 && (B.row_stride != 1 || out.row_stride != 1)) {
      set_error("B@A needs row stride 1 for B and out (column-major)");
      return VS_ERR_LAYOUT;
    }
    if ((B.cols > 1 && B.col_stride < w) || (out.cols > 1 && out.col_stride < w)) {
      set_error("column stride smaller than the width");
      return VS_ERR_LAYOUT;
    }
    X = DenseView{B.ptr, B.cols, B.cols > 1 ? B.col_stride : w};
    Y = DenseView{out.ptr, out.cols, out.cols > 1 ? out.col_stride : w};
  }
  if (w > 0 && Y.rows > 0 && !Y.p) return invalid("out pointer is NULL");
  if (w > 0 && X.rows > 0 && !X.p) return invalid("B pointer is NULL");
  // B and out must not overlap
  const int64_t bx = extent_bytes(B), ox = extent_bytes(out);
  if (bx > 0 && ox > 0) {
    const char *b0 = static_cast<const char *>(B.ptr), *o0 = static_cast<const char *>(out.ptr);
    if (b0 < o0 + ox && o0 < b0 + bx) {
      set_error("B and out overlap");
      return VS_ERR_LAYOUT;
    }
  }
  aligned = (dir == VS_A_B) == (m.major == VS_MAJOR_ROW);
  X.f64 = Y.f64 = B.dtype == VS_F64;
  return VS_OK;
}

}  // namespace

namespace vs_derive {
// Copies `rows` rows of `row_bytes` bytes from host memory mapped into the
// device's address space (src, pitch src_ld bytes) to device memory (dst,
// pitch dst_ld bytes), U bytes per load: many SMs' loads in flight over the
// CPU-GPU link.  U divides row_bytes and both pitches; both bases are U-aligned.
template <typename U>
__global__ void copy_rows_kernel(const char *__restrict__ src, int64_t src_ld, char *__restrict__ dst,
                                 int64_t dst_ld, int64_t rows, int64_t row_bytes) {
  const int64_t per_row = row_bytes / (int64_t)sizeof(U);
  const int64_t total = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, c = i - r * per_row;
    *reinterpret_cast<U *>(dst + r * dst_ld + c * (int64_t)sizeof(U)) =
        *reinterpret_cast<const U *>(src + r * src_ld + c * (int64_t)sizeof(U));
  }
}

// values[e] * factors[e], one rounding in T (vs_scale_entries)
template <typename T>
__global__ void scale_values_kernel(const T *__restrict__ v, const T *__restrict__ f, int64_t n,
                                    T *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = v[i] * f[i];
}

// Normalized views: g(v) elementwise, and row scalings of dense operands.
template <typename T>
__device__ __forceinline__ T apply_map(T v, int map) {
  if (map == VS_MAP_LOG1P) return log1p(v);
  if (map == VS_MAP_SQRT) return sqrt(v);
  return v;
}

template <typename T>
__global__ void map_values_kernel(const T *__restrict__ v, int64_t n, int map, T *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = apply_map(v[i], map);
}

// out[r, c] = X[r, c] * s[r] (out row stride w); in == out allowed for the
// post-scaling of a result (ldx then its own stride, out = X)
template <typename T>
__global__ void scale_rows_kernel(const T *X, int64_t rows, int64_t ldx, int64_t w,
                                  const T *__restrict__ s, T *out, int64_t ldo) {
  const int64_t n = rows * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / w, c = i - r * w;
    out[r * ldo + c] = X[r * ldx + c] * s[r];
  }
}

// The gather floor: entries in storage order, Q = w / 4 lanes per entry, each
// loading 16 bytes of the entry's operand row; U entries per lane in flight.
template <int U>
__global__ void __launch_bounds__(256) gather_floor_kernel(const int32_t *__restrict__ idx,
                                                          int64_t nnz, const float4 *__restrict__ X,
                                                          int64_t ldx4, int q, float *sink) {
  const int lane = threadIdx.x & 31;
  const int per = 32 / q;  // entries per warp step
  const int ql = lane % q, slot = lane / q;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (slot < per) {
    const int64_t stride = nwarps * per;
    int64_t n = warp * per + slot;
    for (; n + (U - 1) * stride < nnz; n += U * stride) {
      int j[U];
#pragma unroll
      for (int u = 0; u < U; ++u) j[u] = __ldg(idx + n + u * stride);
      float4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) x[u] = __ldg(X + (size_t)(uint32_t)j[u] * ldx4 + ql);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        acc.x += x[u].x;
        acc.y += x[u].y;
        acc.z += x[u].z;
        acc.w += x[u].w;
      }
    }
    for (; n < nnz; n += stride) {
      const float4 x = __ldg(X + (size_t)(uint32_t)__ldg(idx + n) * ldx4 + ql);
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
  }
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = acc.x + acc.y + acc.z + acc.w;
}
}  // namespace vs_derive

namespace vs {
// The product in the slice frame: the aligned gather, or a misaligned variant.
// Y.scale (an output-row scaling) is fused by the gather; the scatter
// variants apply it with a pass over Y afterwards.
vs_status run_product(vs_handle_s &h, const Matrix &m, const Matrix *t, DenseView X, DenseView Y,
                      int64_t w, bool aligned, vs_variant variant, cudaStream_t stream) {
  if (aligned) return launch_gather(m, X, Y, w, stream);
  if (variant == VS_TRANSPOSED || (variant == VS_DETERMINISTIC && t)) {
    if (!t) return invalid("VS_TRANSPOSED needs vs_attach_transpose first");
    return launch_gather(*t, X, Y, w, stream);
  }
  if (X.f64 && m.dtype == VS_F32) {
    set_error("float64 operands with a float32/VCS matrix: misaligned products need the "
              "transposed route (vs_attach_transpose)");
    return VS_ERR_UNSUPPORTED;
  }
  DenseView Yp = Y;
  Yp.scale = nullptr;
  VS_TRY(variant == VS_ATOMIC ? launch_scatter_atomic(m, X, Yp, w, stream)
                              : launch_scatter_two_phase(h, m, X, Yp, w, stream));
  if (Y.scale && Y.rows > 0) {
    const unsigned grid = (unsigned)std::min<int64_t>(4096, (Y.rows * w + 255) / 256);
    if (Y.f64)
      vs_derive::scale_rows_kernel<double><<<grid, 256, 0, stream>>>(
          static_cast<const double *>(Y.p), Y.rows, Y.ld, w, static_cast<const double *>(Y.scale),
          static_cast<double *>(Y.p), Y.ld);
    else
      vs_derive::scale_rows_kernel<float><<<grid, 256, 0, stream>>>(
          static_cast<const float *>(Y.p), Y.rows, Y.ld, w, static_cast<const float *>(Y.scale),
          static_cast<float *>(Y.p), Y.ld);
    VS_LAUNCH_CHECK();
  }
  return VS_OK;
}
}  // namespace vs

extern "C" {

vs_status vs_build_csr(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                       const int32_t *d_col, const void *d_val, vs_dtype dtype, vs_major major,
                       cudaStream_t stream, vs_handle *out) {
  return build_common(VS_LAYOUT_CSR, n_rows, n_cols, nnz, d_row, d_col, d_val, dtype, major,
                      nullptr, stream, out);
}

vs_status vs_build_vcs(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                       const int32_t *d_col, const float *d_val, vs_major major,
                       cudaStream_t stream, vs_handle *out) {
  return build_common(VS_LAYOUT_VCS, n_rows, n_cols, nnz, d_row, d_col, d_val, VS_F32, major,
                      nullptr, stream, out);
}

vs_status vs_build_csr_opts(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                            const int32_t *d_col, const void *d_val, vs_dtype dtype,
                            vs_major major, const vs_build_options *opts, cudaStream_t stream,
                            vs_handle *out) {
  return build_common(VS_LAYOUT_CSR, n_rows, n_cols, nnz, d_row, d_col, d_val, dtype, major, opts,
                      stream, out);
}

vs_status vs_build_vcs_opts(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                            const int32_t *d_col, const float *d_val, vs_major major,
                            const vs_build_options *opts, cudaStream_t stream, vs_handle *out) {
  return build_common(VS_LAYOUT_VCS, n_rows, n_cols, nnz, d_row, d_col, d_val, VS_F32, major,
                      opts, stream, out);
}

vs_status vs_spmm(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                  vs_variant variant, cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (!B || !out) return invalid("NULL operand descriptor");
  if (variant != VS_DETERMINISTIC && variant != VS_ATOMIC && variant != VS_TRANSPOSED &&
      variant != VS_TWO_PHASE)
    return invalid("unknown variant");
  DenseView X, Y;
  int64_t w = 0;
  bool aligned = false;
  VS_TRY(frame(A->A, *B, *out, dir, X, Y, w, aligned));
  if (w == 0 || Y.rows == 0) return VS_OK;
  return run_product(*A, A->A, A->T, X, Y, w, aligned, variant, stream);
}

vs_status vs_spmm_view(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                       vs_variant variant, const vs_view *view, cudaStream_t stream) {
  if (!view) return vs_spmm(A, B, out, dir, variant, stream);
  if (!valid_handle(A)) return invalid("NULL handle");
  if (!B || !out) return invalid("NULL operand descriptor");
  if (variant != VS_DETERMINISTIC && variant != VS_ATOMIC && variant != VS_TRANSPOSED &&
      variant != VS_TWO_PHASE)
    return invalid("unknown variant");
  if (view->map != VS_MAP_IDENTITY && view->map != VS_MAP_LOG1P && view->map != VS_MAP_SQRT)
    return invalid("unknown value map");
  DenseView X, Y;
  int64_t w = 0;
  bool aligned = false;
  VS_TRY(frame(A->A, *B, *out, dir, X, Y, w, aligned));
  if (w == 0 || Y.rows == 0) return VS_OK;
  if (variant == VS_TRANSPOSED && !A->T) return invalid("VS_TRANSPOSED needs vs_attach_transpose first");
  // views of the stored matrices (nothing here is freed: the arrays stay the handle's)
  Matrix m = A->A, tv;
  const Matrix *t = nullptr;
  if (A->T) {
    tv = *A->T;
    t = &tv;
  }
  if (view->map != VS_MAP_IDENTITY) {
    auto map_into = [&](Matrix &mm, Scratch &dst) -> vs_status {
      const bool vcs = mm.layout == VS_LAYOUT_VCS;
      const int64_t n = vcs ? mm.R : mm.nnz;
      const size_t es = vcs ? sizeof(float) : mm.dsize();
      VS_TRY(dst.reserve(es * (size_t)(n + 16), stream));
      if (n > 0) {
        const unsigned grid = (unsigned)std::min<int64_t>(4096, (n + 255) / 256);
        if (!vcs && mm.dtype == VS_F64)
          vs_derive::map_values_kernel<double><<<grid, 256, 0, stream>>>(
              static_cast<const double *>(mm.vals), n, (int)view->map, static_cast<double *>(dst.p));
        else
          vs_derive::map_values_kernel<float><<<grid, 256, 0, stream>>>(
              static_cast<const float *>(mm.vals), n, (int)view->map, static_cast<float *>(dst.p));
        VS_LAUNCH_CHECK();
      }
      mm.vals = dst.p;
      for (Matrix &g : mm.segs)  // a wide matrix's segments view the mapped values
        g.vals = static_cast<char *>(dst.p) + (size_t)(vcs ? g.seg_run0 : g.seg_entry0) * es;
      return VS_OK;
    };
    VS_TRY(map_into(m, A->view_vals));
    if (t) VS_TRY(map_into(tv, A->view_tvals));
  }
  // the contracted axis scales X (a scaled copy); the output axis scales Y rows
  const void *xs = dir == VS_A_B ? view->col_scale : view->row_scale;
  Y.scale = dir == VS_A_B ? view->row_scale : view->col_scale;
  if (xs && X.rows > 0) {
    const size_t es = X.f64 ? 8 : 4;
    VS_TRY(A->view_X.reserve(es * (size_t)(X.rows * w + 16), stream));
    const unsigned grid = (unsigned)std::min<int64_t>(4096, (X.rows * w + 255) / 256);
    if (X.f64)
      vs_derive::scale_rows_kernel<double><<<grid, 256, 0, stream>>>(
          static_cast<const double *>(X.p), X.rows, X.ld, w, static_cast<const double *>(xs),
          static_cast<double *>(A->view_X.p), w);
    else
      vs_derive::scale_rows_kernel<float><<<grid, 256, 0, stream>>>(
          static_cast<const float *>(X.p), X.rows, X.ld, w, static_cast<const float *>(xs),
          static_cast<float *>(A->view_X.p), w);
    VS_LAUNCH_CHECK();
    const bool f64 = X.f64;
    X = DenseView{A->view_X.p, X.rows, w};
    X.f64 = f64;
  }
  return run_product(*A, m, t, X, Y, w, aligned, variant, stream);
}

vs_status vs_spmm_noalloc(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                          cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (!B || !out) return invalid("NULL operand descriptor");
  DenseView X, Y;
  int64_t w = 0;
  bool aligned = false;
  VS_TRY(frame(A->A, *B, *out, dir, X, Y, w, aligned));
  if (w == 0 || Y.rows == 0) return VS_OK;
  if (aligned) return launch_gather(A->A, X, Y, w, stream);
  if (A->T) return launch_gather(*A->T, X, Y, w, stream);
  if (X.f64 && A->A.dtype == VS_F32) {
    set_error("float64 operands with a float32/VCS matrix: misaligned products need the "
              "transposed route (vs_attach_transpose)");
    return VS_ERR_UNSUPPORTED;
  }
  return launch_scatter_two_phase_static(A->A, X, Y, w, stream);
}

vs_status vs_spmm_host(vs_handle A, const vs_dense *B_host, const vs_dense *out_host,
                       vs_direction dir, vs_variant variant, cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (!B_host || !out_host) return invalid("NULL operand descriptor");
  DenseView X, Y;
  int64_t w = 0;
  bool aligned = false;
  VS_TRY(frame(A->A, *B_host, *out_host, dir, X, Y, w, aligned));
  if (w == 0 || Y.rows == 0) return VS_OK;
  const size_t es = X.f64 ? 8 : 4;
  const int64_t wpad = (w + 3) / 4 * 4;  // keep device rows 16-byte aligned
  // Gather routes store every output element exactly once with plain stores,
  // so a pinned, device-mapped `out` is written in place by the kernel (over
  // the CPU-GPU link, while it computes) instead of staged and copied back.
  const bool gather_route =
      aligned || variant == VS_TRANSPOSED || (variant == VS_DETERMINISTIC && A->T);
  void *out_dev = nullptr;
  if (gather_route) {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, out_host->ptr) == cudaSuccess &&
        pa.type == cudaMemoryTypeHost && pa.devicePointer)
      out_dev = pa.devicePointer;
    else
      cudaGetLastError();  // not mapped: staged below
  }
  VS_TRY(A->stage_B.reserve((size_t)std::max<int64_t>(X.rows, 1) * wpad * es, stream));
  if (!out_dev) VS_TRY(A->stage_out.reserve((size_t)Y.rows * wpad * es, stream));
  // B from mapped (pinned) host memory: a copy kernel, whose loads from every
  // SM keep more of the CPU-GPU link busy than one copy engine does
  void *b_dev = nullptr;
  if (X.rows > 0) {
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, B_host->ptr) == cudaSuccess &&
        pa.type == cudaMemoryTypeHost && pa.devicePointer)
      b_dev = pa.devicePointer;
    else
      cudaGetLastError();  // not mapped: copied by the copy engine below
  }
  if (b_dev) {
    const int64_t rb = w * (int64_t)es, sld = X.ld * (int64_t)es, dld = wpad * (int64_t)es;
    const bool v16 = rb % 16 == 0 && sld % 16 == 0 && reinterpret_cast<uintptr_t>(b_dev) % 16 == 0;
    const int64_t units = X.rows * (rb / (v16 ? 16 : 4));
    const unsigned grid =
        (unsigned)std::max<int64_t>(1, std::min<int64_t>((int64_t)A->A.n_sm * 8, (units + 255) / 256));
    if (v16)
      vs_derive::copy_rows_kernel<uint4><<<grid, 256, 0, stream>>>(
          static_cast<const char *>(b_dev), sld, static_cast<char *>(A->stage_B.p), dld, X.rows, rb);
    else
      vs_derive::copy_rows_kernel<uint32_t><<<grid, 256, 0, stream>>>(
          static_cast<const char *>(b_dev), sld, static_cast<char *>(A->stage_B.p), dld, X.rows, rb);
    VS_LAUNCH_CHECK();
  } else if (X.rows > 0 && X.ld == wpad && w == wpad)
    VS_CUDA(cudaMemcpyAsync(A->stage_B.p, X.p, (size_t)X.rows * wpad * es,
                            cudaMemcpyHostToDevice, stream));
  else if (X.rows > 0)
    VS_CUDA(cudaMemcpy2DAsync(A->stage_B.p, wpad * es, X.p, X.ld * es, w * es, X.rows,
                              cudaMemcpyHostToDevice, stream));
  vs_dense Bd{}, Od{};
  if (dir == VS_A_B) {
    Bd = vs_dense{A->stage_B.p, B_host->rows, B_host->cols, wpad, 1, B_host->dtype};
    Od = vs_dense{A->stage_out.p, out_host->rows, out_host->cols, wpad, 1, out_host->dtype};
  } else {
    Bd = vs_dense{A->stage_B.p, B_host->rows, B_host->cols, 1, wpad, B_host->dtype};
    Od = vs_dense{A->stage_out.p, out_host->rows, out_host->cols, 1, wpad, out_host->dtype};
  }
  if (out_dev) {
    Od = *out_host;
    Od.ptr = out_dev;
  }
  VS_TRY(vs_spmm(A, &Bd, &Od, dir, variant, stream));
  if (out_dev) {
    // written in place
  } else if (Y.ld == wpad && w == wpad)
    VS_CUDA(cudaMemcpyAsync(Y.p, A->stage_out.p, (size_t)Y.rows * wpad * es,
                            cudaMemcpyDeviceToHost, stream));
  else
    VS_CUDA(cudaMemcpy2DAsync(Y.p, Y.ld * es, A->stage_out.p, wpad * es, w * es, Y.rows,
                              cudaMemcpyDeviceToHost, stream));
  // the failure flags come back with the output, so one synchronisation ends the call
  std::vector<int *> flags;
  failure_flags(*A, flags);
  if ((int)flags.size() > A->host_flag_cap) {
    if (A->host_flags) cudaFreeHost(A->host_flags);
    A->host_flags = nullptr;
    A->host_flag_cap = 0;
    void *hf = nullptr;
    VS_CUDA(cudaHostAlloc(&hf, sizeof(int) * flags.size(), cudaHostAllocDefault));
    A->host_flags = static_cast<int *>(hf);
    A->host_flag_cap = (int)flags.size();
  }
  for (size_t k = 0; k < flags.size(); ++k) {
    A->host_flags[k] = 0;
    VS_CUDA(cudaMemcpyAsync(A->host_flags + k, flags[k], sizeof(int), cudaMemcpyDeviceToHost,
                            stream));
  }
  VS_CUDA(cudaStreamSynchronize(stream));
  int any = 0;
  for (size_t k = 0; k < flags.size(); ++k) any |= A->host_flags[k];
  if (any) return vs_device_status(A, stream);  // clears the flags; reports the gave-up wait
  return VS_OK;
}

vs_status vs_attach_transpose(vs_handle A, cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (A->T) return VS_OK;
  Matrix *t = new (std::nothrow) Matrix();
  if (!t) {
    set_error("host allocation failed");
    return VS_ERR_ALLOC;
  }
  t->tt_req_rows = A->A.tt_req_rows;
  vs_status st = build_transpose(A->A, *t, stream);
  if (st == VS_OK) st = prepare_matrix(*t, stream);
  if (st != VS_OK) {
    std::string msg = last_error();
    cudaStreamSynchronize(stream);
    free_matrix(*t);
    delete t;
    set_error(msg);
    return st;
  }
  if (A->forced_g) set_group_size(*t, A->forced_g);
  A->T = t;
  return VS_OK;
}

vs_status vs_force_group_size(vs_handle A, int32_t g) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (g != 0 && g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32)
    return invalid("group size must be 0, 1, 2, 4, 8, 16 or 32");
  A->forced_g = g;
  for (Matrix *m : {&A->A, A->T})
    if (m) set_group_size(*m, g);
  return VS_OK;
}

vs_status vs_transpose(vs_handle A, cudaStream_t stream, vs_handle *out) {
  if (!out) return invalid("out handle pointer is NULL");
  *out = nullptr;
  if (!valid_handle(A)) return invalid("NULL handle");
  vs_handle h = new (std::nothrow) vs_handle_s();
  if (!h) {
    set_error("host allocation failed");
    return VS_ERR_ALLOC;
  }
  h->device = A->device;
  h->A.tt_req_rows = A->A.tt_req_rows;
  vs_status st = build_transpose(A->A, h->A, stream);
  if (st == VS_OK) {
    // build_transpose stores A along its other axis; read as the same major
    // axis, those arrays are the transpose Aᵀ (n_cols x n_rows)
    Matrix &m = h->A;
    std::swap(m.n_rows, m.n_cols);
    m.major = A->A.major;
    st = prepare_matrix(m, stream);
  }
  if (st != VS_OK) {
    std::string msg = last_error();
    cudaStreamSynchronize(stream);
    free_matrix(h->A);
    delete h;
    set_error(msg);
    return st;
  }
  *out = h;
  return VS_OK;
}

vs_status vs_scale_entries(vs_handle A, const void *factors, cudaStream_t stream, vs_handle *out) {
  if (!out) return invalid("out handle pointer is NULL");
  *out = nullptr;
  if (!valid_handle(A)) return invalid("NULL handle");
  const Matrix &a = A->A;
  if (a.layout != VS_LAYOUT_CSR) {
    set_error("vs_scale_entries needs a CSR handle: a per-entry factor would split VCS runs");
    return VS_ERR_LAYOUT;
  }
  if (a.nnz > 0 && !factors) return invalid("NULL factors");
  VS_TRY(share_index_arrays(A->A));
  vs_handle h = new (std::nothrow) vs_handle_s();
  if (!h) {
    set_error("host allocation failed");
    return VS_ERR_ALLOC;
  }
  h->device = A->device;
  Matrix &m = h->A;
  m = a;  // shape, kernel parameters and the shared index arrays
  m.vals = nullptr;
  m.partials = nullptr;
  m.err = nullptr;
  for (Matrix &g : m.segs) {  // a wide matrix's segments get their own values view and scratch
    g.vals = nullptr;
    g.partials = nullptr;
    g.err = nullptr;
  }
  auto fail = [&](vs_status st) {
    std::string msg = last_error();
    cudaStreamSynchronize(stream);
    free_matrix(m);
    delete h;
    set_error(msg);
    return st;
  };
  vs_status st = dev_alloc(&m.vals, m.dsize() * (size_t)(m.nnz + 16));
  if (st != VS_OK) return fail(st);
  auto scratch = [&](Matrix &g) -> vs_status {
    if (g.n_shares > 0)
      VS_TRY(dev_alloc(&g.partials, sizeof(double) * kMaxBlockWidth * (size_t)g.n_shares));
    VS_TRY(dev_alloc((void **)&g.err, sizeof(int)));
    VS_CUDA(cudaMemsetAsync(g.err, 0, sizeof(int), stream));
    return VS_OK;
  };
  if (m.wide) {
    for (Matrix &g : m.segs) {
      g.vals = static_cast<char *>(m.vals) + (size_t)g.seg_entry0 * m.dsize();
      if ((st = scratch(g)) != VS_OK) return fail(st);
    }
  } else if ((st = scratch(m)) != VS_OK) {
    return fail(st);
  }
  if (m.nnz > 0) {
    const unsigned grid = (unsigned)std::min<int64_t>(4096, (m.nnz + 255) / 256);
    if (m.dtype == VS_F64)
      vs_derive::scale_values_kernel<double><<<grid, 256, 0, stream>>>(
          static_cast<const double *>(a.vals), static_cast<const double *>(factors), m.nnz,
          static_cast<double *>(m.vals));
    else
      vs_derive::scale_values_kernel<float><<<grid, 256, 0, stream>>>(
          static_cast<const float *>(a.vals), static_cast<const float *>(factors), m.nnz,
          static_cast<float *>(m.vals));
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(cuda_status(e, "scale_values_kernel"));
  }
  *out = h;
  return VS_OK;
}

vs_status vs_gather_floor(vs_handle A, const vs_dense *B, vs_direction dir, cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (!B) return invalid("NULL operand descriptor");
  if (dir != VS_A_B && dir != VS_B_A) return invalid("unknown direction");
  // B in the slice frame, as vs_spmm would read it (width axis contiguous)
  const bool ab = dir == VS_A_B;
  const int64_t w = ab ? B->cols : B->rows;
  const int64_t rows = ab ? B->rows : B->cols;
  const int64_t ld = ab ? (B->rows > 1 ? B->row_stride : w) : (B->cols > 1 ? B->col_stride : w);
  if (rows != (ab ? A->A.n_cols : A->A.n_rows)) {
    set_error("B does not match the matrix for this direction");
    return VS_ERR_SHAPE;
  }
  if (w > 1 && (ab ? B->col_stride : B->row_stride) != 1) {
    set_error("the width axis of B must have stride 1");
    return VS_ERR_LAYOUT;
  }
  const DenseView X{B->ptr, rows, ld};
  const bool aligned = ab == (A->A.major == VS_MAJOR_ROW);
  if (B->dtype != VS_F32 || w % 4 != 0 || w > 64 || (reinterpret_cast<uintptr_t>(X.p) % 16) ||
      X.ld % 4 != 0) {
    set_error("vs_gather_floor needs float32 16-byte-aligned rows, width a multiple of 4 up to 64");
    return VS_ERR_UNSUPPORTED;
  }
  if (!aligned && !A->T) {  // the misaligned product gathers nothing without the transpose
    set_error("vs_gather_floor of a misaligned direction needs vs_attach_transpose");
    return VS_ERR_UNSUPPORTED;
  }
  const Matrix &m = aligned ? A->A : *A->T;
  if (w == 0 || m.nnz == 0) return VS_OK;
  if (rows > 0 && !X.p) return invalid("B pointer is NULL");
  int n_sm = 0, dev = 0;
  VS_CUDA(cudaGetDevice(&dev));
  VS_CUDA(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev));
  const unsigned grid = (unsigned)(n_sm * 8);
  VS_TRY(A->floor_sink.reserve(sizeof(float) * grid * 256, stream));
  vs_derive::gather_floor_kernel<8><<<grid, 256, 0, stream>>>(
      m.idx, m.nnz, static_cast<const float4 *>(X.p), X.ld / 4, (int)(w / 4),
      static_cast<float *>(A->floor_sink.p));
  VS_LAUNCH_CHECK();
  return VS_OK;
}

vs_status vs_device_status(vs_handle A, cudaStream_t stream) {
  if (!valid_handle(A)) return invalid("NULL handle");
  VS_CUDA(cudaStreamSynchronize(stream));
  int flags = 0;
  std::vector<int *> errs;
  failure_flags(*A, errs);
  for (int *e : errs) {
    int f = 0;
    VS_CUDA(cudaMemcpy(&f, e, sizeof f, cudaMemcpyDeviceToHost));
    if (f) VS_CUDA(cudaMemset(e, 0, sizeof f));
    flags |= f;
  }
  if (flags) {
    set_error((flags & 2) ? "a product kernel met an entry outside its range (inconsistent "
                            "matrix arrays); its output is not valid"
                          : "a product kernel's bounded wait gave up; its output is not valid");
    return VS_ERR_TIMEOUT;
  }
  return VS_OK;
}

void vs_test_stall_producers(int launches) { g_stall_launches.store(launches < 0 ? 0 : launches); }

vs_status vs_info(vs_handle A, vs_info_t *info) {
  if (!valid_handle(A) || !info) return invalid("NULL argument");
  const Matrix &m = A->A;
  std::memset(info, 0, sizeof *info);
  info->layout = m.layout;
  info->major = m.major;
  info->dtype = m.dtype;
  info->group_size = m.g;
  info->n_rows = m.n_rows;
  info->n_cols = m.n_cols;
  info->nnz = m.nnz;
  info->n_runs = m.R;
  info->chunk_len = kBlockEntries;
  info->n_long_slices = m.n_long;
  info->n_chunks = m.n_chunks;
  info->n_blocks = m.n_blocks;
  info->has_transpose = A->T != nullptr;
  info->pointer_bits = m.wide ? 64 : 32;
  info->n_segments = m.wide ? (int32_t)m.segs.size() : 1;
  info->two_phase_tiles = m.tt_rows > 0 ? m.tt_tiles : 0;
  return VS_OK;
}

vs_status vs_export(vs_handle A, vs_arrays *arrays) {
  if (!valid_handle(A) || !arrays) return invalid("NULL argument");
  const Matrix &m = A->A;
  std::memset(arrays, 0, sizeof *arrays);
  arrays->ptr = m.wide ? (const void *)m.ptr64 : (const void *)m.ptr;
  arrays->indices = m.idx;
  arrays->values = m.vals;
  if (m.layout == VS_LAYOUT_VCS)
    arrays->value_ptr = m.wide ? (const void *)m.vptr64 : (const void *)m.vptr;
  arrays->n_major = m.n_major;
  arrays->nnz = m.nnz;
  arrays->n_runs = m.R;
  arrays->pointer_bits = m.wide ? 64 : 32;
  return VS_OK;
}

vs_status vs_handle_bytes(vs_handle A, int64_t *layout_bytes, int64_t *scratch_bytes) {
  if (!valid_handle(A)) return invalid("NULL handle");
  if (layout_bytes) *layout_bytes = A->A.layout_bytes();
  if (scratch_bytes) {
    int64_t s = A->A.meta_bytes() + (int64_t)A->tp_partials.bytes + (int64_t)A->tb_scratch.bytes +
                (int64_t)A->wide_tmp.bytes + (int64_t)A->stage_B.bytes + (int64_t)A->stage_out.bytes;
    if (A->T) s += A->T->layout_bytes() + A->T->meta_bytes();
    *scratch_bytes = s;
  }
  return VS_OK;
}

vs_status vs_destroy(vs_handle A) {
  if (!A) return VS_OK;
  cudaDeviceSynchronize();
  free_matrix(A->A);
  if (A->T) {
    free_matrix(*A->T);
    delete A->T;
  }
  A->tp_partials.release();
  A->tb_scratch.release();
  if (A->host_flags) cudaFreeHost(A->host_flags);
  A->stage_B.release();
  A->stage_out.release();
  A->wide_tmp.release();
  A->view_vals.release();
  A->view_tvals.release();
  A->view_X.release();
  A->floor_sink.release();
  delete A;
  return VS_OK;
}

const char *vs_status_string(vs_status s) {
  switch (s) {
    case VS_OK: return "ok";
    case VS_ERR_INVALID: return "invalid argument";
    case VS_ERR_SHAPE: return "shape mismatch";
    case VS_ERR_LAYOUT: return "unsupported operand layout";
    case VS_ERR_RANGE: return "coordinate out of range";
    case VS_ERR_ALLOC: return "allocation failed";
    case VS_ERR_CUDA: return "CUDA error";
    case VS_ERR_TIMEOUT: return "device wait timed out";
    case VS_ERR_UNSUPPORTED: return "unsupported";
    case VS_ERR_NAN: return "NaN value";
  }
  return "unknown status";
}

const char *vs_last_error(void) { return last_error(); }

int32_t vs_version(void) { return 100; }

int64_t vs_kernel_launches(void) { return launch_count(); }

}  // extern "C"
