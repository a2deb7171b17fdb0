// scatter.cu -- the misaligned direction: for every major slice s and entry
// (t, a) of s, Y[t, :] += a * X[s, :].  Covers VCSC@B, B@VCSR, CSC@B and B@CSR.
//
// "Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": the misaligned directions add into the output with atomics, which
// makes them nondeterministic in the last bits.  Two schemes live here:
//
//  * atomic: zero-fill Y, then each warp takes a slice (or a chunk of a long
//    slice), loads X[s, :] once and adds a * X[s, :] into row t with vector
//    reductions (red.global.add.v4.f32).
//
//  * two-phase (deterministic): the slices are cut into C contiguous chunks
//    (balanced by entries, C fixed by the matrix) and Y into tiles of rows
//    that fit in shared memory.  Phase 1: block (tile, chunk) accumulates, in
//    slice order and entry order, the chunk's contributions to its tile in
//    shared memory; each warp owns a band of the tile's rows, so no two
//    threads ever update one element concurrently.  Phase 2 adds the C chunk
//    partials of every element in chunk order.  The order of every element's
//    sum therefore depends on the matrix alone.
#include <algorithm>

#include "device_utils.cuh"
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float fma_t(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_t(double a, double b, double c) { return fma(a, b, c); }

struct ScatterArgs {
  const int32_t *ptr;
  const int32_t *idx;
  const void *vals;
  const int32_t *vptr;
  const void *X;
  int64_t ldx;
  void *Y;
  int64_t ldy;
  int n_major;
  int w;
  int G;  // slots per slice
  int S;  // slices per warp
  int L;
  int n_chunk_tasks;
  const int4 *tasks;
};

template <bool VCS, typename A>
__device__ __forceinline__ void slice_range(const A &a, int s, int &e0, int &e1, int &rlo,
                                            int &rhi) {
  if (VCS) {
    rlo = a.ptr[s];
    rhi = a.ptr[s + 1];
    e0 = a.vptr[rlo];
    e1 = a.vptr[rhi];
  } else {
    rlo = rhi = 0;
    e0 = a.ptr[s];
    e1 = a.ptr[s + 1];
  }
}

// ------------------------------------------------------------------ atomic

template <typename T, int VEC, int Q, int CI, bool VCS>
__global__ void __launch_bounds__(kThreads) scatter_atomic_kernel(const ScatterArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int G = a.G;
  const int ql = lane & (Q - 1);
  const int slot = (lane / Q) & (G - 1);
  const int sub = lane / (Q * G);

  int slice = -1, n0 = 0, n1 = 0, rlo = 0, rhi = 0;
  if (warp < a.n_chunk_tasks) {
    const int4 task = a.tasks[warp];
    int e0, e1;
    slice_range<VCS>(a, task.x, e0, e1, rlo, rhi);
    if (sub == 0) {
      slice = task.x;
      n0 = e0 + task.y * a.L;
      n1 = min(e1, n0 + a.L);
    }
  } else {
    const int64_t s = (warp - a.n_chunk_tasks) * a.S + sub;
    if (s < a.n_major) {
      int e0, e1;
      slice_range<VCS>(a, (int)s, e0, e1, rlo, rhi);
      if (e1 - e0 <= a.L) {
        slice = (int)s;
        n0 = e0;
        n1 = e1;
      }
    }
  }
  if (slice < 0) return;

  const T *__restrict__ X = static_cast<const T *>(a.X);
  T *__restrict__ Y = static_cast<T *>(a.Y);
  const T *__restrict__ vals = static_cast<const T *>(a.vals);
  const float *__restrict__ rvals = static_cast<const float *>(a.vals);
  T x[CI][VEC];
  bool colok[CI];
  int col0[CI];
#pragma unroll
  for (int ci = 0; ci < CI; ++ci) {
    col0[ci] = (ci * Q + ql) * VEC;
    colok[ci] = col0[ci] < a.w;
    if (colok[ci]) Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)slice * a.ldx + col0[ci])), x[ci]);
  }
  int r = 0, rend = 0;
  T v = T(0);
  if (VCS) {
    const int n = n0 + slot;
    if (n < n1) {
      int lo = rlo, hi = rhi - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.vptr[mid] <= n) lo = mid;
        else hi = mid - 1;
      }
      r = lo;
      rend = a.vptr[r + 1];
      v = (T)rvals[r];
    }
  }
#pragma unroll 4
  for (int n = n0 + slot; n < n1; n += G) {
    const int t = ld_stream(a.idx + n);
    T av;
    if (VCS) {
      if (n >= rend) {
        do {
          ++r;
          rend = a.vptr[r + 1];
        } while (n >= rend);
        v = (T)rvals[r];
      }
      av = v;
    } else {
      av = ld_stream(vals + n);
    }
#pragma unroll
    for (int ci = 0; ci < CI; ++ci) {
      if (!colok[ci]) continue;
      T c[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) c[e] = av * x[ci][e];
      red_add(Y + (int64_t)t * a.ldy + col0[ci], c);
    }
  }
}

// ------------------------------------------------------------------ zero fill

template <typename T>
__global__ void zero_fill_kernel(T *__restrict__ Y, int64_t rows, int64_t w, int64_t ld) {
  const int64_t total = rows * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / w, c = i - r * w;
    Y[r * ld + c] = T(0);
  }
}

template <typename T>
__global__ void zero_fill_vec_kernel(float4 *__restrict__ Y, int64_t n16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    Y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ two-phase

struct TwoPhaseArgs {
  const int32_t *ptr;
  const int32_t *idx;
  const void *vals;
  const int32_t *vptr;
  const void *X;
  int64_t ldx;
  void *out;      // Y (C == 1) or the chunk partials
  int64_t ldo;    // row stride of `out`
  int64_t part_stride;  // elements between chunk partials (C > 1)
  const int32_t *bounds;  // [C+1] slice boundaries of the chunks
  int64_t n_t;    // rows of Y
  int tile_rows;  // rows per tile
  int w;
};

// Block (tile blockIdx.x, chunk blockIdx.y).  Shared memory: tile_rows x w of T.
template <typename T, int VEC, int Q, int CI, bool VCS>
__global__ void __launch_bounds__(kThreads) two_phase_kernel(const TwoPhaseArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T *tile = reinterpret_cast<T *>(smem_raw);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int NW = kThreads / 32;
  constexpr int E = 32 / Q;  // entries handled per step
  const int64_t t0 = (int64_t)blockIdx.x * a.tile_rows;
  const int rows = (int)(a.n_t - t0 < a.tile_rows ? a.n_t - t0 : a.tile_rows);
  const int band = (rows + NW - 1) / NW;
  const int my_lo = wid * band, my_hi = min(rows, my_lo + band);  // tile-relative rows
  const int w = a.w;

  for (int i = threadIdx.x; i < rows * w; i += kThreads) tile[i] = T(0);
  __syncthreads();

  const T *__restrict__ X = static_cast<const T *>(a.X);
  const T *__restrict__ vals = static_cast<const T *>(a.vals);
  const float *__restrict__ rvals = static_cast<const float *>(a.vals);
  const int ql = lane & (Q - 1), grp = lane / Q;
  int col0[CI];
  bool colok[CI];
#pragma unroll
  for (int ci = 0; ci < CI; ++ci) {
    col0[ci] = (ci * Q + ql) * VEC;
    colok[ci] = col0[ci] < w;
  }

  const int s_begin = a.bounds[blockIdx.y], s_end = a.bounds[blockIdx.y + 1];
  if (my_lo < my_hi) {
    for (int s = s_begin; s < s_end; ++s) {
      int e0, e1, rlo, rhi;
      slice_range<VCS>(a, s, e0, e1, rlo, rhi);
      if (e0 == e1) continue;
      T x[CI][VEC];
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
        if (colok[ci])
          Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)s * a.ldx + col0[ci])), x[ci]);
      int r = rlo;  // VCS: run of this lane's entry (monotone in n)
      for (int base = e0; base < e1; base += 32) {
        const int n = base + lane;
        int t = -1;
        T av = T(0);
        if (n < e1) {
          const int tt = ld_stream(a.idx + n) - (int)t0;
          if (tt >= my_lo && tt < my_hi) {
            t = tt;
            if (VCS) {
              while (a.vptr[r + 1] <= n) ++r;
              av = (T)rvals[r];
            } else {
              av = ld_stream(vals + n);
            }
          }
        }
        unsigned bits = __ballot_sync(kFullMask, t >= 0);
        while (bits) {
          // the k-th of the next E selected entries goes to lane group k, in entry order
          const int cnt = min(E, __popc(bits));
          int src = 0;
          if (grp < cnt) {
            unsigned b = bits;
            for (int k = 0; k < grp; ++k) b &= b - 1;  // drop the grp lowest set bits
            src = __ffs(b) - 1;
          }
          int tk = __shfl_sync(kFullMask, t, src);
          const T ak = __shfl_sync(kFullMask, av, src);
          if (grp >= cnt) tk = -1;
          // consume the first cnt set bits
          for (int k = 0; k < cnt; ++k) bits &= bits - 1;
          // duplicate rows inside the step are applied in entry order, one round each
          const unsigned peers = __match_any_sync(kFullMask, tk);
          const int rank = __popc(peers & lanemask_lt()) / Q;
          int rounds = tk >= 0 ? rank : 0;
#pragma unroll
          for (int d = 16; d >= 1; d >>= 1) rounds = max(rounds, __shfl_xor_sync(kFullMask, rounds, d));
          for (int rd = 0; rd <= rounds; ++rd) {
            if (tk >= 0 && rank == rd) {
#pragma unroll
              for (int ci = 0; ci < CI; ++ci) {
                if (!colok[ci]) continue;
                V *p = reinterpret_cast<V *>(tile + (int64_t)tk * w + col0[ci]);
                T cur[VEC];
                Ops::unpack(*p, cur);
#pragma unroll
                for (int e = 0; e < VEC; ++e) cur[e] = fma_t(ak, x[ci][e], cur[e]);
                *p = Ops::pack(cur);
              }
            }
            __syncwarp();
          }
        }
      }
    }
  }
  __syncthreads();
  // write the tile (the final Y when C == 1, else this chunk's partial)
  T *__restrict__ out = static_cast<T *>(a.out) + (int64_t)blockIdx.y * a.part_stride;
  for (int i = threadIdx.x; i < rows * w; i += kThreads) {
    const int rr = i / w, c = i - rr * w;
    out[(t0 + rr) * a.ldo + c] = tile[i];
  }
}

// Y[t, c] = sum over chunks k (in order) of P[k][t, c].
template <typename T>
__global__ void combine_kernel(const T *__restrict__ P, int C, int64_t part_stride, int64_t n_t,
                               int w, T *__restrict__ Y, int64_t ldy) {
  const int64_t total = n_t * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / w;
    const int c = (int)(i - t * w);
    T sum = P[i];
    for (int k = 1; k < C; ++k) sum = sum + P[(int64_t)k * part_stride + i];
    Y[t * ldy + c] = sum;
  }
}

inline int pow2ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

template <typename T, bool VCS>
using ScatterPtr = void (*)(const ScatterArgs);
template <typename T, bool VCS>
using TwoPhasePtr = void (*)(const TwoPhaseArgs);

struct Shape {
  bool vec;
  int Q, CI, VEC;
};

template <typename T>
Shape pick_shape(int wb, const void *xp, const void *yp, int64_t ldx, int64_t ldy) {
  constexpr int VW = 16 / sizeof(T);
  Shape sh;
  sh.vec = wb % VW == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(yp) % 16 == 0 && ldx % VW == 0 && ldy % VW == 0;
  if (sh.vec) {
    const int ncol = wb / VW;
    sh.VEC = VW;
    sh.Q = std::min(16, pow2ceil(ncol));
    sh.CI = (ncol + sh.Q - 1) / sh.Q;
  } else {
    sh.VEC = 1;
    sh.Q = std::min(32, pow2ceil(wb));
    sh.CI = (wb + sh.Q - 1) / sh.Q;
  }
  return sh;
}

// Instantiates K<T, VEC, Q, CI, VCS> for the shapes pick_shape can return.
template <typename T, bool VCS, template <typename, int, int, int, bool> class K>
typename K<T, 1, 1, 1, VCS>::Ptr pick_kernel(const Shape &sh) {
  constexpr int VW = 16 / sizeof(T);
  if (sh.vec) {
    if (sh.CI == 1) {
      switch (sh.Q) {
        case 1: return K<T, VW, 1, 1, VCS>::get();
        case 2: return K<T, VW, 2, 1, VCS>::get();
        case 4: return K<T, VW, 4, 1, VCS>::get();
        case 8: return K<T, VW, 8, 1, VCS>::get();
        case 16: return K<T, VW, 16, 1, VCS>::get();
      }
    } else if (sh.CI == 2 && sh.Q == 16) {
      return K<T, VW, 16, 2, VCS>::get();
    }
  } else {
    if (sh.CI == 1) {
      switch (sh.Q) {
        case 1: return K<T, 1, 1, 1, VCS>::get();
        case 2: return K<T, 1, 2, 1, VCS>::get();
        case 4: return K<T, 1, 4, 1, VCS>::get();
        case 8: return K<T, 1, 8, 1, VCS>::get();
        case 16: return K<T, 1, 16, 1, VCS>::get();
        case 32: return K<T, 1, 32, 1, VCS>::get();
      }
    } else if (sh.CI == 2 && sh.Q == 32) {
      return K<T, 1, 32, 2, VCS>::get();
    }
  }
  return nullptr;
}

template <typename T, int VEC, int Q, int CI, bool VCS>
struct AtomicK {
  using Ptr = void (*)(const ScatterArgs);
  static Ptr get() { return scatter_atomic_kernel<T, VEC, Q, CI, VCS>; }
};
template <typename T, int VEC, int Q, int CI, bool VCS>
struct TwoPhaseK {
  using Ptr = void (*)(const TwoPhaseArgs);
  static Ptr get() { return two_phase_kernel<T, VEC, Q, CI, VCS>; }
};

template <typename T, bool VCS>
vs_status atomic_typed(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  for (int64_t c0 = 0; c0 < w; c0 += kMaxBlockWidth) {
    const int wb = (int)std::min<int64_t>(kMaxBlockWidth, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    Shape sh = pick_shape<T>(wb, xp, yp, X.ld, Y.ld);
    auto k = pick_kernel<T, VCS, AtomicK>(sh);
    if (!k) {
      set_error("no scatter kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    ScatterArgs a;
    a.ptr = m.ptr;
    a.idx = m.idx;
    a.vals = m.vals;
    a.vptr = m.vptr;
    a.X = xp;
    a.ldx = X.ld;
    a.Y = yp;
    a.ldy = Y.ld;
    a.n_major = (int)m.n_major;
    a.w = wb;
    a.G = std::max(1, std::min(m.g, 32 / sh.Q));
    a.S = 32 / (sh.Q * a.G);
    a.L = m.L;
    a.n_chunk_tasks = (int)m.n_chunks;
    a.tasks = m.chunk_tasks;
    const int64_t warps = m.n_chunks + (m.n_major + a.S - 1) / a.S;
    const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > 0) {
      k<<<(unsigned)blocks, kThreads, 0, s>>>(a);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

constexpr int kTwoPhaseSmem = 200 * 1024;

template <typename T, bool VCS>
vs_status two_phase_typed(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y, int64_t w,
                          cudaStream_t s) {
  const int C = m.tp_chunks;
  const int64_t n_t = Y.rows;
  for (int64_t c0 = 0; c0 < w; c0 += kMaxBlockWidth) {
    const int wb = (int)std::min<int64_t>(kMaxBlockWidth, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    Shape sh = pick_shape<T>(wb, xp, yp, X.ld, C == 1 ? Y.ld : wb);
    if (C > 1 && sh.vec && wb % (16 / sizeof(T)) != 0) sh.vec = false;
    auto k = pick_kernel<T, VCS, TwoPhaseK>(sh);
    if (!k) {
      set_error("no two-phase kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    const int64_t row_bytes = (int64_t)wb * sizeof(T);
    const int tile_rows = (int)std::max<int64_t>(1, std::min<int64_t>(n_t, kTwoPhaseSmem / row_bytes));
    const int64_t tiles = (n_t + tile_rows - 1) / tile_rows;
    const size_t smem = (size_t)tile_rows * row_bytes;
    VS_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kTwoPhaseSmem));
    TwoPhaseArgs a;
    a.ptr = m.ptr;
    a.idx = m.idx;
    a.vals = m.vals;
    a.vptr = m.vptr;
    a.X = xp;
    a.ldx = X.ld;
    a.bounds = m.tp_bounds;
    a.n_t = n_t;
    a.tile_rows = tile_rows;
    a.w = wb;
    if (C == 1) {
      a.out = yp;
      a.ldo = Y.ld;
      a.part_stride = 0;
    } else {
      const size_t need = (size_t)C * n_t * wb * sizeof(T);
      VS_TRY(h.tp_partials.reserve(need, s));
      a.out = h.tp_partials.p;
      a.ldo = wb;
      a.part_stride = n_t * wb;
    }
    dim3 grid((unsigned)tiles, (unsigned)C);
    k<<<grid, kThreads, smem, s>>>(a);
    VS_LAUNCH_CHECK();
    if (C > 1) {
      const int64_t total = n_t * wb;
      const unsigned blocks = (unsigned)std::min<int64_t>(152 * 8, (total + 255) / 256);
      combine_kernel<T><<<std::max(1u, blocks), 256, 0, s>>>(
          static_cast<const T *>(h.tp_partials.p), C, n_t * wb, n_t, wb, yp, Y.ld);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

}  // namespace

vs_status launch_zero_fill(DenseView Y, int64_t w, size_t dsize, cudaStream_t s) {
  if (w <= 0 || Y.rows <= 0) return VS_OK;
  const int64_t total = Y.rows * w;
  const unsigned blocks = (unsigned)std::min<int64_t>(152 * 8, (total + 255) / 256);
  if (Y.ld == w && reinterpret_cast<uintptr_t>(Y.p) % 16 == 0 && (total * dsize) % 16 == 0) {
    const int64_t n16 = total * (int64_t)dsize / 16;
    zero_fill_vec_kernel<float><<<std::max(1u, std::min<unsigned>(blocks, (unsigned)((n16 + 255) / 256))), 256, 0, s>>>(
        static_cast<float4 *>(Y.p), n16);
  } else if (dsize == 8) {
    zero_fill_kernel<double><<<std::max(1u, blocks), 256, 0, s>>>(static_cast<double *>(Y.p), Y.rows, w, Y.ld);
  } else {
    zero_fill_kernel<float><<<std::max(1u, blocks), 256, 0, s>>>(static_cast<float *>(Y.p), Y.rows, w, Y.ld);
  }
  VS_LAUNCH_CHECK();
  return VS_OK;
}

vs_status launch_scatter_atomic(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                cudaStream_t s) {
  if (w <= 0) return VS_OK;
  VS_TRY(launch_zero_fill(Y, w, m.dsize(), s));
  if (m.n_major == 0 || m.nnz == 0) return VS_OK;
  if (m.layout == VS_LAYOUT_VCS) return atomic_typed<float, true>(m, X, Y, w, s);
  if (m.dtype == VS_F64) return atomic_typed<double, false>(m, X, Y, w, s);
  return atomic_typed<float, false>(m, X, Y, w, s);
}

vs_status launch_scatter_two_phase(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y,
                                   int64_t w, cudaStream_t s) {
  if (w <= 0 || Y.rows == 0) return VS_OK;
  if (m.n_major == 0 || m.nnz == 0) return launch_zero_fill(Y, w, m.dsize(), s);
  if (m.layout == VS_LAYOUT_VCS) return two_phase_typed<float, true>(h, m, X, Y, w, s);
  if (m.dtype == VS_F64) return two_phase_typed<double, false>(h, m, X, Y, w, s);
  return two_phase_typed<float, false>(h, m, X, Y, w, s);
}

}  // namespace vs
