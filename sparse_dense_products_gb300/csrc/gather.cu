// gather.cu -- the aligned direction: Y[s, :] = sum over the entries (t, a)
// of major slice s of a * X[t, :].  Covers CSR@B, VCSR@B, B@VCSC and CSC@B'
// (through the transpose identity the caller maps every aligned product onto
// this slice frame).
//
// "Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": one warp per major slice, lanes split between the dense width and
// the slice's nonzeros so narrow widths leave no lanes idle; aligned
// directions accumulate in registers and reduce with shuffles.
// "Regridder", "How it is built": each slice gets a group of g threads, g set
// by the matrix alone (the mean entries per slice rounded down to a power of
// two, capped at a warp), summed in a fixed tree, so a product repeats exactly
// and a column gives the same numbers alone or in a batch.
//
// The summation order of one output element (s, c) is fixed by the matrix:
//   * logical partial k (0 <= k < g) sums, with fused multiply-adds in entry
//     order, the entries n of the slice (or chunk) with (n - start) mod g == k;
//   * the g partials meet in the butterfly p[k] += p[k + h] for
//     h = g/2, g/4, ..., 1;
//   * a slice longer than L entries is cut into chunks of L; chunk results are
//     added in chunk order ((c0 + c1) + c2) + ... by the last chunk to finish.
// Physically a lane holds NP = g / G of the logical partials (G slots per
// slice, Q lanes per slot across the width); in-lane adds then shuffles
// reproduce the same tree for every width, so bits never depend on w.
#include <algorithm>

#include "device_utils.cuh"
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kThreads = 256;

struct GatherArgs {
  const int32_t *ptr;   // [n_major+1]
  const int32_t *idx;   // [nnz]
  const void *vals;     // CSR: [nnz] of T; VCS: [R] float
  const int32_t *vptr;  // VCS: [R+1]
  const void *X;
  int64_t ldx;
  void *Y;
  int64_t ldy;
  int n_major;
  int w;      // columns in this block (<= kMaxBlockWidth)
  int G;      // physical slots per slice (g / NP)
  int S;      // slices per warp in the regular part
  int L;      // chunk length
  int n_chunk_tasks;
  const int4 *tasks;  // {slice, chunk k, long id, first partial}
  void *partials;     // [n_chunks][kMaxBlockWidth] of T
  int *counters;      // [n_long]
};

template <bool VCS>
__device__ __forceinline__ void slice_range(const GatherArgs &a, int s, int &e0, int &e1, int &rlo,
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

// VEC: elements per vector access; Q: lanes per slot; NP: logical partials per
// lane; CI: column vectors per lane; VCS: layout.
template <typename T, int VEC, int Q, int NP, int CI, bool VCS>
__global__ void __launch_bounds__(kThreads) gather_kernel(const GatherArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int G = a.G;
  const int ql = lane & (Q - 1);
  const int slot = (lane / Q) & (G - 1);
  const int sub = lane / (Q * G);

  int slice = -1, n0 = 0, n1 = 0, rlo = 0, rhi = 0, nch = 0;
  const bool chunk = warp < a.n_chunk_tasks;
  int4 task = make_int4(0, 0, 0, 0);
  if (chunk) {
    task = a.tasks[warp];
    int e0, e1;
    slice_range<VCS>(a, task.x, e0, e1, rlo, rhi);
    nch = (e1 - e0 + a.L - 1) / a.L;
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
      if (e1 - e0 <= a.L) {  // longer slices belong to chunk tasks
        slice = (int)s;
        n0 = e0;
        n1 = e1;
      }
    }
  }

  const T *__restrict__ X = static_cast<const T *>(a.X);
  const T *__restrict__ vals = static_cast<const T *>(a.vals);
  const float *__restrict__ rvals = static_cast<const float *>(a.vals);

  T acc[NP][CI][VEC];
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int ci = 0; ci < CI; ++ci)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i][ci][e] = T(0);

  bool colok[CI];
  int col0[CI];
#pragma unroll
  for (int ci = 0; ci < CI; ++ci) {
    col0[ci] = (ci * Q + ql) * VEC;
    colok[ci] = col0[ci] < a.w;
  }

  // VCS: the run holding the lane's current entry
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

  const int step = G * NP;
  for (int base = n0 + slot; base < n1; base += step) {
    int j[NP];
    T av[NP];
    bool ok[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int n = base + i * G;
      ok[i] = n < n1;
      j[i] = ok[i] ? ld_stream(a.idx + n) : 0;
      if (!VCS) av[i] = ok[i] ? ld_stream(vals + n) : T(0);
    }
    if (VCS) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const int n = base + i * G;
        if (ok[i] && n >= rend) {
          do {
            ++r;
            rend = a.vptr[r + 1];
          } while (n >= rend);
          v = (T)rvals[r];
        }
        av[i] = v;
      }
    }
    V x[NP][CI];
#pragma unroll
    for (int i = 0; i < NP; ++i)
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
        if (ok[i] && colok[ci])
          x[i][ci] = ld_gather(reinterpret_cast<const V *>(X + (int64_t)j[i] * a.ldx + col0[ci]));
#pragma unroll
    for (int i = 0; i < NP; ++i)
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
        if (ok[i] && colok[ci]) {
          T xe[VEC];
          Ops::unpack(x[i][ci], xe);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[i][ci][e] = fma(av[i], xe[e], acc[i][ci][e]);
        }
  }

  // fixed tree: in-lane levels (strides h*G), then across slots (strides < G)
#pragma unroll
  for (int h = NP / 2; h >= 1; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i)
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[i][ci][e] = acc[i][ci][e] + acc[i + h][ci][e];
  for (int sft = G >> 1; sft >= 1; sft >>= 1)
#pragma unroll
    for (int ci = 0; ci < CI; ++ci)
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        acc[0][ci][e] = acc[0][ci][e] + __shfl_xor_sync(kFullMask, acc[0][ci][e], sft * Q);

  T *__restrict__ Y = static_cast<T *>(a.Y);
  if (!chunk) {
    if (slice >= 0 && slot == 0) {
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
        if (colok[ci])
          *reinterpret_cast<V *>(Y + (int64_t)slice * a.ldy + col0[ci]) = Ops::pack(acc[0][ci]);
    }
    return;
  }

  // chunk of a long slice: publish the partial, the last chunk to arrive combines
  T *__restrict__ P = static_cast<T *>(a.partials);
  if (slice >= 0 && slot == 0) {
#pragma unroll
    for (int ci = 0; ci < CI; ++ci)
      if (colok[ci])
        *reinterpret_cast<V *>(P + (int64_t)(task.w + task.y) * kMaxBlockWidth + col0[ci]) =
            Ops::pack(acc[0][ci]);
  }
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(a.counters + task.z, 1) == nch - 1;
  last = __shfl_sync(kFullMask, last, 0);
  if (!last) return;
  __threadfence();
  if (sub == 0 && slot == 0) {
#pragma unroll
    for (int ci = 0; ci < CI; ++ci) {
      if (!colok[ci]) continue;
      T sum[VEC];
      for (int k = 0; k < nch; ++k) {
        const V pv = __ldcg(reinterpret_cast<const V *>(P + (int64_t)(task.w + k) * kMaxBlockWidth +
                                                         col0[ci]));
        T pe[VEC];
        Ops::unpack(pv, pe);
#pragma unroll
        for (int e = 0; e < VEC; ++e) sum[e] = k == 0 ? pe[e] : sum[e] + pe[e];
      }
      *reinterpret_cast<V *>(Y + (int64_t)task.x * a.ldy + col0[ci]) = Ops::pack(sum);
    }
  }
  if (lane == 0) a.counters[task.z] = 0;  // re-armed for the next launch
}

// ------------------------------------------------------------------ dispatch

template <typename T, bool VCS>
using KernelPtr = void (*)(const GatherArgs);

template <typename T, int VEC, int Q, int CI, bool VCS>
KernelPtr<T, VCS> pick_np(int np) {
  switch (np) {
    case 1: return gather_kernel<T, VEC, Q, 1, CI, VCS>;
    case 2: if constexpr (Q >= 2) return gather_kernel<T, VEC, Q, 2, CI, VCS>; break;
    case 4: if constexpr (Q >= 4) return gather_kernel<T, VEC, Q, 4, CI, VCS>; break;
    case 8: if constexpr (Q >= 8) return gather_kernel<T, VEC, Q, 8, CI, VCS>; break;
    case 16: if constexpr (Q >= 16) return gather_kernel<T, VEC, Q, 16, CI, VCS>; break;
  }
  return nullptr;
}

template <typename T, int VEC, int CI, bool VCS>
KernelPtr<T, VCS> pick_q(int q, int np) {
  switch (q) {
    case 1: return pick_np<T, VEC, 1, CI, VCS>(np);
    case 2: return pick_np<T, VEC, 2, CI, VCS>(np);
    case 4: return pick_np<T, VEC, 4, CI, VCS>(np);
    case 8: return pick_np<T, VEC, 8, CI, VCS>(np);
    case 16: return pick_np<T, VEC, 16, CI, VCS>(np);
  }
  return nullptr;
}

template <typename T, bool VCS>
KernelPtr<T, VCS> pick_scalar(int ci) {
  switch (ci) {
    case 1: return gather_kernel<T, 1, 1, 1, 1, VCS>;
    case 2: return gather_kernel<T, 1, 1, 1, 2, VCS>;
    case 4: return gather_kernel<T, 1, 1, 1, 4, VCS>;
    case 8: return gather_kernel<T, 1, 1, 1, 8, VCS>;
    case 16: return gather_kernel<T, 1, 1, 1, 16, VCS>;
    case 32: return gather_kernel<T, 1, 1, 1, 32, VCS>;
    case 64: return gather_kernel<T, 1, 1, 1, 64, VCS>;
  }
  return nullptr;
}

inline int pow2ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

template <typename T, bool VCS>
vs_status launch_typed(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  constexpr int VW = 16 / sizeof(T);  // elements per 16-byte vector
  for (int64_t c0 = 0; c0 < w; c0 += kMaxBlockWidth) {
    const int wb = (int)std::min<int64_t>(kMaxBlockWidth, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    const bool vec = wb % VW == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(yp) % 16 == 0 && X.ld % VW == 0 &&
                     Y.ld % VW == 0;
    int Q, NP, CI, G;
    KernelPtr<T, VCS> k = nullptr;
    if (vec) {
      const int ncol = wb / VW;
      Q = std::min(16, pow2ceil(ncol));
      CI = (ncol + Q - 1) / Q;
      G = std::min(m.g, 32 / Q);
      NP = m.g / G;
      if (CI == 1) k = pick_q<T, VW, 1, VCS>(Q, NP);
      else if constexpr (sizeof(T) == 8) k = pick_q<T, VW, 2, VCS>(Q, NP);
    } else {
      Q = 1;
      CI = pow2ceil(wb);
      G = m.g;
      NP = 1;
      k = pick_scalar<T, VCS>(CI);
    }
    if (!k) {
      set_error("no gather kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    GatherArgs a;
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
    a.G = G;
    a.S = 32 / (Q * G);
    a.L = m.L;
    a.n_chunk_tasks = (int)m.n_chunks;
    a.tasks = m.chunk_tasks;
    a.partials = m.partials;
    a.counters = m.counters;
    const int64_t warps = m.n_chunks + (m.n_major + a.S - 1) / a.S;
    const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > 0) {
      k<<<(unsigned)blocks, kThreads, 0, s>>>(a);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

}  // namespace

vs_status launch_gather(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  if (w <= 0 || m.n_major == 0) return VS_OK;
  if (m.layout == VS_LAYOUT_VCS) return launch_typed<float, true>(m, X, Y, w, s);
  if (m.dtype == VS_F64) return launch_typed<double, false>(m, X, Y, w, s);
  return launch_typed<float, false>(m, X, Y, w, s);
}

}  // namespace vs
