// gather.cu -- the aligned direction: Y[s, :] = sum over the entries (t, a)
// of major slice s of a * X[t, :].  Covers CSR@B, VCSR@B, B@VCSC and B@CSC
// (every aligned product maps onto this slice frame, see vs_api.cu), and the
// misaligned products run over an attached exact transpose.
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
// Summation order of one output element (s, c), fixed by the matrix alone:
//   * a run of entries (a whole short slice, or one warp's share of a chunk
//     of a long slice) is summed as g logical partials -- partial k takes the
//     entries n with (n - start) mod g == k, with fused multiply-adds in entry
//     order -- which meet in the butterfly p[k] += p[k + h], h = g/2, ..., 1;
//   * a long slice is cut into chunks (at most kBlockEntries entries and
//     kBlockRuns runs, cut points fixed by the matrix) and every chunk into
//     shares of kShareEntries entries; each share is one such run, and the
//     share results are added in share order ((p0 + p1) + p2) + ... by the
//     last share of the slice to finish.
// Physically a lane holds NP = g / G of the logical partials (G slots per
// slice, Q lanes per slot across the width); in-lane adds then shuffles
// reproduce the same tree for every width, so bits never depend on w.
//
// Data movement: entries, values, slice pointers and runs arrive in shared
// memory by bulk copies through a 4-deep ring fed by a producer warp
// (stage.cuh); the dense rows X[t, :] are gathered through L1 with 16-byte
// vector loads.
#include <algorithm>

#include "stage.cuh"

namespace vs {
namespace {

struct GatherArgs {
  StageArrays st;
  const void *X;
  int64_t ldx;
  void *Y;
  int64_t ldy;
  int w;          // columns in this block (<= kMaxBlockWidth)
  int G;          // physical slots per slice (g / NP)
  int S;          // slices per warp task
  void *partials; // [n_shares][kMaxBlockWidth] of T
  int *counters;  // [n_long]
};

// Sums entries [n0, n1) of one slice into acc (logical partial (n - n0) mod g
// lives in lane slot (n - n0) mod G, register (n - n0) / G mod NP), then runs
// the fixed tree.  (VCS entries carry their run's value, expanded on chip.)
template <typename T, int VEC, int Q, int NP, int CI, bool VCS>
__device__ __forceinline__ void gather_range(const Staged<T, VCS> &sv, const T *__restrict__ X,
                                             int64_t ldx, int n0, int n1, int G,
                                             int slot, const int (&col0)[CI],
                                             const bool (&colok)[CI], T (&acc)[NP][CI][VEC]) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int ci = 0; ci < CI; ++ci)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i][ci][e] = T(0);

  const int step = G * NP;
  for (int base = n0 + slot; base < n1; base += step) {
    int j[NP];
    T av[NP];
    bool ok[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int n = base + i * G;
      ok[i] = n < n1;
      j[i] = ok[i] ? sv.idx[n] : 0;
      av[i] = ok[i] ? sv.vals[n] : T(0);
    }
    V x[NP][CI];
#pragma unroll
    for (int i = 0; i < NP; ++i)
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
        if (ok[i] && colok[ci])
          x[i][ci] = ld_gather(reinterpret_cast<const V *>(X + (int64_t)j[i] * ldx + col0[ci]));
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
  // the fixed tree: in-lane levels (strides h*G), then across slots (strides < G)
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
}

template <typename T, int VEC, int Q, int NP, int CI, bool VCS>
__global__ void __launch_bounds__(kPipeThreads, 2) gather_kernel(const GatherArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  extern __shared__ __align__(128) unsigned char smem[];
  const Pipe<T, VCS> pipe{smem};
  pipe.init();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (wid == kWarpsPerCta) {  // the producer warp
    pipe.produce(a.st, blockIdx.x, a.st.n_blocks, gridDim.x);
    return;
  }
  const int G = a.G;
  const int ql = lane & (Q - 1);
  const int slot = (lane / Q) & (G - 1);
  const int sub = lane / (Q * G);
  const T *__restrict__ X = static_cast<const T *>(a.X);
  T *__restrict__ Y = static_cast<T *>(a.Y);
  int col0[CI];
  bool colok[CI];
#pragma unroll
  for (int ci = 0; ci < CI; ++ci) {
    col0[ci] = (ci * Q + ql) * VEC;
    colok[ci] = col0[ci] < a.w;
  }

  int i = 0;
  for (int b = blockIdx.x; b < a.st.n_blocks; b += gridDim.x, ++i) {
    if (!pipe.acquire(i, a.st)) return;
    const Block k = load_block(a.st.blocks, b);
    const Staged<T, VCS> sv = stage_views<T, VCS>(k, pipe.buf(i % kStages));
    const int units = block_units(k, a.S);
    T acc[NP][CI][VEC];
    for (int u = pipe.grab(i); u < units; u = pipe.grab(i)) {
      if (k.type == 0) {
        // ---- S consecutive slices, one per sub-group
        if (VCS) {
          const int sa = k.s0 + u * a.S, sb = min(k.s1, sa + a.S);
          expand_runs<T, VCS>(k, pipe.buf(i % kStages), sv.vptr[sv.ptr[sa]], sv.vptr[sv.ptr[sb]],
                              sv.ptr[sa], sv.ptr[sb]);
        }
        const int s = k.s0 + u * a.S + sub;
        const bool mine = s < k.s1;
        int n0 = 0, n1 = 0;
        if (mine) {
          if (VCS) {
            n0 = sv.vptr[sv.ptr[s]];
            n1 = sv.vptr[sv.ptr[s + 1]];
          } else {
            n0 = sv.ptr[s];
            n1 = sv.ptr[s + 1];
          }
        }
        gather_range<T, VEC, Q, NP, CI, VCS>(sv, X, a.ldx, n0, n1, G, slot, col0, colok, acc);
        if (mine && slot == 0) {
#pragma unroll
          for (int ci = 0; ci < CI; ++ci)
            if (colok[ci])
              *reinterpret_cast<V *>(Y + (int64_t)s * a.ldy + col0[ci]) = Ops::pack(acc[0][ci]);
        }
      } else {
        // ---- share u of a chunk of a long slice: publish its partial; the last
        // share of the slice to arrive adds all of them in share order
        if (VCS)
          expand_runs<T, VCS>(k, pipe.buf(i % kStages), k.e0 + u * kShareEntries,
                              min(k.e1, k.e0 + (u + 1) * kShareEntries), k.r0, k.r1);
        const int n0 = sub == 0 ? k.e0 + u * kShareEntries : 0;
        const int n1 = sub == 0 ? min(k.e1, n0 + kShareEntries) : 0;
        gather_range<T, VEC, Q, NP, CI, VCS>(sv, X, a.ldx, n0, n1, G, slot, col0, colok, acc);
        T *__restrict__ P = static_cast<T *>(a.partials);
        if (sub == 0 && slot == 0) {
#pragma unroll
          for (int ci = 0; ci < CI; ++ci)
            if (colok[ci])
              *reinterpret_cast<V *>(P + (int64_t)(k.first + u) * kMaxBlockWidth + col0[ci]) =
                  Ops::pack(acc[0][ci]);
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(a.counters + k.lid, 1) == k.nsh - 1;
        last = __shfl_sync(kFullMask, last, 0);
        if (last) {
          __threadfence();
          for (int c = lane; c < a.w; c += 32) {
            T sum = __ldcg(P + (int64_t)k.sfirst * kMaxBlockWidth + c);
            for (int q = 1; q < k.nsh; ++q)
              sum = sum + __ldcg(P + (int64_t)(k.sfirst + q) * kMaxBlockWidth + c);
            Y[(int64_t)k.s0 * a.ldy + c] = sum;
          }
          if (lane == 0) a.counters[k.lid] = 0;  // re-armed for the next launch
        }
      }
    }
    pipe.release(i);
  }
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
  constexpr int smem = pipe_smem_bytes<T, VCS>(0);
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
    a.st = StageArrays{m.ptr, m.idx, m.vals, m.vptr, m.blocks, (int)m.n_blocks, m.err,
                       nullptr, 0, 0, 0};
    a.X = xp;
    a.ldx = X.ld;
    a.Y = yp;
    a.ldy = Y.ld;
    a.w = wb;
    a.G = G;
    a.S = 32 / (Q * G);
    a.partials = m.partials;
    a.counters = m.counters;
    int per_sm = 0;
    VS_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    VS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kPipeThreads, smem));
    const int64_t grid = std::min<int64_t>(m.n_blocks, (int64_t)std::max(1, per_sm) * m.n_sm);
    if (grid > 0) {
      k<<<(unsigned)grid, kPipeThreads, smem, s>>>(a);
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
