// gather_impl.cuh -- the aligned direction: Y[s, :] = sum over the entries
// (t, a) of major slice s of a * X[t, :].  Covers CSR@B, VCSR@B, B@VCSC and
// B@CSC (every aligned product maps onto this slice frame, see vs_api.cu), and
// the misaligned products that run over an attached exact transpose.
// Instantiated per value type and layout by gather_f32_csr.cu,
// gather_f32_vcs.cu and gather_f64_csr.cu.
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
//   * a run of entries (a whole short slice, or one share of a long slice) is
//     summed as g logical partials -- partial k takes the entries n with
//     (n - start) mod g == k, with fused multiply-adds in entry order -- which
//     meet in the butterfly p[k] += p[k + h], h = g/2, ..., 1;
//   * a long slice is cut into chunks (at most kBlockEntries entries and
//     kBlockRuns runs, cut points fixed by the matrix) and every chunk into
//     shares of kShareEntries entries; share_combine_kernel adds the m share
//     results of the slice: lane j of a warp sums shares j, j + 32, ... in
//     order, then the 32 lane sums meet in a butterfly.
// Physically G slots of a slice each hold NP = g / G partials in registers
// (Q lanes per slot across a tile of Q * VEC columns; wider products take
// several column passes over the same staged entries; narrow ones put several
// slices in one warp).  In-lane adds, then shuffles, reproduce the same tree
// for every width, so bits never depend on w, nor on where X is read from.
//
// Data movement: entries, values, slice pointers, runs and the block's
// descriptor arrive in shared memory by bulk copies through a ring of stage
// buffers fed by a producer warp (stage.cuh); VCS run values are expanded to
// per-entry values in shared memory by the producer side.  The dense rows
// X[t, :] come either from a shared-memory slab holding all of X (when it
// fits: one CTA per SM copies it in once) or through L1 with 16-byte vector
// loads.
#pragma once

#include <algorithm>

#include "stage.cuh"

namespace vs {
namespace gather_detail {

struct GatherArgs {
  StageArrays st;
  const void *X;
  int64_t ldx;
  void *Y;
  int64_t ldy;
  int w;           // columns in this launch (<= kMaxBlockWidth)
  int n_x;         // rows of X (shared-memory variant: rows copied into the slab)
  void *partials;  // [n_shares][kMaxBlockWidth] of T
  const void *yscale;  // optional: Y[s, :] *= yscale[s] at the store
  int stall;           // test hook: the producer issues nothing (see vs_test_stall_producers)
};

// Where the rows X[t, :] come from.  Each lane holds the address of its own
// VEC columns in row 0 (a valid column even for lanes past the width, whose
// results are never stored, so loads need no predicate).
template <typename T, int VEC, bool XS>
struct XSource;
// Through L1: X in global memory, row stride `ldb` bytes.
template <typename T, int VEC>
struct XSource<T, VEC, false> {
  using V = typename VecT<T, VEC>::type;
  const char *base;
  uint32_t ldb;
  __device__ __forceinline__ V load(int t) const {
    return ld_gather(reinterpret_cast<const V *>(base + (size_t)(uint32_t)t * ldb));
  }
};
// Shared memory: a slab of X whose rows hold one column pass (Q * VEC
// elements), copied in once per CTA.
template <typename T, int VEC>
struct XSource<T, VEC, true> {
  using V = typename VecT<T, VEC>::type;
  uint32_t base;
  uint32_t row;  // bytes per slab row
  __device__ __forceinline__ V load(int t) const { return ld_shared<V>(base + (uint32_t)t * row); }
};

// Sums entries [n0, n1) of one slice for this lane's VEC columns and runs the
// fixed tree; acc[0] holds the result in the slice's slot-0 lanes.
template <typename T, typename TV, int VEC, int Q, int G, int NP, bool VCS, class XSrc>
__device__ __forceinline__ void gather_range(const Staged<TV, VCS> &sv, const XSrc &xs, int n0,
                                             int n1, int slot, T (&acc)[NP][VEC]) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  constexpr int STEP = G * NP;
#pragma unroll
  for (int i = 0; i < NP; ++i)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[i][e] = T(0);
  const int nfull = (n1 - n0) / STEP;
  int n = n0 + slot;
  int it = 0;
  // two steps at a time: 2 NP independent loads in flight per lane
  for (; it + 1 < nfull; it += 2, n += 2 * STEP) {
    int j[2 * NP];
    T av[2 * NP];
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) {
      j[i] = sv.idx[n + i * G];
      av[i] = static_cast<T>(sv.vals[n + i * G]);
    }
    V x[2 * NP];
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) x[i] = xs.load(j[i]);
#pragma unroll
    for (int i = 0; i < 2 * NP; ++i) {  // step it, then step it + 1, partial by partial
      T xe[VEC];
      Ops::unpack(x[i], xe);
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i % NP][e] = fma(av[i], xe[e], acc[i % NP][e]);
    }
  }
  for (; it < nfull; ++it, n += STEP) {
    int j[NP];
    T av[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      j[i] = sv.idx[n + i * G];
      av[i] = static_cast<T>(sv.vals[n + i * G]);
    }
    V x[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) x[i] = xs.load(j[i]);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      T xe[VEC];
      Ops::unpack(x[i], xe);
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i][e] = fma(av[i], xe[e], acc[i][e]);
    }
  }
  // the last, partial step
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const int nn = n + i * G;
    if (nn < n1) {
      const int jj = sv.idx[nn];
      const T a = static_cast<T>(sv.vals[nn]);
      const V x = xs.load(jj);
      T xe[VEC];
      Ops::unpack(x, xe);
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i][e] = fma(a, xe[e], acc[i][e]);
    }
  }
  // the fixed tree: in-lane levels (strides h*G), then across slots (strides < G)
#pragma unroll
  for (int h = NP / 2; h >= 1; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[i][e] = acc[i][e] + acc[i + h][e];
#pragma unroll
  for (int sft = G / 2; sft >= 1; sft >>= 1)
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      acc[0][e] = acc[0][e] + __shfl_xor_sync(kFullMask, acc[0][e], sft * Q);
}

// Launch shape.  XS = true keeps X in shared memory: 16 consumer warps, 8
// stage buffers, one CTA per SM, the slab taking the rest of the SM's shared
// memory.  XS = false gathers X through L1, two CTAs per SM so that more
// operand rows are in flight from L2: CSR with 12 consumer warps and 6 stage
// buffers each, with one producer warp; VCS with 10 consumer warps and 6 stage
// buffers each.  Expanding VCS run values is a chain of shared-memory round
// trips that one warp cannot keep ahead of the consumers, so VCS splits the
// producer into one issuing warp and kExpanders expanding warps (4 beside the
// slab's 16 consumers, 2 beside the L1 shape's 10).
template <bool XS, bool VCS>
struct GatherShape {
  static constexpr int kWarps = XS ? 16 : (VCS ? 10 : 12);
  static constexpr int kStageBufs = XS ? 8 : 6;
  static constexpr int kExpanders = VCS ? (XS ? 4 : 2) : 0;
  static constexpr int kThreads = (kWarps + 1 + kExpanders) * 32;
  static constexpr int kMinCtas = XS ? 1 : 2;
  // Consumer groups: block i of a CTA goes to group i mod kGroups only, so a
  // warp pays the per-block bookkeeping for 1 / kGroups of the blocks.  Each
  // stage buffer always serves the same group (kGroups divides the stages).
  static constexpr int kGroups = 2;
  static_assert(kStageBufs % kGroups == 0 && kWarps % kGroups == 0, "uneven consumer groups");
  static_assert(kExpanders == 0 || kStageBufs % kExpanders == 0,
                "each stage buffer must always go to the same expanding warp");
};

template <typename T, typename TV, int VEC, int Q, int G, int NP, bool VCS, bool XS>
__global__ void __launch_bounds__(GatherShape<XS, VCS>::kThreads, GatherShape<XS, VCS>::kMinCtas)
    gather_kernel(const GatherArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  using Shape = GatherShape<XS, VCS>;
  constexpr int NW = Shape::kWarps;
  constexpr int NS = Shape::kStageBufs;
  constexpr int S = 32 / (Q * G);  // slices per warp work unit
  constexpr int TW = Q * VEC;      // columns per pass
  extern __shared__ __align__(128) unsigned char smem[];
  const Pipe<TV, VCS, NS> pipe{smem};
  constexpr int GW = NW / Shape::kGroups;  // consumer warps per group
  pipe.init(GW);
  grid_dependency_wait();  // may start while the previous kernel of the stream finishes
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (wid >= NW) {  // the producer warp(s)
    if (a.stall) return;  // nothing issued: every consumer wait gives up after its limit
    if constexpr (Shape::kExpanders == 0)
      pipe.produce(a.st, blockIdx.x, a.st.n_blocks, gridDim.x);
    else if (wid == NW)
      pipe.issue_all(a.st, blockIdx.x, a.st.n_blocks, gridDim.x);
    else
      pipe.expand_share(a.st, blockIdx.x, a.st.n_blocks, gridDim.x, wid - NW - 1,
                        Shape::kExpanders);
    return;
  }
  const int ql = lane % Q;
  const int slot = (lane / Q) % G;
  const int sub = lane / (Q * G);
  const T *__restrict__ X = static_cast<const T *>(a.X);
  T *__restrict__ Y = static_cast<T *>(a.Y);
  const T *__restrict__ ys = static_cast<const T *>(a.yscale);
  T *__restrict__ P = static_cast<T *>(a.partials);
  const int w = a.w;
  const int npass = (w + TW - 1) / TW;

  // XS: copy X[:, 0:w) into the slab, pass by pass ([pass][row][TW], columns
  // past w zero), while the producer already streams the first blocks
  T *slab = reinterpret_cast<T *>(smem + PipeLayout<TV, VCS, NS>::kExtra);
  if constexpr (XS) {
    if (npass == 1 && w == TW && a.ldx == TW && (TW * sizeof(T)) % 16 == 0 &&
        (reinterpret_cast<uintptr_t>(X) & 15) == 0) {
      // X is already in the slab's layout (rows of exactly one pass): bulk
      // copies bring it in while the producer streams the first blocks
      const uint32_t total = (uint32_t)a.n_x * TW * (uint32_t)sizeof(T);
      if (threadIdx.x == 0) {
        constexpr uint32_t kChunk = 32768;
        mbar_arrive_expect_tx(pipe.slab_landed(), total);
        for (uint32_t off = 0; off < total; off += kChunk)
          bulk_load(reinterpret_cast<unsigned char *>(slab) + off,
                    reinterpret_cast<const unsigned char *>(X) + off, min(kChunk, total - off),
                    pipe.slab_landed());
      }
      if (!mbar_wait_bounded(pipe.slab_landed(), 0, kWaitLimitNs)) {
        pipe.give_up(a.st);
        return;
      }
    } else {
      const int nv = a.n_x * Q;  // vectors per pass
      for (int p = 0; p < npass; ++p)
        for (int v = threadIdx.x; v < nv; v += NW * 32) {
          const int r = v / Q, c = p * TW + (v % Q) * VEC;
          V x{};
          if (c < w) x = ld_gather(reinterpret_cast<const V *>(X + (int64_t)r * a.ldx + c));
          *reinterpret_cast<V *>(slab + ((int64_t)p * a.n_x + r) * TW + (v % Q) * VEC) = x;
        }
      named_barrier(1, NW * 32);
    }
  }
  auto source = [&](int cp) {
    // this lane's columns in pass cp / TW; lanes past the width read column 0
    const int col = cp + ql * VEC < w ? ql * VEC : 0;
    if constexpr (XS) {
      return XSource<T, VEC, true>{
          smem_u32(slab + (size_t)(cp / TW) * a.n_x * TW + col), (uint32_t)(TW * sizeof(T))};
    } else {
      return XSource<T, VEC, false>{reinterpret_cast<const char *>(X + cp + col),
                                    (uint32_t)(a.ldx * (int64_t)sizeof(T))};
    }
  };

  const int gw = wid % GW;  // this warp's place in its group
  int i = wid / GW, rot = 0;  // rot: units the group handed out so far, mod GW
  for (int b = blockIdx.x + i * gridDim.x; b < a.st.n_blocks;
       b += Shape::kGroups * gridDim.x, i += Shape::kGroups) {
    if (!pipe.acquire(i, a.st)) return;
    unsigned char *buf = pipe.buf(i % NS);
    const Block k = stage_desc<TV, VCS>(buf);
    const Staged<TV, VCS> sv = stage_views<TV, VCS>(k, buf);
    const int units = block_units(k, S);
    T acc[NP][VEC];
    // work units go round-robin to the consumer warps, continuing across blocks
    const int u0 = (gw - rot + GW) % GW;
    rot = (rot + units) % GW;
    for (int u = u0; u < units; u += GW) {
      if (k.type == 0) {
        // ---- S consecutive slices, one per sub-group
        const int sa = k.s0 + u * S;
        const int s = sa + sub;
        const bool mine = s < k.s1;
        int n0 = 0, n1 = 0;
        if (mine) {
          n0 = VCS ? sv.vptr[sv.ptr[s]] : sv.ptr[s];
          n1 = VCS ? sv.vptr[sv.ptr[s + 1]] : sv.ptr[s + 1];
        }
        for (int cp = 0; cp < npass * TW; cp += TW) {
          const int col = cp + ql * VEC;
          gather_range<T, TV, VEC, Q, G, NP, VCS>(sv, source(cp), n0, n1, slot, acc);
          if (mine && slot == 0 && col < w) {
            if (ys) {
              const T f = ys[s];
#pragma unroll
              for (int e = 0; e < VEC; ++e) acc[0][e] = acc[0][e] * f;
            }
            *reinterpret_cast<V *>(Y + (int64_t)s * a.ldy + col) = Ops::pack(acc[0]);
          }
        }
      } else {
        // ---- share u of a chunk of a long slice: its partial goes to the
        // share table; share_combine_kernel adds the shares of each slice
        const int na = k.e0 + u * kShareEntries, nb = min(k.e1, na + kShareEntries);
        const int n0 = sub == 0 ? na : 0, n1 = sub == 0 ? nb : 0;
        for (int cp = 0; cp < npass * TW; cp += TW) {
          const int col = cp + ql * VEC;
          gather_range<T, TV, VEC, Q, G, NP, VCS>(sv, source(cp), n0, n1, slot, acc);
          if (sub == 0 && slot == 0 && col < w)
            *reinterpret_cast<V *>(P + (int64_t)(k.first + u) * kMaxBlockWidth + col) =
                Ops::pack(acc[0]);
        }
      }
    }
    pipe.release(i);
  }
}

// Y[s, c] of every long slice s from its share partials p_0 .. p_{m-1}: 32
// lane sums s_j = p_j + p_{j+32} + ... (in order, from zero), then the
// butterfly s_j += s_{j^h}, h = 16, 8, 4, 2, 1.  One warp per long slice:
// lane j loads whole partial rows (16 columns at a time, 16-byte vectors),
// so every load of the warp is in flight at once.  The order depends on the
// share count alone.
template <typename T>
__global__ void __launch_bounds__(256) share_combine_kernel(const T *__restrict__ P,
                                                            const int4 *__restrict__ longs,
                                                            int64_t n_long, int w,
                                                            T *__restrict__ Y, int64_t ldy,
                                                            const T *__restrict__ ys) {
  constexpr int VW = 16 / sizeof(T);  // elements per 16-byte vector
  constexpr int CB = 16;              // columns per pass
  using V = typename VecT<T, VW>::type;
  using Ops = VecOps<T, VW>;
  const int lane = threadIdx.x & 31;
  const int64_t l = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  grid_dependency_wait();  // launched early: the gather's partials must be complete
  if (l >= n_long) return;
  const int4 d = longs[l];  // {slice, first share, shares, 0}
  // columns [c0, c0 + CB) of a partial row lie inside its kMaxBlockWidth
  // slots (entries past w hold no result and are never stored)
  for (int c0 = 0; c0 < w; c0 += CB) {
    T s[CB];
#pragma unroll
    for (int e = 0; e < CB; ++e) s[e] = T(0);
    // rows lane, lane + 32, ...: kRows of them loaded before their adds
    constexpr int kRows = 4;
    for (int q0 = lane; q0 < d.z; q0 += 32 * kRows) {
      V v[kRows][CB / VW];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int q = q0 + 32 * r;
        const V *row = reinterpret_cast<const V *>(P + (int64_t)(d.y + q) * kMaxBlockWidth + c0);
#pragma unroll
        for (int k = 0; k < CB / VW; ++k) v[r][k] = q < d.z ? __ldcg(row + k) : V{};
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (q0 + 32 * r >= d.z) break;
#pragma unroll
        for (int k = 0; k < CB / VW; ++k) {
          T x[VW];
          Ops::unpack(v[r][k], x);
#pragma unroll
          for (int e = 0; e < VW; ++e) s[k * VW + e] = s[k * VW + e] + x[e];
        }
      }
    }
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
      for (int e = 0; e < CB; ++e) s[e] = s[e] + __shfl_xor_sync(kFullMask, s[e], h);
    T out = s[0];
#pragma unroll
    for (int e = 1; e < CB; ++e)
      if (lane == e) out = s[e];
    if (ys) out = out * ys[d.x];
    if (lane < CB && c0 + lane < w) Y[(int64_t)d.x * ldy + c0 + lane] = out;
  }
}

// ------------------------------------------------------------------ dispatch

template <typename T, bool VCS>
using KernelPtr = void (*)(const GatherArgs);

// Slots per slice G = min(g, kMaxSlots); each lane then holds NP = g / G <= 4
// logical partials, and a warp works on 32 / (Q G) slices at a time.
#ifndef VS_MAX_SLOTS
#define VS_MAX_SLOTS 8
#endif
constexpr int kMaxSlots = VS_MAX_SLOTS;

template <typename T, typename TV, int VEC, int Q, int G, bool VCS, bool XS>
KernelPtr<T, VCS> pick_np(int np) {
  if constexpr (G == kMaxSlots || G * Q == 32) {
    if constexpr (Q * G * 2 <= 64)
      if (np == 2) return gather_kernel<T, TV, VEC, Q, G, 2, VCS, XS>;
    if constexpr (Q * G * 4 <= 128)
      if (np == 4) return gather_kernel<T, TV, VEC, Q, G, 4, VCS, XS>;
  }
  return np == 1 ? gather_kernel<T, TV, VEC, Q, G, 1, VCS, XS> : nullptr;
}

template <typename T, typename TV, int VEC, int Q, bool VCS, bool XS>
KernelPtr<T, VCS> pick_g(int G, int np) {
  switch (G) {
    case 1: return pick_np<T, TV, VEC, Q, 1, VCS, XS>(np);
    case 2: return pick_np<T, TV, VEC, Q, 2, VCS, XS>(np);
    case 4: return pick_np<T, TV, VEC, Q, 4, VCS, XS>(np);
    case 8: return pick_np<T, TV, VEC, Q, 8, VCS, XS>(np);
    case 16: if constexpr (kMaxSlots >= 16 && Q <= 2) return pick_np<T, TV, VEC, Q, 16, VCS, XS>(np); break;
    case 32: if constexpr (kMaxSlots >= 32 && Q == 1) return pick_np<T, TV, VEC, Q, 32, VCS, XS>(np); break;
  }
  return nullptr;
}

template <typename T, typename TV, int VEC, bool VCS, bool XS>
KernelPtr<T, VCS> pick_q(int Q, int G, int np) {
  switch (Q) {
    case 1: return pick_g<T, TV, VEC, 1, VCS, XS>(G, np);
    case 2: return pick_g<T, TV, VEC, 2, VCS, XS>(G, np);
    case 4: return pick_g<T, TV, VEC, 4, VCS, XS>(G, np);
  }
  return nullptr;
}

// Lane tiling of a launch of wb columns: 16-byte vectors when the operands
// allow them, Q lanes per slot (one vector, or one element, each, up to 4),
// TW = Q * VEC columns per pass.
struct Tiling {
  bool vec;
  int Q, TW;
};
template <typename T>
Tiling gather_tiling(int wb, const void *xp, const void *yp, int64_t ldx, int64_t ldy) {
  constexpr int VW = 16 / sizeof(T);
  const bool vec = wb % VW == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(yp) % 16 == 0 && ldx % VW == 0 && ldy % VW == 0;
  const int ncol = vec ? wb / VW : wb;
  const int Q = ncol >= 3 ? 4 : ncol;
  return Tiling{vec, Q, Q * (vec ? VW : 1)};
}

// Shared memory per CTA beyond the pipeline that the X slab may take.
constexpr int64_t kSmemOptIn = 227 * 1024;
template <typename TV, bool VCS>
constexpr int64_t slab_budget() {
  return kSmemOptIn - pipe_smem_bytes<TV, VCS, GatherShape<true, VCS>::kStageBufs>(0);
}

// Whether X fits the shared-memory slab for at least one column pass.
template <typename T, typename TV, bool VCS>
bool slab_fits(const Matrix &m, DenseView X, DenseView Y, int64_t w) {
  const int wb = (int)std::min<int64_t>(kMaxBlockWidth, w);
  const Tiling t = gather_tiling<T>(wb, X.p, Y.p, X.ld, Y.ld);
  return m.n_minor > 0 && m.n_minor * t.TW * (int64_t)sizeof(T) <= slab_budget<TV, VCS>();
}

// T: the dense operands and sums; TV: the stored values (float for VCS, and
// for a float CSR matrix with double operands).
template <typename T, typename TV, bool VCS, bool XS>
vs_status launch_typed(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s) {
  constexpr int VW = 16 / sizeof(T);
  using Shape = GatherShape<XS, VCS>;
  if ((uint64_t)X.ld * sizeof(T) >= (uint64_t(1) << 32)) {  // row offsets are 32-bit products
    set_error("dense operand row stride too large");
    return VS_ERR_UNSUPPORTED;
  }
  for (int64_t c0 = 0; c0 < w;) {
    int wb = (int)std::min<int64_t>(kMaxBlockWidth, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    const Tiling t = gather_tiling<T>(wb, xp, yp, X.ld, Y.ld);
    int64_t slab = 0;
    if constexpr (XS) {
      const int64_t pass = m.n_minor * t.TW * (int64_t)sizeof(T);
      const int64_t fit = slab_budget<TV, VCS>() / pass;  // column passes the slab holds
      if (fit < 1) {
        set_error("dense operand does not fit the shared-memory slab");
        return VS_ERR_UNSUPPORTED;
      }
      wb = (int)std::min<int64_t>(wb, fit * t.TW);
      slab = (wb + t.TW - 1) / t.TW * pass;
    }
    const int G = std::min(std::min(m.g, kMaxSlots), 32 / t.Q);
    const int NP = m.g / G;
    KernelPtr<T, VCS> k = t.vec ? pick_q<T, TV, VW, VCS, XS>(t.Q, G, NP)
                                : pick_q<T, TV, 1, VCS, XS>(t.Q, G, NP);
    if (!k) {
      set_error("no gather kernel for this width and group size");
      return VS_ERR_UNSUPPORTED;
    }
    const int smem = pipe_smem_bytes<TV, VCS, Shape::kStageBufs>((int)slab);
    GatherArgs a;
    a.st = StageArrays{m.ptr, m.idx, m.vals, m.vptr, m.blocks, (int)m.n_blocks, m.err,
                       nullptr, 0, 0, 0};
    a.X = xp;
    a.ldx = X.ld;
    a.Y = yp;
    a.ldy = Y.ld;
    a.w = wb;
    a.n_x = (int)m.n_minor;
    a.partials = m.partials;
    a.yscale = Y.scale;
    a.stall = take_stall() ? 1 : 0;
    int per_sm = 0;
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), Shape::kThreads, smem, &per_sm));
    const int64_t grid = std::min<int64_t>(m.n_blocks, (int64_t)std::max(1, per_sm) * m.n_sm);
    if (grid > 0) {
      VS_CUDA(launch_early(k, dim3((unsigned)grid), dim3(Shape::kThreads), smem, s, a));
      VS_LAUNCH_CHECK();
    }
    if (m.n_long > 0) {
      VS_CUDA(launch_early(share_combine_kernel<T>, dim3((unsigned)((m.n_long + 7) / 8)), dim3(256),
                           0, s, static_cast<const T *>(m.partials),
                           static_cast<const int4 *>(m.longs), m.n_long, wb, yp, Y.ld,
                           static_cast<const T *>(Y.scale)));
      VS_LAUNCH_CHECK();
    }
    c0 += wb;
  }
  return VS_OK;
}

}  // namespace gather_detail
}  // namespace vs
