// scatter.cu -- the misaligned direction: for every major slice s and entry
// (t, a) of s, Y[t, :] += a * X[s, :].  Covers VCSC@B, B@VCSR, CSC@B and B@CSR.
//
// "Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": the misaligned directions add into the output with atomics, which
// makes them nondeterministic in the last bits.  Two schemes live here, both
// fed by the block stream of stage.cuh (entries arrive in shared memory by
// bulk copies, a block ahead):
//
//  * atomic: zero-fill Y, then warps take slices (or shares of a chunk of a
//    long slice), load X[s, :] once and add a * X[s, :] into row t with
//    vector reductions (red.global.add.v4.f32).
//
//  * two-phase (deterministic): the blocks are cut into C consecutive groups
//    (balanced by entries, C fixed by the matrix) and Y into tiles of rows that
//    fit in shared memory.  Phase 1: CTA (tile, group) streams its group's
//    blocks in order and accumulates, in slice order and entry order, the
//    contributions that land in its tile; each warp owns the tile rows t with
//    t mod 8 equal to its number (interleaved, so the popular rows of a skewed
//    matrix spread over the warps), so no two threads update one element
//    concurrently, and duplicate
//    rows met together are applied one after another in entry order.  Phase 2
//    adds the C group partials of every element in group order.  The order of
//    every element's sum therefore depends on the matrix alone.
#include <algorithm>
#include <mutex>
#include <string>

#include "stage.cuh"

namespace vs {
namespace {

__device__ __forceinline__ float fma_t(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fma_t(double a, double b, double c) { return fma(a, b, c); }

// ------------------------------------------------------------------ atomic

struct ScatterArgs {
  StageArrays st;
  const void *X;
  int64_t ldx;
  void *Y;
  int64_t ldy;
  int w;
  int G;  // slots per slice
  int S;  // slices per warp task
};

// Entries [n0, n1) of slice s: Y[t, :] += a * x for each, slot-strided.
template <typename T, int VEC, int Q, int CI, bool VCS>
__device__ __forceinline__ void scatter_range(const Staged<T, VCS> &sv, const T (&x)[CI][VEC],
                                              T *__restrict__ Y, int64_t ldy, int n0, int n1,
                                              int G, int slot, const int (&col0)[CI],
                                              const bool (&colok)[CI]) {
#pragma unroll 4
  for (int n = n0 + slot; n < n1; n += G) {
    const int t = sv.idx[n];
    const T av = sv.vals[n];
#pragma unroll
    for (int ci = 0; ci < CI; ++ci) {
      if (!colok[ci]) continue;
      T c[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) c[e] = av * x[ci][e];
      red_add(Y + (int64_t)t * ldy + col0[ci], c);
    }
  }
}

template <typename T, int VEC, int Q, int CI, bool VCS>
__global__ void __launch_bounds__(kPipeThreads) scatter_atomic_kernel(const ScatterArgs a) {
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

  int i = 0, rot = 0;  // rot: units handed out so far, mod kWarpsPerCta
  for (int b = blockIdx.x; b < a.st.n_blocks; b += gridDim.x, ++i) {
    if (!pipe.acquire(i, a.st)) return;
    const Block k = stage_desc<T, VCS>(pipe.buf(i % kStages));
    const Staged<T, VCS> sv = stage_views<T, VCS>(k, pipe.buf(i % kStages));
    const int units = block_units(k, a.S);
    T x[CI][VEC];
    // work units go round-robin to the consumer warps, continuing across blocks
    const int u0 = (wid - rot + kWarpsPerCta) % kWarpsPerCta;
    rot = (rot + units) % kWarpsPerCta;
    for (int u = u0; u < units; u += kWarpsPerCta) {
      int s, n0 = 0, n1 = 0;
      if (k.type == 0) {
        s = k.s0 + u * a.S + sub;
        if (s < k.s1) {
          if (VCS) {
            n0 = sv.vptr[sv.ptr[s]];
            n1 = sv.vptr[sv.ptr[s + 1]];
          } else {
            n0 = sv.ptr[s];
            n1 = sv.ptr[s + 1];
          }
        }
      } else {
        s = k.s0;
        if (sub == 0) {
          n0 = k.e0 + u * kShareEntries;
          n1 = min(k.e1, n0 + kShareEntries);
        }
      }
      if (n0 < n1) {
#pragma unroll
        for (int ci = 0; ci < CI; ++ci)
          if (colok[ci])
            Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)s * a.ldx + col0[ci])),
                        x[ci]);
        scatter_range<T, VEC, Q, CI, VCS>(sv, x, Y, a.ldy, n0, n1, G, slot, col0, colok);
      }
    }
    pipe.release(i);
  }
}

// ------------------------------------------------------------------ zero fill

// Y[r, c] += T[r, c] (T contiguous with row stride w)
template <typename T>
__global__ void add_into_kernel(const T *__restrict__ src, int64_t rows, int64_t w,
                                T *__restrict__ Y, int64_t ld) {
  const int64_t total = rows * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / w, c = i - r * w;
    Y[r * ld + c] = Y[r * ld + c] + src[i];
  }
}

template <typename T>
__global__ void zero_fill_kernel(T *__restrict__ Y, int64_t rows, int64_t w, int64_t ld) {
  const int64_t total = rows * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / w, c = i - r * w;
    Y[r * ld + c] = T(0);
  }
}

__global__ void zero_fill_vec_kernel(float4 *__restrict__ Y, int64_t n16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    Y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ two-phase

struct TwoPhaseArgs {
  StageArrays st;
  const void *X;
  int64_t ldx;
  void *out;              // Y (C == 1) or the group partials
  int64_t ldo;            // row stride of `out`
  int64_t part_stride;    // elements between group partials (C > 1)
  const int32_t *bounds;  // [C+1] block boundaries of the groups
  int64_t n_t;            // rows of Y
  int tile_rows;          // rows per tile
  int w;
  int sorted;             // minor indices ascend inside every run / row
};

// Per-stage record list: the block's entries whose row lies in this CTA's
// tile, in entry order -- key = tile-relative row | (slice - s0) << 16.
template <typename T>
struct RecLayout {
  static constexpr int kKey = 0;
  static constexpr int kVal = kKey + kCapEntries * 4;
  // records sorted by owning warp: warp w's are [kOff[w], kOff[w + 1])
  static constexpr int kOff = kVal + kCapEntries * (int)sizeof(T);
  static constexpr int kBytes = (kOff + 4 * (kWarpsPerCta + 1) + 127) / 128 * 128;
};

// Producer-side scratch (one per CTA): start bitmaps of slices and runs, and
// the ids of the non-empty slices of the current block.
struct PrepLayout {
  static constexpr int kWords = (kCapEntries + 31) / 32 + 1;
  static constexpr int kSliceBits = 0;
  static constexpr int kRunBits = kSliceBits + kWords * 4;
  static constexpr int kSliceIds = kRunBits + kWords * 4;
  static constexpr int kCursor = kSliceIds + kCapSlices * 4;           // per owning warp
  static constexpr int kRange = kCursor + 4 * kWarpsPerCta;            // per run: [a0, b0)
  static constexpr int kBytes = (kRange + 8 * kCapRuns + 127) / 128 * 128;
};


// Two-phase CTA: kWarpsPerCta consumer warps, one warp issuing the copies and
// kPreparers warps turning landed blocks into records (block i goes to
// preparer i mod kPreparers; it divides kStages, so a stage always goes to
// the same preparer and a parity wait never sees an old phase).
constexpr int kPreparers = 4;
constexpr int kTwoPhaseThreads = (kWarpsPerCta + 1 + kPreparers) * 32;
static_assert(kStages % kPreparers == 0, "each stage must always go to the same preparer");

template <typename T, bool VCS>
struct TwoPhaseSmem {
  static constexpr int kPipe = 0;
  static constexpr int kRecs = PipeLayout<T, VCS>::kExtra;
  static constexpr int kPrep = kRecs + kStages * RecLayout<T>::kBytes;
  static constexpr int kTile = kPrep + kPreparers * PrepLayout::kBytes;
};

// First position p in [lo, hi) with idx[p] >= key (hi if none) over indices
// that ascend on [lo, hi), by the whole warp: while more than 32 candidates
// remain, the lanes test the starts of 32 equal segments and the ballot
// keeps the segment holding the boundary; then each lane tests one candidate.
// A block's run (at most kBlockEntries entries) takes two rounds of loads.
__device__ __forceinline__ int warp_lower_bound(const int32_t *idx, int lo, int hi, int key) {
  const int lane = threadIdx.x & 31;
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int p = lo + (lane + 1) * step;
    const int nl = __popc(__ballot_sync(kFullMask, p < hi && idx[p] < key));
    lo += nl * step;
    hi = min(lo + step, hi);
  }
  const int p = lo + lane;
  return lo + __popc(__ballot_sync(kFullMask, p < hi && idx[p] < key));
}

// Producer warp: once block j (number b) has landed, write the records of its
// entries that fall in rows [t0, t0 + rows), in entry order, and mark the
// stage ready.  The slice of an entry and (VCS) its run come from start
// bitmaps counted with popcounts; for sorted runs and a partial tile, only
// each run's sub-range inside the tile is visited.
template <typename T, bool VCS>
__device__ __forceinline__ bool two_phase_prepare(const Pipe<T, VCS> &pipe, const StageArrays &a,
                                                  int j, int b, unsigned char *recs,
                                                  unsigned char *prep, int64_t t0, int rows,
                                                  bool skip_by_search) {
  using LY = StageLayout<T, VCS>;
  using RL = RecLayout<T>;
  const int s = j % kStages;
  if (!mbar_wait_bounded(pipe.full(s), (j / kStages) & 1, kWaitLimitNs)) return false;
  const int lane = threadIdx.x & 31;
  const unsigned lt = lanemask_lt(), le = lt | (1u << lane);
  unsigned char *bp = pipe.buf(s);
  const Block k = stage_desc<T, VCS>(bp);
  const Staged<T, VCS> sv = stage_views<T, VCS>(k, bp);
  const float *rv = VCS ? reinterpret_cast<const float *>(bp + LY::kRvals) - align_down<4>(k.r0)
                        : nullptr;
  unsigned char *rb = recs + s * RL::kBytes;
  uint32_t *key = reinterpret_cast<uint32_t *>(rb + RL::kKey);
  T *val = reinterpret_cast<T *>(rb + RL::kVal);
  int *off = reinterpret_cast<int *>(rb + RL::kOff);
  uint32_t *sbm = reinterpret_cast<uint32_t *>(prep + PrepLayout::kSliceBits);
  uint32_t *rbm = reinterpret_cast<uint32_t *>(prep + PrepLayout::kRunBits);
  int32_t *sid = reinterpret_cast<int32_t *>(prep + PrepLayout::kSliceIds);
  int *cur = reinterpret_cast<int *>(prep + PrepLayout::kCursor);
  int *rng = reinterpret_cast<int *>(prep + PrepLayout::kRange);
  const int eb = align_down<4>(k.e0);
  const int nwords = (k.e1 - eb + 31) / 32;
  constexpr int kOwnMask = kWarpsPerCta - 1;

  // slice and run start bitmaps over the block's entries
  for (int q = lane; q < nwords; q += 32) {
    sbm[q] = 0u;
    if (VCS) rbm[q] = 0u;
  }
  if (lane < kWarpsPerCta) cur[lane] = 0;
  __syncwarp();
  int ns = 0;  // non-empty slices, in order
  if (k.type == 0) {
    for (int base = k.s0; base < k.s1; base += 32) {
      const int sl = base + lane;
      const bool ne = sl < k.s1 &&
                      (VCS ? sv.vptr[sv.ptr[sl]] < sv.vptr[sv.ptr[sl + 1]] : sv.ptr[sl] < sv.ptr[sl + 1]);
      const unsigned m = __ballot_sync(kFullMask, ne);
      if (ne) {
        sid[ns + __popc(m & lt)] = sl - k.s0;
        const int st = (VCS ? sv.vptr[sv.ptr[sl]] : sv.ptr[sl]) - eb;
        atomicOr(&sbm[st >> 5], 1u << (st & 31));
      }
      ns += __popc(m);
    }
  } else {
    if (lane == 0) {
      sid[0] = 0;
      const int st = k.e0 - eb;
      sbm[st >> 5] |= 1u << (st & 31);
    }
    ns = 1;
  }
  if (VCS) {
    for (int r = k.r0 + lane; r < k.r1; r += 32) {
      const int st = max(sv.vptr[r], k.e0) - eb;
      atomicOr(&rbm[st >> 5], 1u << (st & 31));
    }
  }
  __syncwarp();

  // The records are sorted by owning warp (tile row mod kWarpsPerCta), stably:
  // pass 0 counts each warp's records, pass 1 places each record at its
  // warp's cursor.  Within a warp's list the order is the entries' order.
  // `emit` takes one candidate entry per lane (the same on both passes).
  auto emit = [&](int pass, bool in, int tt, uint32_t kk, T vv) {
    const int own = tt & kOwnMask;
    const unsigned peers = __match_any_sync(kFullMask, in ? own : -1);
    const int rank = __popc(peers & lt);
    if (pass == 0) {
      if (in && rank == 0) atomicAdd(&cur[own], __popc(peers));
    } else {
      if (in) {
        const int pos = cur[own] + rank;
        key[pos] = kk;
        val[pos] = vv;
      }
      __syncwarp();
      if (in && rank == 0) cur[own] += __popc(peers);
      __syncwarp();
    }
  };
  for (int pass = 0; pass < 2; ++pass) {
    if (!(VCS && skip_by_search)) {
      // every entry of the block, 32 at a time (pass 0 needs only the rows)
      int sbase = -1, rbase = k.r0 - 1;
      for (int q = 0; q < nwords; ++q) {
        const int n = eb + 32 * q + lane;
        bool in = false;
        int tt = 0;
        if (n >= k.e0 && n < k.e1) {
          tt = (int)(sv.idx[n] - t0);
          in = tt >= 0 && tt < rows;
        }
        uint32_t kk = 0;
        T vv = T(0);
        if (pass == 1) {
          const uint32_t sw = sbm[q];
          const uint32_t rw = VCS ? rbm[q] : 0u;
          const int sidx = sbase + __popc(sw & le);
          const int ridx = rbase + __popc(rw & le);
          sbase += __popc(sw);
          rbase += __popc(rw);
          if (in) {
            kk = (uint32_t)tt | ((uint32_t)sid[sidx] << 16);
            vv = VCS ? (T)rv[ridx] : sv.vals[n];
          }
        }
        emit(pass, in, tt, kk, vv);
      }
    } else {
      // sorted runs, partial tile: per run, only the entries inside [t0, t0 + rows)
      int cur_slice = 0;  // index into sid
      for (int r = k.r0; r < k.r1; ++r) {
        int a0, b0;
        if (pass == 0) {
          const int lo = max(sv.vptr[r], k.e0), hi = min(sv.vptr[r + 1], k.e1);
          // first entry with row >= t0, then first with row >= t0 + rows
          a0 = warp_lower_bound(sv.idx, lo, hi, (int)t0);
          b0 = warp_lower_bound(sv.idx, a0, hi, (int)(t0 + rows));
          if (lane == 0) {
            rng[2 * (r - k.r0)] = a0;
            rng[2 * (r - k.r0) + 1] = b0;
          }
        } else {
          a0 = rng[2 * (r - k.r0)];
          b0 = rng[2 * (r - k.r0) + 1];
        }
        while (cur_slice + 1 < ns) {  // the slice holding run r's first entry
          const int nxt = k.type == 0 ? sv.vptr[sv.ptr[k.s0 + sid[cur_slice + 1]]] : k.e1;
          if (nxt <= max(sv.vptr[r], k.e0)) ++cur_slice;
          else break;
        }
        const uint32_t sk = (uint32_t)sid[cur_slice] << 16;
        const T v = (T)rv[r];
        for (int base = a0; base < b0; base += 32) {
          const int n = base + lane;
          const bool in = n < b0;
          const int tt = in ? (int)(sv.idx[n] - t0) : 0;
          emit(pass, in, tt, (uint32_t)tt | sk, v);
        }
      }
    }
    __syncwarp();
    if (pass == 0) {
      // counts -> offsets (exclusive scan over the owning warps) and cursors
      const int c = lane < kWarpsPerCta ? cur[lane] : 0;
      int incl = c;
#pragma unroll
      for (int d = 1; d < kWarpsPerCta; d <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += y;
      }
      __syncwarp();
      if (lane < kWarpsPerCta) {
        off[lane] = incl - c;
        cur[lane] = incl - c;
      }
      if (lane == kWarpsPerCta - 1) off[kWarpsPerCta] = incl;
      __syncwarp();
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(pipe.ready(s));
  return true;
}

template <typename T, int VEC, int Q, int CI, bool VCS>
struct TwoPhaseWarp {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  static constexpr int E = 32 / Q;  // records applied per step

  __device__ __forceinline__ static void apply(T *tile, int w, int tk, T ak, const T (&x)[CI][VEC],
                                               const int (&col0)[CI], const bool (&colok)[CI]) {
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

  // Applies, in record order, this warp's records [lo, hi) of a block: those
  // whose tile row t has t mod kWarpsPerCta == the warp's number (rows
  // interleaved over the warps, so that the popular rows of a skewed matrix
  // spread out), E records per step.
  __device__ __forceinline__ static void run(const uint32_t *key, const T *val, int lo, int hi,
                                             int s0, const T *__restrict__ X, int64_t ldx, T *tile,
                                             int w, const int (&col0)[CI],
                                             const bool (&colok)[CI]) {
    const int lane = threadIdx.x & 31, grp = lane / Q;
    const unsigned lt = lanemask_lt();
    // one step's record: row, value and the X row of its slice
    auto load = [&](int c0, int &tk, T &ak, T (&x)[CI][VEC]) {
      const int qi = c0 + grp;
      tk = -1;
      ak = T(0);
      if (qi < hi) {
        const uint32_t q = key[qi];
        tk = (int)(q & 0xffffu);
        ak = val[qi];
        const int sl = s0 + (int)(q >> 16);
#pragma unroll
        for (int ci = 0; ci < CI; ++ci)
          if (colok[ci])
            Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)sl * ldx + col0[ci])),
                        x[ci]);
      }
    };
    int tn;
    T an, xn[CI][VEC];
    if (lo < hi) load(lo, tn, an, xn);
    for (int c0 = lo; c0 < hi; c0 += E) {
      const int tk = tn;
      const T ak = an;
      T x[CI][VEC];
#pragma unroll
      for (int ci = 0; ci < CI; ++ci)
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[ci][e] = xn[ci][e];
      if (c0 + E < hi) load(c0 + E, tn, an, xn);  // the next step's loads overlap this step
      const unsigned peers = __match_any_sync(kFullMask, tk);
      const bool dup = tk >= 0 && __popc(peers) > Q;
      if (!__any_sync(kFullMask, dup)) {
        if (tk >= 0) apply(tile, w, tk, ak, x, col0, colok);
      } else {
        // equal rows inside the step: one round per earlier duplicate, in record order
        const int rank = __popc(peers & lt) / Q;
        const int rounds = (int)__reduce_max_sync(kFullMask, tk >= 0 ? (unsigned)rank : 0u) + 1;
        for (int rd = 0; rd < rounds; ++rd) {
          if (tk >= 0 && rank == rd) apply(tile, w, tk, ak, x, col0, colok);
          __syncwarp();
        }
      }
    }
  }
};

// Block (tile blockIdx.x, group blockIdx.y).  The producer warp streams the
// group's blocks and turns each into the records of this tile; consumer warp w
// applies the records of the tile rows it owns.
template <typename T, int VEC, int Q, int CI, bool VCS>
__global__ void __launch_bounds__(kTwoPhaseThreads) two_phase_kernel(const TwoPhaseArgs a) {
  using WP = TwoPhaseWarp<T, VEC, Q, CI, VCS>;
  using SM = TwoPhaseSmem<T, VCS>;
  using RL = RecLayout<T>;
  extern __shared__ __align__(128) unsigned char smem[];
  const Pipe<T, VCS> pipe{smem};
  unsigned char *recs = smem + SM::kRecs;
  unsigned char *prep = smem + SM::kPrep;
  T *tile = reinterpret_cast<T *>(smem + SM::kTile);

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t t0 = (int64_t)blockIdx.x * a.tile_rows;
  const int rows = (int)(a.n_t - t0 < a.tile_rows ? a.n_t - t0 : a.tile_rows);
  const int w = a.w;
  const int b_lo = a.bounds[blockIdx.y], b_hi = a.bounds[blockIdx.y + 1];
  for (int q = threadIdx.x; q < rows * w; q += blockDim.x) tile[q] = T(0);
  pipe.init();  // (its barrier also publishes the zeroed tile)
  if (wid == kWarpsPerCta) {
    // ---- issuing warp: every block of the group, in order
    pipe.issue_all(a.st, b_lo, b_hi, 1);
  } else if (wid > kWarpsPerCta) {
    // ---- preparing warp e: blocks e, e + kPreparers, ... as they land
    const int e = wid - kWarpsPerCta - 1;
    const bool search = VCS && a.sorted && rows < a.n_t;
    for (int i = e; i < b_hi - b_lo; i += kPreparers)
      if (*reinterpret_cast<volatile int *>(pipe.fail()) ||
          !two_phase_prepare<T, VCS>(pipe, a.st, i, b_lo + i, recs, prep + e * PrepLayout::kBytes,
                                     t0, rows, search)) {
        pipe.give_up(a.st);
        break;
      }
  } else {
    const int ql = lane & (Q - 1);
    int col0[CI];
    bool colok[CI];
#pragma unroll
    for (int ci = 0; ci < CI; ++ci) {
      col0[ci] = (ci * Q + ql) * VEC;
      colok[ci] = col0[ci] < w;
    }
    const T *__restrict__ X = static_cast<const T *>(a.X);
    int i = 0;
    for (int b = b_lo; b < b_hi; ++b, ++i) {
      const int st = i % kStages;
      if (!mbar_wait_bounded(pipe.ready(st), (i / kStages) & 1, kWaitLimitNs)) {
        pipe.give_up(a.st);
        break;
      }
      const Block k = stage_desc<T, VCS>(pipe.buf(st));
      const unsigned char *rb = recs + st * RL::kBytes;
      const int *off = reinterpret_cast<const int *>(rb + RL::kOff);
      WP::run(reinterpret_cast<const uint32_t *>(rb + RL::kKey),
              reinterpret_cast<const T *>(rb + RL::kVal), off[wid], off[wid + 1], k.s0, X, a.ldx,
              tile, w, col0, colok);
      pipe.release(i);
    }
  }
  __syncthreads();
  if (*pipe.fail()) return;
  // the tile: final Y when C == 1, else this group's partial
  T *__restrict__ out = static_cast<T *>(a.out) + (int64_t)blockIdx.y * a.part_stride;
  for (int q = threadIdx.x; q < rows * w; q += blockDim.x) {
    const int rr = q / w, c = q - rr * w;
    out[(t0 + rr) * a.ldo + c] = tile[q];
  }
}

// Y[t, c] = sum over groups k (in order) of P[k][t, c].
template <typename T>
__global__ void combine_kernel(const T *__restrict__ P, int C, int64_t part_stride, int64_t n_t,
                               int w, T *__restrict__ Y, int64_t ldy) {
  const int64_t total = n_t * w;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / w;
    const int c = (int)(i - t * w);
    // the partials in group order, kBatch loads in flight before their adds
    constexpr int kBatch = 8;
    T sum = P[i];
    for (int k0 = 1; k0 < C; k0 += kBatch) {
      T v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        v[j] = k0 + j < C ? P[(int64_t)(k0 + j) * part_stride + i] : T(0);
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (k0 + j < C) sum = sum + v[j];
    }
    Y[t * ldy + c] = sum;
  }
}

inline int pow2ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

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
  constexpr int smem = pipe_smem_bytes<T, VCS>(0);
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
    a.st = StageArrays{m.ptr, m.idx, m.vals, m.vptr, m.blocks, (int)m.n_blocks, m.err,
                       xp, X.ld, (int)sizeof(T), wb};
    a.X = xp;
    a.ldx = X.ld;
    a.Y = yp;
    a.ldy = Y.ld;
    a.w = wb;
    a.G = std::max(1, std::min(m.g, 32 / sh.Q));
    a.S = 32 / (sh.Q * a.G);
    int per_sm = 0;
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), kPipeThreads, smem, &per_sm));
    const int64_t grid = std::min<int64_t>(m.n_blocks, (int64_t)std::max(1, per_sm) * m.n_sm);
    if (grid > 0) {
      k<<<(unsigned)grid, kPipeThreads, smem, s>>>(a);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

constexpr int kTwoPhaseSmem = 224 * 1024;

template <typename T, bool VCS>
vs_status two_phase_typed(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y, int64_t w,
                          cudaStream_t s) {
  const int C = m.tp_chunks;
  const int64_t n_t = Y.rows;
  constexpr int stage = TwoPhaseSmem<T, VCS>::kTile;
  for (int64_t c0 = 0; c0 < w; c0 += kMaxBlockWidth) {
    const int wb = (int)std::min<int64_t>(kMaxBlockWidth, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    Shape sh = pick_shape<T>(wb, xp, xp, X.ld, X.ld);  // Y is written element by element
    auto k = pick_kernel<T, VCS, TwoPhaseK>(sh);
    if (!k) {
      set_error("no two-phase kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    const int64_t row_bytes = (int64_t)wb * sizeof(T);
    const int tile_rows = (int)std::max<int64_t>(
        1, std::min<int64_t>(n_t, (kTwoPhaseSmem - stage) / row_bytes));
    const int64_t tiles = (n_t + tile_rows - 1) / tile_rows;
    const size_t smem = stage + (size_t)tile_rows * row_bytes;
    int resident = 0;  // (raises the kernel's shared-memory limit once)
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), kTwoPhaseThreads, (int)smem, &resident));
    TwoPhaseArgs a;
    a.st = StageArrays{m.ptr, m.idx, m.vals, m.vptr, m.blocks, (int)m.n_blocks, m.err,
                       xp, X.ld, (int)sizeof(T), wb};
    a.X = xp;
    a.ldx = X.ld;
    a.bounds = m.tp_bounds;
    a.n_t = n_t;
    a.tile_rows = tile_rows;
    a.w = wb;
    a.sorted = m.sorted_segments ? 1 : 0;
    if (C == 1) {
      a.out = yp;
      a.ldo = Y.ld;
      a.part_stride = 0;
    } else {
      VS_TRY(h.tp_partials.reserve((size_t)C * n_t * wb * sizeof(T), s));
      a.out = h.tp_partials.p;
      a.ldo = wb;
      a.part_stride = n_t * wb;
    }
    dim3 grid((unsigned)tiles, (unsigned)C);
    k<<<grid, kTwoPhaseThreads, smem, s>>>(a);
    VS_LAUNCH_CHECK();
    if (C > 1) {
      const int64_t total = n_t * wb;
      const unsigned blocks = (unsigned)std::min<int64_t>((int64_t)m.n_sm * 8, (total + 255) / 256);
      combine_kernel<T><<<std::max(1u, blocks), 256, 0, s>>>(
          static_cast<const T *>(h.tp_partials.p), C, n_t * wb, n_t, wb, yp, Y.ld);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

// ------------------------------------------------------------------ allocation-free variant

// Scratch for callers that cannot allocate device memory at call time (code
// running inside stream capture, under a memory pool they do not own, or in a
// process whose allocator is reserved for something else): the group partials
// of the two-phase scheme live in this fixed array instead of handle scratch.
// Every GPU that loads the library holds it until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};

// The device address of g_static_scratch on the current device, looked up once
// per device (the host-side name is only a stand-in for it).
vs_status static_scratch_address(void **out) {
  int dev = 0;
  VS_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal beyond the static scratch table");
    return VS_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    VS_CUDA(cudaGetSymbolAddress(&p, g_static_scratch));
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return VS_OK;
}

// The two-phase product with its group partials in g_static_scratch.  The
// column block is narrowed until the partials fit; the order of every
// element's sum does not depend on the column block, so the bits match the
// handle-scratch path.
template <typename T, bool VCS>
vs_status two_phase_static_typed(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                 cudaStream_t s) {
  const int C = m.tp_chunks;
  const int64_t n_t = Y.rows;
  constexpr int stage = TwoPhaseSmem<T, VCS>::kTile;
  constexpr int VW = 16 / sizeof(T);
  void *scratch = nullptr;
  int64_t wmax = kMaxBlockWidth;
  if (C > 1) {
    VS_TRY(static_scratch_address(&scratch));
    const int64_t per_col = (int64_t)C * n_t * (int64_t)sizeof(T);
    wmax = std::min<int64_t>(kMaxBlockWidth, (int64_t)kStaticScratchBytes / std::max<int64_t>(per_col, 1));
    if (wmax >= VW) wmax = wmax / VW * VW;
    // C is bounded at build time so that C copies of the output stay within
    // 64 MiB at width 64, i.e. at most 1 MiB per column: this rejection is a
    // guard, not a path a handle built here can reach
    if (wmax < 1) {
      set_error("vs_spmm_noalloc: the partial sums need " + std::to_string(per_col) +
                " bytes per column; the static scratch holds " +
                std::to_string(kStaticScratchBytes) + " bytes");
      return VS_ERR_UNSUPPORTED;
    }
  }
  for (int64_t c0 = 0; c0 < w; c0 += wmax) {
    const int wb = (int)std::min<int64_t>(wmax, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    Shape sh = pick_shape<T>(wb, xp, xp, X.ld, X.ld);
    auto k = pick_kernel<T, VCS, TwoPhaseK>(sh);
    if (!k) {
      set_error("no two-phase kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    const int64_t row_bytes = (int64_t)wb * sizeof(T);
    const int tile_rows = (int)std::max<int64_t>(
        1, std::min<int64_t>(n_t, (kTwoPhaseSmem - stage) / row_bytes));
    const int64_t tiles = (n_t + tile_rows - 1) / tile_rows;
    const size_t smem = stage + (size_t)tile_rows * row_bytes;
    int resident = 0;  // (raises the kernel's shared-memory limit once)
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), kTwoPhaseThreads, (int)smem, &resident));
    TwoPhaseArgs a;
    a.st = StageArrays{m.ptr, m.idx, m.vals, m.vptr, m.blocks, (int)m.n_blocks, m.err,
                       xp, X.ld, (int)sizeof(T), wb};
    a.X = xp;
    a.ldx = X.ld;
    a.bounds = m.tp_bounds;
    a.n_t = n_t;
    a.tile_rows = tile_rows;
    a.w = wb;
    a.sorted = m.sorted_segments ? 1 : 0;
    if (C == 1) {
      a.out = yp;
      a.ldo = Y.ld;
      a.part_stride = 0;
    } else {
      a.out = scratch;
      a.ldo = wb;
      a.part_stride = n_t * wb;
    }
    dim3 grid((unsigned)tiles, (unsigned)C);
    k<<<grid, kTwoPhaseThreads, smem, s>>>(a);
    VS_LAUNCH_CHECK();
    if (C > 1) {
      const int64_t total = n_t * wb;
      const unsigned blocks = (unsigned)std::min<int64_t>((int64_t)m.n_sm * 8, (total + 255) / 256);
      combine_kernel<T><<<std::max(1u, blocks), 256, 0, s>>>(static_cast<const T *>(scratch), C,
                                                             n_t * wb, n_t, wb, yp, Y.ld);
      VS_LAUNCH_CHECK();
    }
  }
  return VS_OK;
}

}  // namespace

vs_status launch_scatter_two_phase_static(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                          cudaStream_t s) {
  if (w <= 0 || Y.rows == 0) return VS_OK;
  if (m.wide) {
    set_error("vs_spmm_noalloc: a misaligned product of a matrix with 64-bit slice pointers needs "
              "the transposed route (vs_attach_transpose)");
    return VS_ERR_UNSUPPORTED;
  }
  if (m.n_major == 0 || m.nnz == 0) return launch_zero_fill(Y, w, m.dsize(), s);
  if (m.tt_rows > 0) {
    // the group partials in the static array, the column pass narrowed to fit
    const int64_t es = (int64_t)m.dsize();
    void *scratch = nullptr;
    int64_t pass = 64 / es;
    if (m.tt_groups > 1) {
      VS_TRY(static_scratch_address(&scratch));
      const int64_t per_col = (int64_t)m.tt_groups * Y.rows * es;
      pass = std::min<int64_t>(pass, (int64_t)kStaticScratchBytes / std::max<int64_t>(per_col, 1));
      if (pass < 1) {
        set_error("vs_spmm_noalloc: the partial sums need " + std::to_string(per_col) +
                  " bytes per column; the static scratch holds " +
                  std::to_string(kStaticScratchBytes) + " bytes");
        return VS_ERR_UNSUPPORTED;
      }
    }
    return launch_tt_two_phase(m, X, Y, w, scratch, pass, s);
  }
  if (m.layout == VS_LAYOUT_VCS) return two_phase_static_typed<float, true>(m, X, Y, w, s);
  if (m.dtype == VS_F64) return two_phase_static_typed<double, false>(m, X, Y, w, s);
  return two_phase_static_typed<float, false>(m, X, Y, w, s);
}

vs_status launch_combine(const void *P, int C, int64_t n_t, int w, void *Y, int64_t ldy,
                         size_t dsize, int n_sm, cudaStream_t s) {
  const int64_t total = n_t * w;
  const unsigned blocks = (unsigned)std::min<int64_t>((int64_t)n_sm * 8, (total + 255) / 256);
  if (dsize == 8)
    combine_kernel<double><<<std::max(1u, blocks), 256, 0, s>>>(
        static_cast<const double *>(P), C, n_t * w, n_t, w, static_cast<double *>(Y), ldy);
  else
    combine_kernel<float><<<std::max(1u, blocks), 256, 0, s>>>(
        static_cast<const float *>(P), C, n_t * w, n_t, w, static_cast<float *>(Y), ldy);
  VS_LAUNCH_CHECK();
  return VS_OK;
}

vs_status launch_zero_fill(DenseView Y, int64_t w, size_t dsize, cudaStream_t s) {
  if (w <= 0 || Y.rows <= 0) return VS_OK;
  const int64_t total = Y.rows * w;
  const unsigned blocks = (unsigned)std::min<int64_t>(152 * 8, (total + 255) / 256);
  if (Y.ld == w && reinterpret_cast<uintptr_t>(Y.p) % 16 == 0 && (total * dsize) % 16 == 0) {
    const int64_t n16 = total * (int64_t)dsize / 16;
    zero_fill_vec_kernel<<<std::max(1u, std::min<unsigned>(blocks, (unsigned)((n16 + 255) / 256))),
                           256, 0, s>>>(static_cast<float4 *>(Y.p), n16);
  } else if (dsize == 8) {
    zero_fill_kernel<double><<<std::max(1u, blocks), 256, 0, s>>>(static_cast<double *>(Y.p),
                                                                    Y.rows, w, Y.ld);
  } else {
    zero_fill_kernel<float><<<std::max(1u, blocks), 256, 0, s>>>(static_cast<float *>(Y.p), Y.rows,
                                                                  w, Y.ld);
  }
  VS_LAUNCH_CHECK();
  return VS_OK;
}

// The rows X[slice0, ...) of a misaligned product's operand: the operand of a
// wide matrix's segment.
static DenseView segment_rows(DenseView X, const Matrix &g) {
  DenseView Xg = X;
  Xg.p = static_cast<char *>(X.p) + (size_t)g.seg_slice0 * (size_t)X.ld * (X.f64 ? 8 : 4);
  Xg.rows = g.n_major;
  return Xg;
}

vs_status launch_scatter_atomic(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                cudaStream_t s) {
  if (w <= 0) return VS_OK;
  VS_TRY(launch_zero_fill(Y, w, m.dsize(), s));
  if (m.n_major == 0 || m.nnz == 0) return VS_OK;
  if (m.wide) {  // every segment adds into the same zero-filled output
    for (const Matrix &g : m.segs) {
      if (g.nnz == 0) continue;
      const DenseView Xg = segment_rows(X, g);
      if (g.layout == VS_LAYOUT_VCS)
        VS_TRY((atomic_typed<float, true>(g, Xg, Y, w, s)));
      else if (g.dtype == VS_F64)
        VS_TRY((atomic_typed<double, false>(g, Xg, Y, w, s)));
      else
        VS_TRY((atomic_typed<float, false>(g, Xg, Y, w, s)));
    }
    return VS_OK;
  }
  if (m.layout == VS_LAYOUT_VCS) return atomic_typed<float, true>(m, X, Y, w, s);
  if (m.dtype == VS_F64) return atomic_typed<double, false>(m, X, Y, w, s);
  return atomic_typed<float, false>(m, X, Y, w, s);
}

vs_status launch_scatter_two_phase(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y,
                                   int64_t w, cudaStream_t s) {
  if (w <= 0 || Y.rows == 0) return VS_OK;
  if (m.n_major == 0 || m.nnz == 0) return launch_zero_fill(Y, w, m.dsize(), s);
  if (m.wide) {
    // segment 0 writes the output; each later segment's deterministic sum is
    // added to it in segment order (slice order, like the groups of one piece)
    const size_t es = m.dsize();
    bool first = true;
    for (const Matrix &g : m.segs) {
      if (g.nnz == 0) continue;
      const DenseView Xg = segment_rows(X, g);
      if (first) {
        VS_TRY(launch_scatter_two_phase(h, g, Xg, Y, w, s));
        first = false;
        continue;
      }
      VS_TRY(h.wide_tmp.reserve(es * (size_t)(Y.rows * w + 16), s));
      DenseView T = Y;
      T.p = h.wide_tmp.p;
      T.ld = w;
      T.scale = nullptr;
      VS_TRY(launch_scatter_two_phase(h, g, Xg, T, w, s));
      const int64_t total = Y.rows * w;
      const unsigned blocks = (unsigned)std::min<int64_t>((int64_t)m.n_sm * 8, (total + 255) / 256);
      if (es == 8)
        add_into_kernel<double><<<std::max(1u, blocks), 256, 0, s>>>(
            static_cast<const double *>(T.p), Y.rows, w, static_cast<double *>(Y.p), Y.ld);
      else
        add_into_kernel<float><<<std::max(1u, blocks), 256, 0, s>>>(
            static_cast<const float *>(T.p), Y.rows, w, static_cast<float *>(Y.p), Y.ld);
      VS_LAUNCH_CHECK();
    }
    if (first) return launch_zero_fill(Y, w, es, s);
    return VS_OK;
  }
  if (m.tt_rows > 0) {
    const size_t es = m.dsize();
    const int64_t pass = 64 / (int64_t)es;
    void *part = nullptr;
    if (m.tt_groups > 1) {
      VS_TRY(h.tp_partials.reserve((size_t)m.tt_groups * Y.rows * pass * es, s));
      part = h.tp_partials.p;
    }
    return launch_tt_two_phase(m, X, Y, w, part, pass, s);
  }
  if (tb_applies(m, Y.rows)) return launch_tb_two_phase(h, m, X, Y, w, s);
  if (m.layout == VS_LAYOUT_VCS) return two_phase_typed<float, true>(h, m, X, Y, w, s);
  if (m.dtype == VS_F64) return two_phase_typed<double, false>(h, m, X, Y, w, s);
  return two_phase_typed<float, false>(h, m, X, Y, w, s);
}

}  // namespace vs
