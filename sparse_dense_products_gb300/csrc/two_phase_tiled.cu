// two_phase_tiled.cu -- the deterministic misaligned product over tiles of
// output rows.  Covers VCSC@B, B@VCSR, CSC@B and B@CSR for matrices whose
// minor indices ascend inside every run (VCS) or slice (CSR); a CSR whose
// slices are not sorted takes it when its output fits one tile.
//
// "Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": a misaligned product adds a * X[s, :] into row t of Y for every
// entry (t, a) of slice s, so several slices write one row; atomic adds make
// the last bits depend on timing.  Here the order of every element's sum is
// fixed instead:
//
//  * The entries are cut by position into G groups of equal counts (G fixed
//    by the matrix).  CTA (tile k, group c) sums group c's entries that land
//    in tile k into a shared-memory copy of the tile's rows of Y; the G
//    partials of every element are then added in group order.
//  * The minor indices ascend inside a run, so the entries of run r inside
//    tile k form one range.  The matrix keeps where each range starts
//    (tt_tab), and a CTA reads only its own entries.
//  * Warp w of the CTA owns a contiguous range of the tile's rows (tt_own:
//    balanced by the group's entry counts).  Per chunk of kTtChunkRuns runs,
//    the runs' pieces number the chunk's entries in entry order; window by
//    window, each warp lists an equal share of them, and the window is
//    sorted stably by owning warp (counted while listed, then placed); each
//    warp then adds its records in entry order, E per step, rows met twice
//    in one step one after the other.
//
// Every element's sum therefore runs over its group's entries in entry order,
// then over the groups in order: it depends on the matrix alone, not on the
// tiling, the owners, the width or the column pass.
#include <algorithm>
#include <climits>
#include <vector>

#include "device_utils.cuh"
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kTtThreads = kTtWarps * 32;
constexpr int kTtChunkRuns = kTtWarps * 32;  // runs (slices) per chunk: 32 per warp
constexpr int kTtPassBytes = 64;             // widest column pass
constexpr int kTtUnroll = 4;                 // 32-record groups a warp lists before their loads land
constexpr int kTtSub = kTtOwners / kTtWarps; // row owners (of the build) per warp
static_assert(kTtOwners % kTtWarps == 0, "whole owners per warp");

__device__ __forceinline__ float tt_fma(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double tt_fma(double a, double b, double c) { return fma(a, b, c); }

// Shared memory of a CTA; the tile of Y rows comes last.
template <typename T, bool VCS>
struct TtSmem {
  static constexpr int kCap = ((VCS ? 4 : (sizeof(T) == 4 ? 2 : 1)) * 2048) / kTtCtasPerSm;  // records per window
  static constexpr int kList = 0;                                           // u32 [kCap] (listing order)
  static constexpr int kListVal = kList + kCap * 4;                         // CSR: T [kCap]
  static constexpr int kKey = kListVal + (VCS ? 0 : kCap * (int)sizeof(T)); // u32 [kCap] (by owner)
  static constexpr int kVal = kKey + kCap * 4;                              // CSR: T [kCap]
  static constexpr int kSlice = kVal + (VCS ? 0 : kCap * (int)sizeof(T));   // i32 [chunk runs]
  static constexpr int kRunVal = kSlice + kTtChunkRuns * 4;                 // VCS: f32 [chunk runs]
  static constexpr int kCPos = kRunVal + (VCS ? kTtChunkRuns * 4 : 0);      // i32 [chunk runs]
  static constexpr int kCFirst = kCPos + kTtChunkRuns * 4;                  // i32 [chunk runs]
  static constexpr int kCRun = kCFirst + kTtChunkRuns * 4;                  // i32 [chunk runs]
  static constexpr int kCount = kCRun + kTtChunkRuns * 4;                   // i32 [warp][owner warp]
  static constexpr int kCursor = kCount + kTtWarps * kTtWarps * 4;          // i32 [warp][owner warp]
  static constexpr int kTotal = kCursor + kTtWarps * kTtWarps * 4;          // i32 [2][warp]
  static constexpr int kOwner = kTotal + 2 * kTtWarps * 4;                  // u8 [tile rows]
  static constexpr int kTile = (kOwner + kTtRows + 15) / 16 * 16;
  static_assert(kListVal % 16 == 0 && kKey % 16 == 0 && kTile % 16 == 0, "shared-memory alignment");
  static_assert(kTile + kTtRows * kTtPassBytes <= (228 * 1024) / kTtCtasPerSm - 1024,
                "kTtCtasPerSm CTAs fit one multiprocessor's shared memory");
};

struct TtArgs {
  const int32_t *ptr;        // CSR: slice entry starts
  const int32_t *vptr;       // VCS: run entry starts
  const int32_t *idx;        // minor indices
  const void *vals;          // CSR: entry values (T); VCS: run values (float)
  const int32_t *tab;        // [(tiles-1) * pieces]
  const int32_t *run_slice;  // VCS: [R]
  const int32_t *group;      // [3*groups+1]
  const int32_t *own;        // [tiles * groups * (kTtOwners+1)]
  int64_t pieces;            // runs (VCS) or slices (CSR)
  const void *X;             // operand rows, one per slice
  int64_t ldx;
  void *out;                 // Y (one group) or the group partials
  int64_t ldo;
  int64_t part_stride;       // elements between group partials
  int64_t n_t;               // rows of Y
  int *err;                  // set (2) if an entry falls outside the CTA's tile: never, for consistent arrays
  int tile_rows, tiles, groups, w;
};

// Block (tile blockIdx.x, group blockIdx.y), kTtWarps warps; warp w owns the
// rows of the build's owners w * kTtSub .. (w + 1) * kTtSub - 1.  Per chunk of
// runs: the runs' pieces, their records numbered in entry order over the
// chunk, and the non-empty runs listed (compacted) with their first record.
// The records then go through windows of kCap: each warp lists an equal share
// of the window (32 records at a time, located among 32 listed runs by
// shuffles) into the window's listing, counting them per owner; then it
// places its share stably by owner; then each warp adds its records in entry
// order, E per step, rows met twice in one step one after the other.
template <typename T, int VEC, int Q, bool VCS>
__global__ void __launch_bounds__(kTtThreads, kTtCtasPerSm) tt_two_phase_kernel(const TtArgs a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  using SL = TtSmem<T, VCS>;
  constexpr int E = 32 / Q;  // records per step
  constexpr int U = kTtUnroll;
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *list = reinterpret_cast<uint32_t *>(smem + SL::kList);
  T *lval = reinterpret_cast<T *>(smem + SL::kListVal);
  uint32_t *key = reinterpret_cast<uint32_t *>(smem + SL::kKey);
  T *rval = reinterpret_cast<T *>(smem + SL::kVal);
  int32_t *rsl = reinterpret_cast<int32_t *>(smem + SL::kSlice);
  float *rrv = reinterpret_cast<float *>(smem + SL::kRunVal);
  int32_t *cpos = reinterpret_cast<int32_t *>(smem + SL::kCPos);
  int32_t *cfirst = reinterpret_cast<int32_t *>(smem + SL::kCFirst);
  int32_t *crun = reinterpret_cast<int32_t *>(smem + SL::kCRun);
  int *cnt = reinterpret_cast<int *>(smem + SL::kCount);
  int *cur = reinterpret_cast<int *>(smem + SL::kCursor);
  int *wtot = reinterpret_cast<int *>(smem + SL::kTotal);
  uint8_t *owner = smem + SL::kOwner;
  T *tile = reinterpret_cast<T *>(smem + SL::kTile);

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const unsigned lt = lanemask_lt();
  const int tk = blockIdx.x, c = blockIdx.y;
  const int t0 = tk * a.tile_rows;
  const int64_t rem = a.n_t - t0;
  const int rows = rem < a.tile_rows ? (int)rem : a.tile_rows;
  const int w = a.w;
  for (int q = threadIdx.x; q < rows * w; q += kTtThreads) tile[q] = T(0);
  {
    const int32_t *own = a.own + ((int64_t)tk * a.groups + c) * (kTtOwners + 1);
    const int u0 = own[wid * kTtSub] - t0, u1 = own[(wid + 1) * kTtSub] - t0;
    for (int q = u0 + lane; q < u1; q += 32) owner[q] = (uint8_t)wid;
  }
  __syncthreads();

  const int E0 = a.group[c], E1 = a.group[c + 1];
  const int ra = a.group[a.groups + 1 + c], rb = a.group[2 * a.groups + 1 + c];
  const bool first = tk == 0, last = tk == a.tiles - 1;
  const T *__restrict__ X = static_cast<const T *>(a.X);
  const int32_t *__restrict__ idx = a.idx;
  const T *__restrict__ evals = static_cast<const T *>(a.vals);
  const int grp = lane / Q;
  const int col0 = (lane % Q) * VEC;
  const bool colok = col0 < w;
  int *mycnt = cnt + wid * kTtWarps;
  int *mycur = cur + wid * kTtWarps;

  for (int cb = ra; cb < rb; cb += kTtChunkRuns) {
    // ---- this warp's 32 runs of the chunk: the piece of each inside the
    // tile and the group
    {
      const int q = wid * 32 + lane;  // run number inside the chunk
      const int r = cb + q;
      int p0 = 0, n = 0;
      if (r < rb) {
        const int st = VCS ? a.vptr[r] : a.ptr[r];
        const int en = VCS ? a.vptr[r + 1] : a.ptr[r + 1];
        int lo = first ? st : a.tab[(int64_t)(tk - 1) * a.pieces + r];
        int hi = last ? en : a.tab[(int64_t)tk * a.pieces + r];
        lo = max(lo, E0);
        hi = min(hi, E1);
        p0 = lo;
        n = max(hi - lo, 0);
        rsl[q] = VCS ? a.run_slice[r] : r;
        if (VCS) rrv[q] = static_cast<const float *>(a.vals)[r];
      }
      const int incl = warp_inclusive_scan(n);
      const unsigned ne = __ballot_sync(kFullMask, n > 0);
      const int L = __shfl_sync(kFullMask, incl, 31);
      if (lane == 0) {
        wtot[wid] = L;
        wtot[kTtWarps + wid] = __popc(ne);
      }
      __syncthreads();
      int O = 0, OM = 0;  // records and non-empty runs of the earlier warps
#pragma unroll
      for (int k = 0; k < kTtWarps; ++k) {
        O += k < wid ? wtot[k] : 0;
        OM += k < wid ? wtot[kTtWarps + k] : 0;
      }
      if (n > 0) {
        const int m = OM + __popc(ne & lt);
        cpos[m] = O + incl - n;
        cfirst[m] = p0;
        crun[m] = q;
      }
    }
    int Ltot = 0, M = 0;  // the chunk's records and non-empty runs
#pragma unroll
    for (int k = 0; k < kTtWarps; ++k) {
      Ltot += wtot[k];
      M += wtot[kTtWarps + k];
    }
    __syncthreads();

    for (int W0 = 0; W0 < Ltot; W0 += SL::kCap) {
      const int W1 = min(W0 + SL::kCap, Ltot);
      const int span = (W1 - W0 + kTtWarps - 1) / kTtWarps;
      const int b0 = min(W0 + wid * span, W1), b1 = min(b0 + span, W1);  // this warp's share
      if (lane < kTtWarps) mycnt[lane] = 0;
      __syncwarp();
      // ---- list the share, 32 * U records at a time: record p sits in one
      // of the 32 listed runs from j (they are non-empty), found by
      // shuffles; the U groups' loads are issued before any is used
      {
        int j = 0;  // the last listed run starting at or before record b0
        if (b0 < b1) {
          int hi = M - 1;
          while (j < hi) {
            const int mid = (j + hi + 1) / 2;
            if (cpos[mid] <= b0)
              j = mid;
            else
              hi = mid - 1;
          }
        }
        for (int s0 = b0; s0 < b1; s0 += 32 * U) {
          int e[U];
          uint32_t rq[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int p = s0 + 32 * u + lane;
            const bool lst = j + lane < M;
            const int cp = lst ? cpos[j + lane] : INT_MAX;
            int l = 0;
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) {
              const int cl = __shfl_sync(kFullMask, cp, l + sh);
              if (cl <= p) l += sh;
            }
            const int cf = lst ? cfirst[j + lane] : 0;
            const int cr = lst ? crun[j + lane] : 0;
            e[u] = __shfl_sync(kFullMask, cf, l) + p - __shfl_sync(kFullMask, cp, l);
            rq[u] = (uint32_t)__shfl_sync(kFullMask, cr, l);
            j += __shfl_sync(kFullMask, l, 31);
          }
          int row[U];
          T val[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const bool in = s0 + 32 * u + lane < b1;
            row[u] = in ? idx[e[u]] - t0 : -1;
            val[u] = (!VCS && in) ? evals[e[u]] : T(0);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int p = s0 + 32 * u + lane;
            const bool in = p < b1;
            const bool ok = in && (unsigned)row[u] < (unsigned)rows;
            if (in && !ok) atomicOr(a.err, 2);
            if (in) {
              list[p - W0] = ok ? ((uint32_t)row[u] | (rq[u] << 16)) : 0xffffffffu;
              if (!VCS) lval[p - W0] = val[u];
            }
            const int o = ok ? (int)owner[row[u]] : -1;
            const unsigned peers = __match_any_sync(kFullMask, o);
            if (ok && (peers & lt) == 0) mycnt[o] += __popc(peers);
            __syncwarp();
          }
        }
      }
      __syncthreads();
      // ---- where each (warp, owner) goes: owners in order, inside an owner
      // the listing warps in order (= record order); lane o takes owner o
      int tot = 0, before = 0;
      if (lane < kTtWarps) {
#pragma unroll
        for (int k = 0; k < kTtWarps; ++k) {
          const int v = cnt[k * kTtWarps + lane];
          tot += v;
          before += k < wid ? v : 0;
        }
      }
      const int tincl = warp_inclusive_scan(tot);
      if (lane < kTtWarps) mycur[lane] = tincl - tot + before;
      const int ob = __shfl_sync(kFullMask, tincl - tot, wid);  // this warp's own records
      const int oe = ob + __shfl_sync(kFullMask, tot, wid);
      __syncwarp();
      // ---- place the share from the listing, stably per owner
      for (int p = b0 + lane - W0; p - lane < b1 - W0; p += 32) {
        const bool in = p < b1 - W0;
        const uint32_t kk = in ? list[p] : 0xffffffffu;
        const int o = kk != 0xffffffffu ? (int)owner[kk & 0xffffu] : -1;
        const unsigned peers = __match_any_sync(kFullMask, o);
        if (o >= 0) {
          const int pp = mycur[o] + __popc(peers & lt);
          key[pp] = kk;
          if (!VCS) rval[pp] = lval[p];
        }
        __syncwarp();
        if (o >= 0 && (peers & lt) == 0) mycur[o] += __popc(peers);
        __syncwarp();
      }
      __syncthreads();
      // ---- apply this warp's records [ob, oe) in order, E per step
      auto load = [&](int c0, int &tr, T &av, T (&x)[VEC]) {
        const int qi = c0 + grp;
        tr = -1;
        av = T(0);
#pragma unroll
        for (int v = 0; v < VEC; ++v) x[v] = T(0);
        if (qi < oe) {
          const uint32_t kq = key[qi];
          tr = (int)(kq & 0xffffu);
          const int rq = (int)(kq >> 16);
          av = VCS ? (T)rrv[rq] : rval[qi];
          if (colok)
            Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)rsl[rq] * a.ldx + col0)),
                        x);
        }
      };
      auto add = [&](int tr, T av, const T (&x)[VEC]) {
        V *p = reinterpret_cast<V *>(tile + tr * w + col0);
        T y[VEC];
        Ops::unpack(*p, y);
#pragma unroll
        for (int v = 0; v < VEC; ++v) y[v] = tt_fma(av, x[v], y[v]);
        *p = Ops::pack(y);
      };
      int tn;
      T an, xn[VEC];
      load(ob, tn, an, xn);
      for (int c0 = ob; c0 < oe; c0 += E) {
        const int tr = tn;
        const T av = an;
        T x[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) x[v] = xn[v];
        if (c0 + E < oe) load(c0 + E, tn, an, xn);  // the next step's loads overlap this step
        const unsigned peers = __match_any_sync(kFullMask, tr);
        const bool dup = tr >= 0 && __popc(peers) > Q;
        if (!__any_sync(kFullMask, dup)) {
          if (tr >= 0 && colok) add(tr, av, x);
        } else {
          // equal rows inside the step: one round per earlier one, in record order
          const int rank = __popc(peers & lt) / Q;
          const int rounds = (int)__reduce_max_sync(kFullMask, tr >= 0 ? (unsigned)rank : 0u) + 1;
          for (int rd = 0; rd < rounds; ++rd) {
            if (tr >= 0 && colok && rank == rd) add(tr, av, x);
            __syncwarp();
          }
        }
      }
      __syncthreads();
    }
    __syncthreads();  // the chunk's run arrays and totals are rewritten next
  }

  // the tile: final Y with one group, else this group's partial
  T *__restrict__ out = static_cast<T *>(a.out) + (int64_t)c * a.part_stride;
  for (int q = threadIdx.x; q < rows * w; q += kTtThreads) {
    const int rr = q / w, cc = q - rr * w;
    out[(int64_t)(t0 + rr) * a.ldo + cc] = tile[q];
  }
}

using TtKernel = void (*)(const TtArgs);

template <typename T, bool VCS>
TtKernel pick_tt(bool vec, int Q) {
  constexpr int VW = 16 / sizeof(T);
  if (vec) {
    switch (Q) {
      case 1: return tt_two_phase_kernel<T, VW, 1, VCS>;
      case 2: return tt_two_phase_kernel<T, VW, 2, VCS>;
      case 4: return tt_two_phase_kernel<T, VW, 4, VCS>;
    }
  } else {
    switch (Q) {
      case 1: return tt_two_phase_kernel<T, 1, 1, VCS>;
      case 2: return tt_two_phase_kernel<T, 1, 2, VCS>;
      case 4: return tt_two_phase_kernel<T, 1, 4, VCS>;
      case 8: return tt_two_phase_kernel<T, 1, 8, VCS>;
      case 16:
        if constexpr (sizeof(T) == 4) return tt_two_phase_kernel<T, 1, 16, VCS>;
        break;
    }
  }
  return nullptr;
}

int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

template <typename T, bool VCS>
vs_status tt_typed(const Matrix &m, DenseView X, DenseView Y, int64_t w, void *part,
                   int64_t max_pass, cudaStream_t s) {
  constexpr int VW = 16 / sizeof(T);
  const int64_t pass = std::min<int64_t>(kTtPassBytes / (int64_t)sizeof(T), max_pass);
  const int G = m.tt_groups;
  const int64_t n_t = Y.rows;
  if (pass < 1 || (G > 1 && !part)) {
    set_error("tiled two-phase: no room for the group partials");
    return VS_ERR_UNSUPPORTED;
  }
  for (int64_t c0 = 0; c0 < w; c0 += pass) {
    const int wb = (int)std::min<int64_t>(pass, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    const bool vec = wb % VW == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0 && X.ld % VW == 0;
    const TtKernel k = pick_tt<T, VCS>(vec, pow2_at_least(vec ? wb / VW : wb));
    if (!k) {
      set_error("no tiled two-phase kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    const int smem = TtSmem<T, VCS>::kTile + m.tt_rows * wb * (int)sizeof(T);
    int resident = 0;  // (raises the kernel's shared-memory limit once)
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), kTtThreads, smem, &resident));
    TtArgs a;
    a.ptr = m.ptr;
    a.vptr = m.vptr;
    a.idx = m.idx;
    a.vals = m.vals;
    a.tab = m.tt_tab;
    a.run_slice = m.tt_run_slice;
    a.group = m.tt_group;
    a.own = m.tt_own;
    a.pieces = VCS ? m.R : m.n_major;
    a.X = xp;
    a.ldx = X.ld;
    a.n_t = n_t;
    a.err = m.err;
    a.tile_rows = m.tt_rows;
    a.tiles = m.tt_tiles;
    a.groups = G;
    a.w = wb;
    if (G == 1) {
      a.out = yp;
      a.ldo = Y.ld;
      a.part_stride = 0;
    } else {
      a.out = part;
      a.ldo = wb;
      a.part_stride = n_t * wb;
    }
    k<<<dim3((unsigned)m.tt_tiles, (unsigned)G), kTtThreads, smem, s>>>(a);
    VS_LAUNCH_CHECK();
    if (G > 1) VS_TRY(launch_combine(part, G, n_t, wb, yp, Y.ld, sizeof(T), m.n_sm, s));
  }
  return VS_OK;
}

// ------------------------------------------------------------------ the arrays kept with the matrix

// tab[(k-1) * pieces + r] = the first entry of run r whose minor index is at
// least k * tile_rows (the run's end if none), k = 1 .. tiles-1.
__global__ void tt_table_kernel(const int32_t *__restrict__ starts, const int32_t *__restrict__ idx,
                                int64_t pieces, int tiles, int tile_rows, int32_t *__restrict__ tab) {
  const int64_t total = (int64_t)(tiles - 1) * pieces;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = i / pieces + 1;
    const int64_t r = i - (k - 1) * pieces;
    int lo = starts[r], hi = starts[r + 1];
    const int64_t bound = k * tile_rows;
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (idx[mid] < bound)
        lo = mid + 1;
      else
        hi = mid;
    }
    tab[i] = lo;
  }
}

// hist[c * n_minor + t] = entries of group c with minor index t.
__global__ void tt_hist_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ group,
                               int groups, int64_t n_minor, int32_t *__restrict__ hist) {
  const int e_lo = group[0], e_hi = group[groups];
  for (int64_t n = e_lo + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; n < e_hi;
       n += (int64_t)gridDim.x * blockDim.x) {
    int lo = 0, hi = groups - 1;  // the last group starting at or before n
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (group[mid] <= n)
        lo = mid;
      else
        hi = mid - 1;
    }
    atomicAdd(&hist[(int64_t)lo * n_minor + idx[n]], 1);
  }
}

// One warp per (tile, group): own[.. + b] = the first row of owner b, so that
// owner b takes the rows whose count of earlier entries (of this group, in
// this tile) lies in [b * total / B, (b+1) * total / B), B = kTtOwners.
__global__ void tt_split_kernel(const int32_t *__restrict__ hist, int64_t n_minor, int tiles,
                                int groups, int tile_rows, int32_t *__restrict__ own) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t task = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
       task < (int64_t)tiles * groups; task += warps) {
    const int t = (int)(task / groups), c = (int)(task - (int64_t)t * groups);
    const int t0 = t * tile_rows;
    const int64_t rem = n_minor - t0;
    const int rows = rem < tile_rows ? (int)rem : tile_rows;
    const int32_t *h = hist + (int64_t)c * n_minor + t0;
    int total = 0;
    for (int q = lane; q < rows; q += 32) total += h[q];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) total += __shfl_xor_sync(kFullMask, total, d);
    int below[kTtOwners / 32] = {};  // lane l, entry i: rows before owner l + 32 i's first
    int carry = 0;
    for (int q0 = 0; q0 < rows; q0 += 32) {
      const bool ok = q0 + lane < rows;
      const int v = ok ? h[q0 + lane] : 0;
      const int excl = carry + warp_inclusive_scan(v) - v;
#pragma unroll
      for (int i = 0; i < kTtOwners / 32; ++i)
#pragma unroll 1
        for (int l = 0; l < 32; ++l) {
          const int b = 32 * i + l;
          const unsigned m = __ballot_sync(
              kFullMask, ok && (int64_t)excl * kTtOwners < (int64_t)b * total);
          if (l == lane) below[i] += __popc(m);
        }
      carry = __shfl_sync(kFullMask, excl + v, 31);
    }
    int32_t *o = own + task * (kTtOwners + 1);
#pragma unroll
    for (int i = 0; i < kTtOwners / 32; ++i) o[lane + 32 * i] = t0 + (lane + 32 * i == 0 ? 0 : below[i]);
    if (lane == 0) o[kTtOwners] = t0 + rows;
  }
}

}  // namespace

vs_status launch_tt_two_phase(const Matrix &m, DenseView X, DenseView Y, int64_t w, void *part,
                              int64_t max_pass, cudaStream_t s) {
  if (m.layout == VS_LAYOUT_VCS) return tt_typed<float, true>(m, X, Y, w, part, max_pass, s);
  if (m.dtype == VS_F64) return tt_typed<double, false>(m, X, Y, w, part, max_pass, s);
  return tt_typed<float, false>(m, X, Y, w, part, max_pass, s);
}

vs_status build_tiled_two_phase(Matrix &m, const std::vector<int32_t> &ptr,
                                const std::vector<int32_t> &vptr, cudaStream_t s) {
  m.tt_rows = m.tt_tiles = m.tt_groups = 0;
  // a wide matrix's segments view its arrays past leading entries no slice
  // names: they keep the block-stream scheme
  if (m.wide || m.borrowed_idx || m.nnz == 0 || m.n_minor == 0 || m.n_major == 0 ||
      m.tt_req_rows < 0)
    return VS_OK;
  const bool vcs = m.layout == VS_LAYOUT_VCS;
  const int64_t pieces = vcs ? m.R : m.n_major;
  const std::vector<int32_t> &st = vcs ? vptr : ptr;  // [pieces + 1] entry starts
  if ((int64_t)st.size() != pieces + 1) {
    set_error("tiled two-phase: pointer array size");
    return VS_ERR_INVALID;
  }
  const int TR = m.tt_req_rows > 0 ? std::min(m.tt_req_rows, kTtRows) : kTtRows;
  const int64_t T = (m.n_minor + TR - 1) / TR;
  if (T > 1 && !m.sorted_segments) return VS_OK;  // a tile's entries of a run are no range
  const int64_t tab_n = (T - 1) * pieces;
  if (m.tt_req_rows == 0 && (int64_t)sizeof(int32_t) * tab_n > m.layout_bytes() / 2) return VS_OK;
  if (T > (int64_t(1) << 30)) return VS_OK;

  // groups: from the default tiling, so that a requested tile size changes no bits
  const int64_t t_def = (m.n_minor + kTtRows - 1) / kTtRows;
  const int64_t G = std::max<int64_t>(
      1, std::min<int64_t>({256, kTtTargetCtas / t_def, (m.nnz + 4095) / 4096}));
  std::vector<int32_t> grp(3 * G + 1, 0);
  const int64_t e_lo = st[0], e_hi = st[pieces];
  for (int64_t c = 0; c <= G; ++c) grp[c] = (int32_t)(e_lo + (e_hi - e_lo) * c / G);
  auto piece_of = [&](int64_t e) {  // the (non-empty) piece holding entry e
    return (int32_t)(std::upper_bound(st.begin(), st.end(), (int32_t)e) - st.begin() - 1);
  };
  for (int64_t c = 0; c < G; ++c) {
    if (grp[c] < grp[c + 1]) {
      grp[G + 1 + c] = piece_of(grp[c]);
      grp[2 * G + 1 + c] = piece_of(grp[c + 1] - 1) + 1;
    }
  }
  VS_TRY(dev_alloc((void **)&m.tt_group, sizeof(int32_t) * grp.size()));
  VS_CUDA(cudaMemcpyAsync(m.tt_group, grp.data(), sizeof(int32_t) * grp.size(),
                          cudaMemcpyHostToDevice, s));
  std::vector<int32_t> rs;
  if (vcs) {
    rs.resize(m.R);
    for (int64_t sl = 0; sl < m.n_major; ++sl)
      for (int32_t r = ptr[sl]; r < ptr[sl + 1]; ++r) rs[r] = (int32_t)sl;
    VS_TRY(dev_alloc((void **)&m.tt_run_slice, sizeof(int32_t) * rs.size()));
    VS_CUDA(cudaMemcpyAsync(m.tt_run_slice, rs.data(), sizeof(int32_t) * rs.size(),
                            cudaMemcpyHostToDevice, s));
  }
  const int32_t *d_st = vcs ? m.vptr : m.ptr;
  if (T > 1) {
    VS_TRY(dev_alloc((void **)&m.tt_tab, sizeof(int32_t) * tab_n));
    const unsigned blocks = (unsigned)std::min<int64_t>(4096, (tab_n + 255) / 256);
    tt_table_kernel<<<blocks, 256, 0, s>>>(d_st, m.idx, pieces, (int)T, TR, m.tt_tab);
    VS_LAUNCH_CHECK();
  }
  // owners: the group's entry count of every minor index, then the splits
  int32_t *hist = nullptr;
  const int64_t hist_n = G * m.n_minor;
  VS_TRY(dev_alloc((void **)&hist, sizeof(int32_t) * hist_n));
  vs_status st_ok = VS_OK;
  do {
    cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(int32_t) * hist_n, s);
    if (e != cudaSuccess) {
      st_ok = cuda_status(e, "cudaMemsetAsync");
      break;
    }
    const unsigned hb = (unsigned)std::min<int64_t>(4096, (e_hi - e_lo + 255) / 256);
    tt_hist_kernel<<<std::max(1u, hb), 256, 0, s>>>(m.idx, m.tt_group, (int)G, m.n_minor, hist);
    if ((e = cudaGetLastError()) != cudaSuccess) {
      st_ok = cuda_status(e, "tt_hist_kernel");
      break;
    }
    st_ok = dev_alloc((void **)&m.tt_own, sizeof(int32_t) * T * G * (kTtOwners + 1));
    if (st_ok != VS_OK) break;
    const unsigned sb = (unsigned)std::min<int64_t>(4096, (T * G + 7) / 8);
    tt_split_kernel<<<std::max(1u, sb), 256, 0, s>>>(hist, m.n_minor, (int)T, (int)G, TR, m.tt_own);
    if ((e = cudaGetLastError()) != cudaSuccess) {
      st_ok = cuda_status(e, "tt_split_kernel");
      break;
    }
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) st_ok = cuda_status(e, "tiled two-phase build");
  } while (false);
  cudaStreamSynchronize(s);
  cudaFree(hist);
  if (st_ok != VS_OK) return st_ok;
  m.tt_rows = TR;
  m.tt_tiles = (int)T;
  m.tt_groups = (int)G;
  return VS_OK;
}

}  // namespace vs
