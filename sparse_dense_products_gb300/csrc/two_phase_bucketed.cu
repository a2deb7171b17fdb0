// two_phase_bucketed.cu -- the deterministic misaligned product over tiles of
// output rows when no per-(run, tile) offsets are kept with the matrix: its
// output spans so many tiles that the offsets would outweigh the layout (the
// 1M-row and 500,000-row outputs of the large and skewed workloads), or its
// minor indices are not sorted inside slices.
//
// "Add CUDA transfer and matmul kernels for the normalized views", "The
// kernels": the misaligned directions add a * X[s, :] into row t of Y for every
// entry (t, a) of slice s.  Every call here first sorts the entries' records
// stably into buckets (tile of output rows, group of blocks): records (row in
// the tile, slice, value) in handle scratch, each bucket in entry order.  A
// bucket is then what the tiled kernel's pieces are: CTA (tile k, group c)
// reads its bucket's records, sorts each window of them stably by owning warp
// (row ranges balanced by the bucket's row counts) and every warp adds its
// records in entry order, 8 per step, rows met twice in one step one after the
// other; the groups' partials are added in group order.  Every element's sum
// therefore depends on the matrix alone (the groups are the block-stream
// scheme's C groups of consecutive blocks), never on the width.
//
// The sort is a counting sort over superblocks of kTbBlocksPerCta blocks:
// count per (superblock, bucket), an exclusive scan per bucket over the
// superblocks, one over the buckets, then a stable placement (warps in block
// order, lanes in entry order).
#include <algorithm>
#include <climits>
#include <vector>

#include "stage.cuh"

namespace vs {
namespace {

constexpr int kTbWarps = 8;          // bucketing CTAs
constexpr int kTbBlocksPerCta = 64;  // matrix blocks per bucketing CTA, 8 per warp
constexpr int kTbAWarps = 16;        // applying CTAs
constexpr int kTbAThreads = kTbAWarps * 32;
constexpr int kTbPassBytes = 64;
static_assert(kTbBlocksPerCta % kTbWarps == 0, "whole blocks per warp");

__device__ __forceinline__ float tb_fma(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double tb_fma(double a, double b, double c) { return fma(a, b, c); }

struct TbSort {
  const int32_t *ptr;     // CSR: slice entry starts; VCS: slice run starts
  const int32_t *vptr;    // VCS: run entry starts
  const int32_t *idx;
  const void *vals;       // CSR: T per entry; VCS: float per run
  const int4 *blocks;     // [n_blocks][3]
  const int32_t *bounds;  // [C+1] block bounds of the groups
  int n_blocks, C, T, tile_rows;
  int *counts;            // [superblocks][T*C]
  int *tot;               // [T*C]
  int *base;              // [T*C + 1]
  uint16_t *rec_row;      // [nnz] row inside its tile
  int32_t *rec_slice;     // [nnz]
  void *rec_val;          // [nnz] of T
};

// The group of block b: the last c with bounds[c] <= b.
__device__ __forceinline__ int group_of(const int32_t *bounds, int C, int b) {
  int lo = 0, hi = C - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (bounds[mid] <= b)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// A warp's shared-memory view of one block's pieces (runs for VCS, slices for
// CSR): the first entry of each (clipped to the block), then the block's end;
// the slice of each; the run value of each (VCS).
constexpr int kTbPieces = (kCapRuns > kCapSlices ? kCapRuns : kCapSlices) + 1;
struct PieceTab {
  int *start;  // [kTbPieces]
  int *slice;  // [kTbPieces]
  float *val;  // [kTbPieces]
  static constexpr int kBytes = kTbPieces * 12;
  __device__ __forceinline__ static PieceTab at(unsigned char *base) {
    return PieceTab{reinterpret_cast<int *>(base), reinterpret_cast<int *>(base + kTbPieces * 4),
                    reinterpret_cast<float *>(base + kTbPieces * 8)};
  }
};

// Warp-wide: calls f(e, slice, value, valid) for the entries of block k in
// entry order, 32 at a time (every lane calls f the same number of times).
// The block's pieces go to `pt` first; a lane finds its entry's piece there.
template <typename T, bool VCS, class F>
__device__ __forceinline__ void block_entries(const TbSort &a, const Block &k, const PieceTab &pt,
                                              F &&f) {
  const int lane = threadIdx.x & 31;
  int n = 0;  // pieces
  if (VCS) {
    n = k.r1 - k.r0;
    for (int i = lane; i < n; i += 32) {
      const int r = k.r0 + i;
      pt.start[i] = max(a.vptr[r], k.e0);
      pt.val[i] = static_cast<const float *>(a.vals)[r];
      if (k.type != 0) pt.slice[i] = k.s0;
    }
    if (k.type == 0)  // the slice of every run: each lane takes slices, writes their runs
      for (int sl = k.s0 + lane; sl < k.s1; sl += 32)
        for (int r = a.ptr[sl]; r < a.ptr[sl + 1]; ++r) pt.slice[r - k.r0] = sl;
  } else if (k.type == 0) {
    n = k.s1 - k.s0;
    for (int i = lane; i < n; i += 32) {
      pt.start[i] = a.ptr[k.s0 + i];
      pt.slice[i] = k.s0 + i;
    }
  } else {
    n = 1;
    if (lane == 0) {
      pt.start[0] = k.e0;
      pt.slice[0] = k.s0;
    }
  }
  __syncwarp();
  for (int b0 = k.e0; b0 < k.e1; b0 += 32) {
    const int e = b0 + lane;
    const bool ok = e < k.e1;
    int lo = 0, hi = n - 1;  // the last piece starting at or before e (empty ones start there too)
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (pt.start[mid] <= e)
        lo = mid;
      else
        hi = mid - 1;
    }
    const T v = !ok ? T(0) : (VCS ? (T)pt.val[lo] : static_cast<const T *>(a.vals)[e]);
    f(e, pt.slice[lo], v, ok);
  }
  __syncwarp();  // the table is rewritten for the warp's next block
}

// Pass 1: entries per (superblock, bucket).
template <typename T, bool VCS>
__global__ void __launch_bounds__(kTbWarps * 32) tb_count_kernel(const TbSort a) {
  extern __shared__ __align__(16) unsigned char tb_smem[];
  const int B = a.T * a.C, wid = threadIdx.x >> 5;
  int *hist = reinterpret_cast<int *>(tb_smem);  // [T*C]
  const PieceTab pt = PieceTab::at(tb_smem + (B * 4 + 15) / 16 * 16 + wid * PieceTab::kBytes);
  for (int q = threadIdx.x; q < B; q += blockDim.x) hist[q] = 0;
  __syncthreads();
  const int b_lo = blockIdx.x * kTbBlocksPerCta;
  const int b_hi = min(b_lo + kTbBlocksPerCta, a.n_blocks);
  for (int b = b_lo + wid; b < b_hi; b += kTbWarps) {
    const int c = group_of(a.bounds, a.C, b);
    const Block k = load_block(a.blocks, b);
    block_entries<T, VCS>(a, k, pt, [&](int e, int, T, bool ok) {
      if (ok) atomicAdd(&hist[(a.idx[e] / a.tile_rows) * a.C + c], 1);
    });
  }
  __syncthreads();
  for (int q = threadIdx.x; q < B; q += blockDim.x) a.counts[(int64_t)blockIdx.x * B + q] = hist[q];
}

// Per bucket: exclusive scan of its counts over the superblocks, and its total.
__global__ void __launch_bounds__(256) tb_scan_kernel(int *counts, int n_sb, int B, int *tot) {
  const int b = blockIdx.x;
  int running = 0;
  for (int s0 = 0; s0 < n_sb; s0 += 256) {
    const int sb = s0 + threadIdx.x;
    const int v = sb < n_sb ? counts[(int64_t)sb * B + b] : 0;
    int total = 0;
    const int ex = block_exclusive_scan<256>(v, total);
    if (sb < n_sb) counts[(int64_t)sb * B + b] = running + ex;
    running += total;
  }
  if (threadIdx.x == 0) tot[b] = running;
}

// Exclusive scan of the bucket totals (B <= 1024): base[b], base[B] = all.
__global__ void __launch_bounds__(1024) tb_base_kernel(const int *tot, int B, int *base) {
  const int v = threadIdx.x < B ? tot[threadIdx.x] : 0;
  int total = 0;
  const int ex = block_exclusive_scan<1024>(v, total);
  if (threadIdx.x < B) base[threadIdx.x] = ex;
  if (threadIdx.x == 0) base[B] = total;
}

// Pass 2: stable placement.  Warp w takes the superblock's blocks
// w * 8 .. w * 8 + 7 in order; it counts its entries per bucket, the CTA turns
// the counts into starting positions (warps in order), and the warp places its
// entries, lanes in entry order.
template <typename T, bool VCS>
__global__ void __launch_bounds__(kTbWarps * 32) tb_place_kernel(const TbSort a) {
  extern __shared__ __align__(16) unsigned char tb_smem[];
  const int B = a.T * a.C, wid = threadIdx.x >> 5;
  int *cur = reinterpret_cast<int *>(tb_smem);  // [kTbWarps][T*C]
  const PieceTab pt =
      PieceTab::at(tb_smem + (kTbWarps * B * 4 + 15) / 16 * 16 + wid * PieceTab::kBytes);
  const unsigned lt = lanemask_lt();
  for (int q = threadIdx.x; q < kTbWarps * B; q += blockDim.x) cur[q] = 0;
  __syncthreads();
  constexpr int kPer = kTbBlocksPerCta / kTbWarps;
  const int b_lo = blockIdx.x * kTbBlocksPerCta + wid * kPer;
  const int b_hi = min(b_lo + kPer, a.n_blocks);
  int *mine = cur + wid * B;
  for (int b = b_lo; b < b_hi; ++b) {
    const int c = group_of(a.bounds, a.C, b);
    const Block k = load_block(a.blocks, b);
    block_entries<T, VCS>(a, k, pt, [&](int e, int, T, bool ok) {
      const int bk = ok ? (a.idx[e] / a.tile_rows) * a.C + c : -1;
      const unsigned peers = __match_any_sync(kFullMask, bk);
      if (ok && (peers & lt) == 0) mine[bk] += __popc(peers);
      __syncwarp();
    });
  }
  __syncthreads();
  for (int q = threadIdx.x; q < B; q += blockDim.x) {
    int run = a.base[q] + a.counts[(int64_t)blockIdx.x * B + q];
    for (int w = 0; w < kTbWarps; ++w) {
      const int v = cur[w * B + q];
      cur[w * B + q] = run;
      run += v;
    }
  }
  __syncthreads();
  T *rv = static_cast<T *>(a.rec_val);
  for (int b = b_lo; b < b_hi; ++b) {
    const int c = group_of(a.bounds, a.C, b);
    const Block k = load_block(a.blocks, b);
    block_entries<T, VCS>(a, k, pt, [&](int e, int sl, T v, bool ok) {
      const int row = ok ? a.idx[e] : 0;
      const int t = row / a.tile_rows;
      const int bk = ok ? t * a.C + c : -1;
      const unsigned peers = __match_any_sync(kFullMask, bk);
      if (ok) {
        const int p = mine[bk] + __popc(peers & lt);
        a.rec_row[p] = (uint16_t)(row - t * a.tile_rows);
        a.rec_slice[p] = sl;
        rv[p] = v;
      }
      __syncwarp();
      if (ok && (peers & lt) == 0) mine[bk] += __popc(peers);
      __syncwarp();
    });
  }
}

// ------------------------------------------------------------------ apply

template <typename T>
struct TbSmem {
  static constexpr int kCap = sizeof(T) == 4 ? 4096 : 2048;               // records per window
  static constexpr int kKey = 0;                                          // u32 [kCap]: row
  static constexpr int kSlc = kKey + kCap * 4;                            // i32 [kCap]
  static constexpr int kVal = kSlc + kCap * 4;                            // T [kCap]
  static constexpr int kCount = kVal + kCap * (int)sizeof(T);             // i32 [warp][owner]
  static constexpr int kCursor = kCount + kTbAWarps * kTbAWarps * 4;      // i32 [warp][owner]
  static constexpr int kSplit = kCursor + kTbAWarps * kTbAWarps * 4;      // i32 [owner + 1]
  static constexpr int kHist = kSplit + (kTbAWarps + 1) * 4 + 12;         // i32 [tile rows]
  static constexpr int kOwner = kHist + kTtRows * 4;                      // u8 [tile rows]
  static constexpr int kTile = (kOwner + kTtRows + 15) / 16 * 16;
  static_assert(kVal % 16 == 0 && kHist % 16 == 0 && kTile % 16 == 0, "shared-memory alignment");
  static_assert(kTile + kTtRows * kTbPassBytes <= 227 * 1024, "fits one CTA's shared memory");
};

struct TbApply {
  const int *base;            // [T*C + 1]
  const uint16_t *rec_row;
  const int32_t *rec_slice;
  const void *rec_val;
  const void *X;
  int64_t ldx;
  void *out;
  int64_t ldo;
  int64_t part_stride;
  int64_t n_t;
  int tile_rows, C, w;
};

// Block (tile blockIdx.x, group blockIdx.y): bucket blockIdx.x * C + blockIdx.y.
template <typename T, int VEC, int Q>
__global__ void __launch_bounds__(kTbAThreads, 1) tb_apply_kernel(const TbApply a) {
  using V = typename VecT<T, VEC>::type;
  using Ops = VecOps<T, VEC>;
  using SL = TbSmem<T>;
  constexpr int E = 32 / Q;
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t *key = reinterpret_cast<uint32_t *>(smem + SL::kKey);
  int32_t *kslc = reinterpret_cast<int32_t *>(smem + SL::kSlc);
  T *kval = reinterpret_cast<T *>(smem + SL::kVal);
  int *cnt = reinterpret_cast<int *>(smem + SL::kCount);
  int *cur = reinterpret_cast<int *>(smem + SL::kCursor);
  int *split = reinterpret_cast<int *>(smem + SL::kSplit);
  int *hist = reinterpret_cast<int *>(smem + SL::kHist);
  uint8_t *owner = smem + SL::kOwner;
  T *tile = reinterpret_cast<T *>(smem + SL::kTile);

  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const unsigned lt = lanemask_lt();
  const int tk = blockIdx.x, c = blockIdx.y;
  const int bucket = tk * a.C + c;
  const int r0 = a.base[bucket], r1 = a.base[bucket + 1];
  const int t0 = tk * a.tile_rows;
  const int64_t rem = a.n_t - t0;
  const int rows = rem < a.tile_rows ? (int)rem : a.tile_rows;
  const int w = a.w;
  for (int q = threadIdx.x; q < rows * w; q += kTbAThreads) tile[q] = T(0);
  for (int q = threadIdx.x; q < rows; q += kTbAThreads) hist[q] = 0;
  __syncthreads();
  // owners: row ranges balanced by the bucket's row counts
  for (int p = r0 + threadIdx.x; p < r1; p += kTbAThreads) atomicAdd(&hist[a.rec_row[p]], 1);
  __syncthreads();
  if (wid == 0) {
    const int total = r1 - r0;
    int below = 0, carry = 0;  // lane b (1 .. W-1): rows before owner b's first
    for (int q0 = 0; q0 < rows; q0 += 32) {
      const bool ok = q0 + lane < rows;
      const int v = ok ? hist[q0 + lane] : 0;
      const int ex = carry + warp_inclusive_scan(v) - v;
      for (int b = 1; b < kTbAWarps; ++b) {
        const unsigned m =
            __ballot_sync(kFullMask, ok && (int64_t)ex * kTbAWarps < (int64_t)b * total);
        if (lane == b) below += __popc(m);
      }
      carry = __shfl_sync(kFullMask, ex + v, 31);
    }
    if (lane == 0) split[0] = 0;
    if (lane >= 1 && lane < kTbAWarps) split[lane] = below;
    if (lane == kTbAWarps) split[kTbAWarps] = rows;
  }
  __syncthreads();
  for (int q = split[wid] + lane; q < split[wid + 1]; q += 32) owner[q] = (uint8_t)wid;
  __syncthreads();

  const T *__restrict__ X = static_cast<const T *>(a.X);
  const T *__restrict__ rvals = static_cast<const T *>(a.rec_val);
  const int grp = lane / Q;
  const int col0 = (lane % Q) * VEC;
  const bool colok = col0 < w;
  int *mycnt = cnt + wid * kTbAWarps;
  int *mycur = cur + wid * kTbAWarps;

  for (int W0 = r0; W0 < r1; W0 += SL::kCap) {
    const int W1 = min(W0 + SL::kCap, r1);
    const int span = (W1 - W0 + kTbAWarps - 1) / kTbAWarps;
    const int b0 = min(W0 + wid * span, W1), b1 = min(b0 + span, W1);  // this warp's share
    if (lane < kTbAWarps) mycnt[lane] = 0;
    __syncwarp();
    for (int p0 = b0; p0 < b1; p0 += 32) {
      const int p = p0 + lane;
      const int o = p < b1 ? (int)owner[a.rec_row[p]] : -1;
      const unsigned peers = __match_any_sync(kFullMask, o);
      if (o >= 0 && (peers & lt) == 0) mycnt[o] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    int tot = 0, before = 0;
    if (lane < kTbAWarps) {
#pragma unroll
      for (int k = 0; k < kTbAWarps; ++k) {
        const int v = cnt[k * kTbAWarps + lane];
        tot += v;
        before += k < wid ? v : 0;
      }
    }
    const int tincl = warp_inclusive_scan(tot);
    if (lane < kTbAWarps) mycur[lane] = tincl - tot + before;
    const int ob = __shfl_sync(kFullMask, tincl - tot, wid);  // this warp's own records
    const int oe = ob + __shfl_sync(kFullMask, tot, wid);
    __syncwarp();
    for (int p0 = b0; p0 < b1; p0 += 32) {
      const int p = p0 + lane;
      const int row = p < b1 ? (int)a.rec_row[p] : -1;
      const int o = row >= 0 ? (int)owner[row] : -1;
      const unsigned peers = __match_any_sync(kFullMask, o);
      if (o >= 0) {
        const int pp = mycur[o] + __popc(peers & lt);
        key[pp] = (uint32_t)row;
        kslc[pp] = a.rec_slice[p];
        kval[pp] = rvals[p];
      }
      __syncwarp();
      if (o >= 0 && (peers & lt) == 0) mycur[o] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // ---- this warp's records [ob, oe) in order, E per step
    auto load = [&](int q0, int &tr, T &av, T (&x)[VEC]) {
      const int qi = q0 + grp;
      tr = -1;
      av = T(0);
#pragma unroll
      for (int v = 0; v < VEC; ++v) x[v] = T(0);
      if (qi < oe) {
        tr = (int)key[qi];
        av = kval[qi];
        if (colok)
          Ops::unpack(ld_gather(reinterpret_cast<const V *>(X + (int64_t)kslc[qi] * a.ldx + col0)),
                      x);
      }
    };
    auto add = [&](int tr, T av, const T (&x)[VEC]) {
      V *p = reinterpret_cast<V *>(tile + tr * w + col0);
      T y[VEC];
      Ops::unpack(*p, y);
#pragma unroll
      for (int v = 0; v < VEC; ++v) y[v] = tb_fma(av, x[v], y[v]);
      *p = Ops::pack(y);
    };
    int tn;
    T an, xn[VEC];
    load(ob, tn, an, xn);
    for (int q0 = ob; q0 < oe; q0 += E) {
      const int tr = tn;
      const T av = an;
      T x[VEC];
#pragma unroll
      for (int v = 0; v < VEC; ++v) x[v] = xn[v];
      if (q0 + E < oe) load(q0 + E, tn, an, xn);
      const unsigned peers = __match_any_sync(kFullMask, tr);
      const bool dup = tr >= 0 && __popc(peers) > Q;
      if (!__any_sync(kFullMask, dup)) {
        if (tr >= 0 && colok) add(tr, av, x);
      } else {
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

  T *__restrict__ out = static_cast<T *>(a.out) + (int64_t)c * a.part_stride;
  for (int q = threadIdx.x; q < rows * w; q += kTbAThreads) {
    const int rr = q / w, cc = q - rr * w;
    out[(int64_t)(t0 + rr) * a.ldo + cc] = tile[q];
  }
}

using TbKernel = void (*)(const TbApply);

template <typename T>
TbKernel pick_tb(bool vec, int Q) {
  constexpr int VW = 16 / sizeof(T);
  if (vec) {
    switch (Q) {
      case 1: return tb_apply_kernel<T, VW, 1>;
      case 2: return tb_apply_kernel<T, VW, 2>;
      case 4: return tb_apply_kernel<T, VW, 4>;
    }
  } else {
    switch (Q) {
      case 1: return tb_apply_kernel<T, 1, 1>;
      case 2: return tb_apply_kernel<T, 1, 2>;
      case 4: return tb_apply_kernel<T, 1, 4>;
      case 8: return tb_apply_kernel<T, 1, 8>;
      case 16:
        if constexpr (sizeof(T) == 4) return tb_apply_kernel<T, 1, 16>;
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

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

template <typename T, bool VCS>
vs_status tb_typed(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y, int64_t w,
                   cudaStream_t s) {
  constexpr int VW = 16 / sizeof(T);
  const int TR = kTtRows;
  const int64_t n_t = Y.rows;
  const int T_ = (int)((n_t + TR - 1) / TR);
  const int C = m.tp_chunks;
  const int B = T_ * C;
  const int n_sb = (int)((m.n_blocks + kTbBlocksPerCta - 1) / kTbBlocksPerCta);
  const int64_t pass = kTbPassBytes / (int64_t)sizeof(T);
  // handle scratch: counts, totals, bases, records, group partials
  const size_t o_counts = 0;
  const size_t o_tot = align256(o_counts + sizeof(int) * (size_t)n_sb * B);
  const size_t o_base = align256(o_tot + sizeof(int) * (size_t)B);
  const size_t o_slice = align256(o_base + sizeof(int) * (size_t)(B + 1));
  const size_t o_val = align256(o_slice + sizeof(int32_t) * (size_t)m.nnz);
  const size_t o_row = align256(o_val + sizeof(T) * (size_t)m.nnz);
  const size_t o_part = align256(o_row + sizeof(uint16_t) * (size_t)m.nnz);
  const size_t need = o_part + (C > 1 ? sizeof(T) * (size_t)C * n_t * pass : 0);
  VS_TRY(h.tb_scratch.reserve(need, s));
  char *sp = static_cast<char *>(h.tb_scratch.p);
  TbSort so;
  so.ptr = m.ptr;
  so.vptr = m.vptr;
  so.idx = m.idx;
  so.vals = m.vals;
  so.blocks = m.blocks;
  so.bounds = m.tp_bounds;
  so.n_blocks = (int)m.n_blocks;
  so.C = C;
  so.T = T_;
  so.tile_rows = TR;
  so.counts = reinterpret_cast<int *>(sp + o_counts);
  so.tot = reinterpret_cast<int *>(sp + o_tot);
  so.base = reinterpret_cast<int *>(sp + o_base);
  so.rec_slice = reinterpret_cast<int32_t *>(sp + o_slice);
  so.rec_val = sp + o_val;
  so.rec_row = reinterpret_cast<uint16_t *>(sp + o_row);
  void *part = sp + o_part;
  // the records, once per call
  {
    const int smem = (B * 4 + 15) / 16 * 16 + kTbWarps * PieceTab::kBytes;
    int resident = 0;  // (raises the kernel's shared-memory limit once)
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(tb_count_kernel<T, VCS>),
                            kTbWarps * 32, smem, &resident));
    tb_count_kernel<T, VCS><<<n_sb, kTbWarps * 32, smem, s>>>(so);
    VS_LAUNCH_CHECK();
  }
  tb_scan_kernel<<<B, 256, 0, s>>>(so.counts, n_sb, B, so.tot);
  VS_LAUNCH_CHECK();
  tb_base_kernel<<<1, 1024, 0, s>>>(so.tot, B, so.base);
  VS_LAUNCH_CHECK();
  {
    const int smem = (kTbWarps * B * 4 + 15) / 16 * 16 + kTbWarps * PieceTab::kBytes;
    int resident = 0;  // (raises the kernel's shared-memory limit once)
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(tb_place_kernel<T, VCS>),
                            kTbWarps * 32, smem, &resident));
    tb_place_kernel<T, VCS><<<n_sb, kTbWarps * 32, smem, s>>>(so);
    VS_LAUNCH_CHECK();
  }
  // the products, one column pass at a time
  for (int64_t c0 = 0; c0 < w; c0 += pass) {
    const int wb = (int)std::min<int64_t>(pass, w - c0);
    const T *xp = static_cast<const T *>(X.p) + c0;
    T *yp = static_cast<T *>(Y.p) + c0;
    const bool vec = wb % VW == 0 && reinterpret_cast<uintptr_t>(xp) % 16 == 0 && X.ld % VW == 0;
    const TbKernel k = pick_tb<T>(vec, pow2_at_least(vec ? wb / VW : wb));
    if (!k) {
      set_error("no bucketed two-phase kernel for this width");
      return VS_ERR_UNSUPPORTED;
    }
    const int smem = TbSmem<T>::kTile + TR * wb * (int)sizeof(T);
    int resident = 0;
    VS_TRY(kernel_occupancy(reinterpret_cast<const void *>(k), kTbAThreads, smem, &resident));
    TbApply aa;
    aa.base = so.base;
    aa.rec_row = so.rec_row;
    aa.rec_slice = so.rec_slice;
    aa.rec_val = so.rec_val;
    aa.X = xp;
    aa.ldx = X.ld;
    aa.n_t = n_t;
    aa.tile_rows = TR;
    aa.C = C;
    aa.w = wb;
    if (C == 1) {
      aa.out = yp;
      aa.ldo = Y.ld;
      aa.part_stride = 0;
    } else {
      aa.out = part;
      aa.ldo = wb;
      aa.part_stride = n_t * wb;
    }
    k<<<dim3((unsigned)T_, (unsigned)C), kTbAThreads, smem, s>>>(aa);
    VS_LAUNCH_CHECK();
    if (C > 1) VS_TRY(launch_combine(part, C, n_t, wb, yp, Y.ld, sizeof(T), m.n_sm, s));
  }
  return VS_OK;
}

}  // namespace

bool tb_applies(const Matrix &m, int64_t n_out) {
  if (m.wide || m.borrowed_idx || m.nnz == 0 || m.n_blocks == 0 || m.tp_chunks < 1) return false;
  const int64_t tiles = (n_out + kTtRows - 1) / kTtRows;
  return tiles * m.tp_chunks <= kTbMaxBuckets && m.nnz < (int64_t(1) << 31);
}

vs_status launch_tb_two_phase(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y, int64_t w,
                              cudaStream_t s) {
  if (m.layout == VS_LAYOUT_VCS) return tb_typed<float, true>(h, m, X, Y, w, s);
  if (m.dtype == VS_F64) return tb_typed<double, false>(h, m, X, Y, w, s);
  return tb_typed<float, false>(h, m, X, Y, w, s);
}

}  // namespace vs
