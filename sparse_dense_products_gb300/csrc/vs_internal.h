// vs_internal.h -- handle layout, status helpers and launcher declarations
// shared by the translation units of libvs.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <memory>
#include <string>
#include <vector>

#include "../../include/vs.h"

namespace vs {

// ------------------------------------------------------------------ errors

void set_error(const std::string &msg);
const char *last_error();

struct Err {
  vs_status code;
  std::string msg;
};

// Returns VS_ERR_CUDA (with the message) if the last CUDA call failed.
vs_status cuda_status(cudaError_t e, const char *what);

#define VS_CUDA(call)                                          \
  do {                                                         \
    cudaError_t e_ = (call);                                   \
    if (e_ != cudaSuccess) return ::vs::cuda_status(e_, #call); \
  } while (0)

// Counts one kernel launch and checks that it was accepted.
void note_launch();
int64_t launch_count();
#define VS_LAUNCH_CHECK()                     \
  do {                                        \
    ::vs::note_launch();                      \
    VS_CUDA(cudaGetLastError());              \
  } while (0)

#define VS_TRY(call)                 \
  do {                               \
    vs_status s_ = (call);           \
    if (s_ != VS_OK) return s_;      \
  } while (0)

// ------------------------------------------------------------------ layout

// Matrix blocks streamed through shared memory (stage.cuh): at most this many
// entries, runs and slices per block.  A slice with more entries (or, in VCS,
// more runs) is "long": it is cut into chunks within the same limits, and each
// chunk into shares of kShareEntries entries.  The cut points depend on the
// matrix only, so the summation order does too.
constexpr int kBlockEntries = 1024;
constexpr int kBlockRuns = 256;
constexpr int kBlockSlices = 256;
constexpr int kShareEntries = 256;
constexpr int kWarpsPerCta = 8;   // consumer warps; one more warp produces

// Widest column block one kernel launch handles; wider products loop.
constexpr int kMaxBlockWidth = 64;

// Tiled two-phase: warps per CTA, row owners the build balances (8 per
// warp), default and largest rows per tile, CTAs resident per multiprocessor
// (the tile takes most of its shared memory), and the CTA count the group
// count aims at (one per multiprocessor of a GB300).
constexpr int kTtWarps = 16;
constexpr int kTtOwners = kTtWarps * 8;
constexpr int kTtRows = 2048;
constexpr int kTtCtasPerSm = 1;
constexpr int kTtTargetCtas = 152 * kTtCtasPerSm;
// Bucketed two-phase: at most this many (tile, group) buckets.
constexpr int kTbMaxBuckets = 1024;

// One stored layout of a matrix: CSR/CSC or VCSR/VCSC.
struct Matrix {
  vs_layout layout = VS_LAYOUT_CSR;
  vs_major major = VS_MAJOR_ROW;
  vs_dtype dtype = VS_F32;
  int64_t n_rows = 0, n_cols = 0;
  int64_t n_major = 0, n_minor = 0;
  int64_t nnz = 0;
  int64_t R = 0;  // VCS runs (CSR: nnz)

  int32_t *ptr = nullptr;   // [n_major+1]  CSR slice starts / VCS run starts
  int32_t *idx = nullptr;   // [nnz]        minor indices
  void *vals = nullptr;     // CSR: [nnz] of dtype; VCS: [R] float32
  int32_t *vptr = nullptr;  // VCS: [R+1]  index starts of the runs

  // Matrix-only kernel parameters.
  int g = 1;                    // group size: threads per slice (power of 2 in [1, 32])
  int64_t n_blocks = 0;         // staged blocks
  int4 *blocks = nullptr;       // [n_blocks][3] descriptors (stage.cuh)
  int64_t n_long = 0;           // long slices
  int64_t n_chunks = 0;         // chunks over all long slices
  int64_t n_shares = 0;         // shares over all long slices
  int4 *longs = nullptr;        // [n_long] {slice, first share, shares, 0}
  void *partials = nullptr;     // [n_shares * kMaxBlockWidth] slots of 8 bytes (sums of the operand type)
  int *err = nullptr;           // device flag: a bounded wait gave up
  bool sorted_segments = false; // minor indices ascend inside every run / row
  int n_sm = 1;                 // multiprocessors of the device the matrix lives on

  // Two-phase (deterministic misaligned) chunking: C groups of consecutive
  // blocks with balanced entry counts, fixed by the matrix.
  int tp_chunks = 0;                // C
  int32_t *tp_bounds = nullptr;     // [C+1] block boundaries of the groups

  // Tiled two-phase: the output rows (the minor axis) in tiles of tt_rows.
  // With minor indices ascending in every run (slice), the entries of run r
  // inside tile k form one range, and tt_tab holds where each such range
  // starts, so that the CTA of a tile visits its own entries only.  The
  // entries are cut into tt_groups groups by position (fixed by the matrix
  // and never by the tiling); tt_own balances each (tile, group)'s rows over
  // the CTA's row owners by the group's entry counts.  tt_rows == 0: not built
  // (the block-stream scheme above runs instead).
  int tt_req_rows = 0;              // rows per tile asked for at build (0: kTtRows)
  int tt_rows = 0;                  // rows per tile
  int tt_tiles = 0;                 // tiles over the minor axis
  int tt_groups = 0;                // entry groups
  int32_t *tt_tab = nullptr;        // [(tiles-1) * pieces]: first entry of run r at minor >= k*tt_rows, row k-1
  int32_t *tt_run_slice = nullptr;  // VCS: [R] the slice of every run
  int32_t *tt_group = nullptr;      // [3*groups+1]: entry bounds, first runs, ends of runs
  int32_t *tt_own = nullptr;        // [tiles * groups * (kTtOwners+1)] first row of each owner

  // When set, the index arrays (ptr, idx, vptr, blocks, longs, tp_bounds, the
  // tt_ arrays, and for a wide matrix ptr64, vptr64 and its segments' index arrays) are shared
  // with other matrices (vs_scale_entries) and freed with the last reference;
  // vals, partials and err always belong to this matrix (its segments').
  std::shared_ptr<void> index_owner;

  // Wide matrices: 64-bit slice pointers with int32 indices ("Regridder",
  // "Why not cuSPARSE").  The stored layout is ptr64 (CSR entry starts, or VCS
  // run starts) and for VCS vptr64 (run entry starts), with idx and vals as
  // usual; ptr and vptr stay null.  The kernels run over `segs`: consecutive
  // slice ranges of fewer than 2^31 entries (and runs), each an ordinary
  // int32 matrix with slice pointers relative to its first entry (and run)
  // whose idx and vals view this matrix's arrays.  Every slice keeps the
  // summation tree it would have in one piece (the group size is the whole
  // matrix's), so the products have the same bits as an int32 build.
  bool wide = false;
  int64_t *ptr64 = nullptr;     // [n_major + 1]
  int64_t *vptr64 = nullptr;    // VCS: [R + 1]
  int64_t seg_entries = 0;      // wide: at most this many entries per segment (one longer slice alone)
  std::vector<Matrix> segs;     // wide: the kernel segments, in slice order
  // A segment: its first slice in the wide matrix, and where its views of
  // the wide matrix's arrays start (idx at seg_entry0, VCS values at
  // seg_run0): the 16-byte boundary at or before its first entry (run), so
  // its pointers count seg_lead_e entries (seg_lead_r runs) of the previous
  // segment first, which none of its slices names.  Once they are views
  // (borrowed_idx, borrowed_vals) they are never freed here.
  int64_t seg_slice0 = 0, seg_entry0 = 0, seg_run0 = 0;
  int seg_lead_e = 0, seg_lead_r = 0;
  bool borrowed_idx = false, borrowed_vals = false;  // idx / vals are such views

  size_t dsize() const { return dtype == VS_F64 ? 8 : 4; }
  int64_t layout_bytes() const;
  int64_t meta_bytes() const;
};

// Scratch that grows on demand, owned by a handle.
struct Scratch {
  void *p = nullptr;
  size_t bytes = 0;
  vs_status reserve(size_t need, cudaStream_t s);
  void release();
};

// Group size rule ("Regridder", "How it is built": as many threads as an
// average slice has entries, up to a warp): the largest power of two <= the
// mean entries per slice, clamped to [1, 32].
inline int group_size_rule(int64_t nnz, int64_t n_major) {
  int g = 1;
  if (n_major > 0) {
    const int64_t mean = nnz / n_major;
    while (g * 2 <= mean && g < 32) g *= 2;
  }
  return g;
}

void free_matrix(Matrix &m);
void set_group_size(Matrix &m, int g);
vs_status dev_alloc(void **p, size_t bytes);
vs_status share_index_arrays(Matrix &m);

}  // namespace vs

struct vs_handle_s {
  vs::Matrix A;
  vs::Matrix *T = nullptr;  // exact transpose (other major), once attached
  int device = 0;
  vs::Scratch tp_partials;   // two-phase chunk partials
  vs::Scratch tb_scratch;    // bucketed two-phase: the call's records and partials
  vs::Scratch stage_B, stage_out;  // host-operand staging (vs_spmm_host)
  int *host_flags = nullptr;       // pinned: the failure flags of A and T (their segments), read back by vs_spmm_host
  int host_flag_cap = 0;           // ints host_flags holds
  vs::Scratch wide_tmp;            // two-phase over a wide matrix: one segment's sum before it is added
  vs::Scratch view_vals, view_tvals, view_X;  // normalized views: mapped values, scaled X
  vs::Scratch floor_sink;                      // vs_gather_floor's per-thread sums
  int forced_g = 0;                            // vs_force_group_size (0: the matrix rule)
};

namespace vs {

// ------------------------------------------------------------------ builders (assembly.cu)

// Builds a CSR/CSC (layout CSR) or VCSR/VCSC (layout VCS) from device COO.
// `major_idx` / `minor_idx` are the COO coordinates along the major / minor
// axis.  Fills `m` (device arrays owned by m).  Synchronises `s`.
vs_status build_matrix(Matrix &m, vs_layout layout, vs_major major, vs_dtype dtype,
                       int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                       const int32_t *d_col, const void *d_val, cudaStream_t s);

// Builds a wide matrix (64-bit slice pointers, kernel segments of at most
// `seg_entries` entries) from device COO of any length: the global checks and
// per-slice counts run over all entries, then each segment's entries are
// selected in input order and assembled like build_matrix; finally each
// segment is prepared (prepare_matrix) with the whole matrix's group size.
// Synchronises `s`.
vs_status build_wide(Matrix &m, vs_layout layout, vs_major major, vs_dtype dtype, int64_t n_rows,
                     int64_t n_cols, int64_t nnz, const int32_t *d_row, const int32_t *d_col,
                     const void *d_val, int64_t seg_entries, cudaStream_t s);

// Builds the other-major layout of `src` into `dst` from src's own arrays
// (wide when src is; dst then still needs prepare_matrix unless wide).
vs_status build_transpose(const Matrix &src, Matrix &dst, cudaStream_t s);

// The default segment size of wide matrices: the most entries an int32
// segment takes with room for the padded over-reads of its arrays.
constexpr int64_t kMaxSegmentEntries = (int64_t(1) << 31) - (int64_t(1) << 21);

// Fills the matrix-only kernel parameters of `m` (g, chunk tasks, two-phase
// chunk bounds) from its device arrays.  Synchronises `s`.
vs_status prepare_matrix(Matrix &m, cudaStream_t s);

// ------------------------------------------------------------------ products

// Dense operand in the slice frame: row r of X is the dense vector that pairs
// with index r; Y likewise.  Strides in elements; the width axis is contiguous.
struct DenseView {
  void *p;
  int64_t rows;
  int64_t ld;
  // Output only: when set, row r of the result is multiplied by scale[r]
  // before it is stored (the gather fuses it; other kernels take a pass).
  const void *scale = nullptr;
  // The dense operands are float64 (for a float32 or VCS matrix: the mixed
  // products, float values with float64 operands and sums).
  bool f64 = false;
};

// Aligned gather: Y[s, 0:w] = sum over entries (t, a) of slice s of a * X[t, 0:w].
vs_status launch_gather(const Matrix &m, DenseView X, DenseView Y, int64_t w, cudaStream_t s);

// Misaligned scatter with atomic adds into a zero-filled Y.
vs_status launch_scatter_atomic(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                cudaStream_t s);

// Tiled two-phase (m.tt_rows > 0) over column passes of at most 64 bytes and
// at most `max_pass` columns: each pass writes Y directly (one group) or the
// group partials into `part` (groups * Y.rows * max_pass elements), which
// combine_kernel then adds in group order.
vs_status launch_tt_two_phase(const Matrix &m, DenseView X, DenseView Y, int64_t w, void *part,
                              int64_t max_pass, cudaStream_t s);

// Y[t, 0:w] = sum over groups k (in order) of P[k][t, 0:w] (P: [C][n_t][w]
// of `dsize`-byte elements).
vs_status launch_combine(const void *P, int C, int64_t n_t, int w, void *Y, int64_t ldy,
                         size_t dsize, int n_sm, cudaStream_t s);

// Bucketed two-phase: whether it serves `m` (no tiled arrays kept) for an output
// of n_out rows, and the product (handle scratch holds each call's records).
bool tb_applies(const Matrix &m, int64_t n_out);
vs_status launch_tb_two_phase(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y, int64_t w,
                              cudaStream_t s);

// Builds the tiled two-phase arrays of `m` (nothing when they do not apply or
// would exceed half the layout's bytes).  `ptr` / `vptr` are host copies of
// m's slice and run pointers.  Synchronises `s`.
vs_status build_tiled_two_phase(Matrix &m, const std::vector<int32_t> &ptr,
                                const std::vector<int32_t> &vptr, cudaStream_t s);

// Misaligned scatter, deterministic two-phase.
vs_status launch_scatter_two_phase(vs_handle_s &h, const Matrix &m, DenseView X, DenseView Y,
                                   int64_t w, cudaStream_t s);

// The same two-phase product with its partial sums in a statically allocated
// device array (no allocation at call time).
vs_status launch_scatter_two_phase_static(const Matrix &m, DenseView X, DenseView Y, int64_t w,
                                          cudaStream_t s);

// Resident CTAs per SM of `kernel` launched with `threads` threads and
// `smem` bytes of dynamic shared memory, with the kernel allowed the SM's
// whole opt-in shared memory.  Cached per (device, kernel, threads, smem), so
// a product's host path makes no such query after its first call.
vs_status kernel_occupancy(const void *kernel, int threads, int smem, int *per_sm);

// Test hook of the failure path (vs_test_stall_producers): true when this
// gather launch's producer is to issue nothing, so that its consumers' bounded
// waits run out.
bool take_stall();

// Y[0:rows, 0:w] = 0 with row stride ld.
vs_status launch_zero_fill(DenseView Y, int64_t w, size_t dsize, cudaStream_t s);

}  // namespace vs
