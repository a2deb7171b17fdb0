/*
 * vs.h -- C ABI of libvs: sparse x dense products over CSR and the
 * value-grouped VCS layout, on one GB300 GPU (sm_103a).
 *
 * What the library computes (page title, section):
 *
 *  - "Add CUDA transfer and matmul kernels for the normalized views"
 *    (vsparse PR #61), "The layout stays compressed": a VCS matrix keeps, for
 *    each major slice, its nonzeros grouped into runs that share one value:
 *    major_ptr -> (values, value_ptr) -> indices.  It is never expanded to one
 *    float per nonzero.  VCSR: major = rows; VCSC: major = columns.
 *  - Same page, "The kernels": four product directions, VCSR@B, VCSC@B, B@VCSR
 *    and B@VCSC.  A direction is "aligned" when the output's disjoint axis is
 *    the major one (VCSR@B, B@VCSC) and "misaligned" otherwise.
 *  - "Regridder" (regridding PR #70), "How it is built": CSR assembly is a
 *    counting sort (count each row's entries, then place them at the rows'
 *    cursors); a row keeps its entries in element order.  Products are
 *    row-parallel with a thread group whose size depends only on the matrix,
 *    so a product repeats exactly and a column gives the same numbers alone
 *    or in a batch.  The exact transpose is kept once built.
 *
 * Conventions shared by every entry point:
 *
 *  - All device pointers are caller-owned unless stated otherwise.  A handle
 *    owns copies of the matrix arrays and any scratch it needs; it keeps no
 *    pointer to caller memory after its build call returns.
 *  - Every call is enqueued on the caller's `stream` and is asynchronous,
 *    except where a call documents a synchronisation.  The caller keeps the
 *    buffers alive until the stream has passed the call.
 *  - Errors are returned as vs_status; nothing is thrown across the ABI.
 *    vs_last_error() gives a message for the calling thread's last failure.
 *    On error, output buffers are left in an unspecified state.
 *  - Indices (minor coordinates) are int32, so rows and columns stay below
 *    2^31.  Slice pointers are int32 when nnz < 2^31, and int64 ("Regridder",
 *    "Why not cuSPARSE": 64-bit row pointers with 32-bit indices) for larger
 *    matrices or when vs_build_options asks for them.
 *  - Dense operands are described by vs_dense (logical rows x cols plus
 *    strides in elements).  The width axis of B and out must have stride 1:
 *    for A@B that is the column axis (row-major B and out); for B@A it is the
 *    row axis (B and out stored column-major).  Otherwise VS_ERR_LAYOUT.
 *  - out is overwritten (beta = 0).  A slice with no entries yields zeros.
 *    B and out must not overlap.
 *  - A handle's scratch (long-slice share partials, two-phase partials,
 *    host staging) serves every call on that handle: calls on one handle
 *    from several host threads at once, or whose work overlaps on the GPU
 *    (different streams), must be serialised by the caller.  Different
 *    handles are independent.
 */
#ifndef VS_H
#define VS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct vs_handle_s *vs_handle;

typedef enum {
    VS_OK = 0,
    VS_ERR_INVALID = 1,     /* bad argument, unknown enum value, NULL handle/pointer */
    VS_ERR_SHAPE = 2,       /* operand shapes do not match the matrix and direction */
    VS_ERR_LAYOUT = 3,      /* width axis not contiguous, or overlapping operands */
    VS_ERR_RANGE = 4,       /* a COO coordinate lies outside the matrix */
    VS_ERR_ALLOC = 5,       /* device or host allocation failed */
    VS_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
    VS_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up */
    VS_ERR_UNSUPPORTED = 8, /* valid request this build does not implement */
    VS_ERR_NAN = 9          /* a NaN value where VCS needs a run key */
} vs_status;

typedef enum { VS_F32 = 0, VS_F64 = 1 } vs_dtype;
typedef enum { VS_MAJOR_ROW = 0, VS_MAJOR_COL = 1 } vs_major;
typedef enum { VS_A_B = 0, VS_B_A = 1 } vs_direction;
typedef enum { VS_LAYOUT_CSR = 0, VS_LAYOUT_VCS = 1 } vs_layout;

/*
 * Product variants.  Aligned directions always run the deterministic gather;
 * the variant matters only for misaligned directions (VCSC@B, B@VCSR, CSC@B,
 * B@CSR):
 *   VS_DETERMINISTIC  bit-reproducible: the gather over the exact transpose
 *                     when the handle holds one (vs_attach_transpose), else the
 *                     two-phase scheme.
 *   VS_ATOMIC         zero-fill out, then scatter with atomic adds (the pages'
 *                     design); not bit-reproducible.
 *   VS_TRANSPOSED     the aligned gather over the exact transpose held by the
 *                     handle; VS_ERR_INVALID without one.  Bit-identical on
 *                     repeats.
 *   VS_TWO_PHASE      per-block partial sums over tiles of the output in
 *                     shared memory, then a combine in a fixed chunk order.
 *                     Bit-identical on repeats.
 */
typedef enum {
    VS_DETERMINISTIC = 0,
    VS_ATOMIC = 1,
    VS_TRANSPOSED = 2,
    VS_TWO_PHASE = 3
} vs_variant;

typedef struct {
    void *ptr;            /* first element */
    int64_t rows, cols;   /* logical shape */
    int64_t row_stride;   /* elements between (r, c) and (r+1, c) */
    int64_t col_stride;   /* elements between (r, c) and (r, c+1) */
    vs_dtype dtype;
} vs_dense;

typedef struct {
    int32_t layout;         /* vs_layout */
    int32_t major;          /* vs_major */
    int32_t dtype;          /* vs_dtype of the stored values */
    int32_t group_size;     /* g: threads that share one slice, a power of two in [1, 32] */
    int64_t n_rows, n_cols; /* matrix shape */
    int64_t nnz;            /* stored entries (explicit zeros and duplicates kept) */
    int64_t n_runs;         /* VCS: number of runs R; CSR: nnz */
    int64_t chunk_len;      /* L: a slice with more than L entries (VCS: or more than L/4
                               runs) is "long" and is cut into chunks of at most L entries */
    int64_t n_long_slices;  /* long slices */
    int64_t n_chunks;       /* chunks over all long slices */
    int64_t n_blocks;       /* blocks the kernels stream (runs of short slices, or chunks) */
    int32_t has_transpose;  /* 1 once vs_attach_transpose succeeded */
    int32_t pointer_bits;   /* 32 or 64: the width of the stored slice pointers */
    int32_t n_segments;     /* kernel segments (64-bit pointers: consecutive slice ranges of
                               fewer than 2^31 entries each; 1 otherwise) */
    int32_t two_phase_tiles; /* tiles of output rows of the tiled two-phase scheme (the
                               deterministic misaligned product without a transpose);
                               0: the block-stream two-phase scheme runs instead */
} vs_info_t;

typedef struct {
    const void *ptr;          /* n_major+1: CSR slice starts, or VCS major_ptr (run starts);
                                 int32, or int64 when pointer_bits is 64 */
    const int32_t *indices;   /* nnz minor indices */
    const void *values;       /* CSR: nnz values of the handle dtype; VCS: R float32 run values */
    const void *value_ptr;    /* VCS: R+1 index starts of the runs, int32 or int64 like ptr;
                                 CSR: NULL */
    int64_t n_major, nnz, n_runs;
    int32_t pointer_bits;     /* 32 or 64 */
    int32_t reserved;
} vs_arrays;

/*
 * Build options (vs_build_csr_opts, vs_build_vcs_opts).
 *   pointer_bits     0: automatic -- int32 slice pointers below 2^31 entries,
 *                    int64 from 2^31 on; 32 or 64 to choose (32 with 2^31 or
 *                    more entries is VS_ERR_UNSUPPORTED).  With int64 pointers
 *                    the stored layout is ptr (and VCS value_ptr) of int64 with
 *                    int32 indices; the products run the same kernels over
 *                    consecutive slice ranges ("segments") of fewer than 2^31
 *                    entries, and give the same bits as an int32 build.
 *   segment_entries  0: the largest segment the int32 kernels take (about
 *                    2^31 entries); otherwise at most this many entries per
 *                    segment (a slice with more is a segment of its own) --
 *                    lets a small matrix run the many-segment path, as one of
 *                    more than 2^31 entries does.
 *   two_phase_tile_rows
 *                    0: 2048; otherwise 1 .. 2048 -- the output rows per tile
 *                    of the tiled two-phase scheme (VS_TWO_PHASE on a matrix
 *                    whose minor indices ascend inside every run or slice).
 *                    With 0 its per-(run, tile) entry offsets are kept only
 *                    while they take at most half the layout's bytes; a value
 *                    asked for always builds them; -1 never does.  Without
 *                    them VS_TWO_PHASE sorts each call's entries into
 *                    (tile, group) buckets in handle scratch (at most 1,024
 *                    buckets; about 10-14 bytes per entry), or, past that,
 *                    streams the matrix's blocks per tile.  The tile size
 *                    changes no result bit: it lets a small matrix run the
 *                    many-tile path.
 */
typedef struct {
    int32_t pointer_bits;
    int32_t two_phase_tile_rows;
    int64_t segment_entries;
} vs_build_options;

/*
 * vs_build_csr -- CSR (major = VS_MAJOR_ROW) or CSC (VS_MAJOR_COL) of COO
 * triples by a stable counting sort on the device ("Regridder", "How it is
 * built"): per-slice counts, exclusive scan into the slice pointer, then
 * placement at slice cursors so that every slice keeps its entries in COO
 * input order.  Duplicates and explicit zeros are kept; values are copied
 * bit for bit.
 *
 *   n_rows, n_cols   matrix shape (>= 0, < 2^31)
 *   nnz              number of triples (>= 0; from 2^31 on the slice pointers
 *                    are int64, see vs_build_options)
 *   d_row, d_col     device int32[nnz] coordinates
 *   d_val            device values[nnz] of `dtype` (float32 or float64)
 *   major            VS_MAJOR_ROW for CSR, VS_MAJOR_COL for CSC
 *   stream           stream the build runs on
 *   out              receives the new handle (owned by the caller; vs_destroy)
 *
 * Synchronises `stream` once, to read back the coordinate-range check.
 * Returns VS_ERR_RANGE if a coordinate lies outside the matrix.
 */
vs_status vs_build_csr(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                       const int32_t *d_col, const void *d_val, vs_dtype dtype, vs_major major,
                       cudaStream_t stream, vs_handle *out);

/*
 * vs_build_csr_opts, vs_build_vcs_opts -- vs_build_csr and vs_build_vcs with
 * build options (NULL: the defaults, as vs_build_csr / vs_build_vcs).  nnz may
 * reach 2^31 and beyond with 64-bit slice pointers; rows and columns stay
 * below 2^31.  The assembly is the same counting sort: the range and NaN checks
 * and the per-slice counts run over all entries, then each segment's entries
 * are selected in input order and placed like an int32 build's, so the
 * arrays are those of one stable sort.  Errors as for vs_build_csr /
 * vs_build_vcs; VS_ERR_INVALID for bad options, VS_ERR_UNSUPPORTED when one
 * slice holds 2^31 entries or more.
 */
vs_status vs_build_csr_opts(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                            const int32_t *d_col, const void *d_val, vs_dtype dtype,
                            vs_major major, const vs_build_options *opts, cudaStream_t stream,
                            vs_handle *out);
vs_status vs_build_vcs_opts(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                            const int32_t *d_col, const float *d_val, vs_major major,
                            const vs_build_options *opts, cudaStream_t stream, vs_handle *out);

/*
 * vs_build_vcs -- VCSR (major = VS_MAJOR_ROW) or VCSC (VS_MAJOR_COL) of COO
 * triples ("Add CUDA transfer and matmul kernels ...", "The layout stays
 * compressed").  Entries are stably sorted on the device by the key
 * (major, value, minor), the value ordered by the IEEE total order of its
 * float32 bits (-0.0 and +0.0 form separate runs).  A run is a maximal group
 * with equal (major, value); runs of a slice are in ascending value, indices
 * in a run ascending.  Values are float32 (all device floating-point arrays of
 * the view are float32 on that page).
 *
 * Arguments as for vs_build_csr, with float32 values.  Synchronises `stream`
 * once to read back the run count and checks.  Returns VS_ERR_NAN for a NaN
 * value, VS_ERR_RANGE for an out-of-range coordinate.
 */
vs_status vs_build_vcs(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *d_row,
                       const int32_t *d_col, const float *d_val, vs_major major,
                       cudaStream_t stream, vs_handle *out);

/*
 * vs_spmm -- out = A @ B (dir = VS_A_B) or out = B @ A (dir = VS_B_A).
 *
 *   A        handle from vs_build_csr / vs_build_vcs
 *   B        device operand: A@B: n_cols x w, column stride 1;
 *                            B@A: w x n_rows, row stride 1
 *   out      device output:  A@B: n_rows x w, column stride 1;
 *                            B@A: w x n_cols, row stride 1
 *   dir      VS_A_B or VS_B_A
 *   variant  see vs_variant (matters for misaligned directions only)
 *   stream   stream the product runs on
 *
 * B and out have the handle's dtype, or both float64 with a float32 CSR or a
 * VCS handle (float32 stored values, float64 products and sums; misaligned
 * directions then need the transposed route).  Vector loads are used when the
 * width and strides are multiples of 16 bytes and the pointers are 16-byte
 * aligned.
 * w = 0 or an empty matrix returns VS_OK after writing zeros where out has
 * elements.  No allocation happens here for VS_ATOMIC, VS_TRANSPOSED and
 * aligned directions; the two-phase scheme may grow the handle's scratch on
 * first use with a new width (stream-ordered).  Calls on
 * the same handle must not overlap on the GPU (they share scratch).
 * VS_TRANSPOSED needs vs_attach_transpose first, else VS_ERR_INVALID.
 * Errors: VS_ERR_INVALID (NULL handle or descriptor, unknown direction or
 * variant, dtypes that do not match as above), VS_ERR_SHAPE (shapes that
 * do not fit A), VS_ERR_LAYOUT (width axis not of stride 1, a stride smaller
 * than the width, B and out overlapping), VS_ERR_UNSUPPORTED (float64
 * operands with a float32 matrix on the two-phase or atomic route, a row
 * stride of 2^32 bytes or more), VS_ERR_ALLOC / VS_ERR_CUDA from the runtime.
 * A kernel whose bounded wait gave up marks the handle; vs_device_status
 * reports it.
 */
vs_status vs_spmm(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                  vs_variant variant, cudaStream_t stream);

/*
 * vs_spmm_noalloc -- the deterministic product of vs_spmm (VS_DETERMINISTIC)
 * for callers that must not allocate device memory when they run a product:
 * code running inside stream capture, code whose device memory comes from a
 * pool or allocator it does not control, or code that may not call cudaMalloc
 * at that point.  It calls no cudaMalloc, cudaFree or allocating library
 * routine.  (The pages have no counterpart: this entry point exists for such
 * callers only.)
 *
 * Arguments, layouts and results as for vs_spmm with VS_DETERMINISTIC: aligned
 * directions, and misaligned ones on a handle that holds its transpose, run
 * the same gather (which needs no scratch beyond what the handle got at build
 * time); other misaligned products run the same two-phase scheme, with its
 * per-group partial sums in a fixed 32 MiB device array that the
 * library declares statically -- every GPU that loads the library holds those
 * 32 MiB until the process exits.  Results are bit-identical to vs_spmm's.
 * The column block is narrowed until the partial sums fit; a product whose
 * partials do not fit even one column returns VS_ERR_UNSUPPORTED with the
 * sizes in vs_last_error().
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array, which keeps whatever the last call
 * left in it; calls whose work overlaps on the GPU (other streams, other
 * threads) race on it and must be serialised by the caller.  For a matrix
 * with 64-bit slice pointers a misaligned product needs the transposed route
 * (VS_ERR_UNSUPPORTED otherwise).  The looked-up
 * address is kept for the life of the process, so resetting a device
 * (cudaDeviceReset) while the library is loaded is not supported.
 */
vs_status vs_spmm_noalloc(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                          cudaStream_t stream);

/*
 * Normalized views ("Add CUDA transfer and matmul kernels for the normalized
 * views": a view applies a transform g to the stored values and carries
 * O(n_rows + n_cols) statistics; the recipes themselves are not defined
 * there, so this is the generic hook).  The view of A is
 *     V = diag(row_scale) . g(A) . diag(col_scale)
 * with g applied to every stored value (a VCS matrix maps each run's value
 * once, so the layout stays compressed).
 */
typedef enum {
    VS_MAP_IDENTITY = 0,  /* g(v) = v */
    VS_MAP_LOG1P = 1,     /* g(v) = log(1 + v), in the value dtype */
    VS_MAP_SQRT = 2       /* g(v) = sqrt(v), in the value dtype */
} vs_value_map;

typedef struct {
    vs_value_map map;
    const void *row_scale; /* device, n_rows values of the dense dtype, or NULL (ones) */
    const void *col_scale; /* device, n_cols values of the dense dtype, or NULL (ones) */
} vs_view;

/*
 * vs_spmm_view -- out = V@B (dir VS_A_B) or B@V (VS_B_A) for the view V of A
 * defined by `view` (NULL: V = A, the same as vs_spmm).  Variants and layout
 * rules as for vs_spmm.  The scale of the output axis is applied when the
 * gather stores a row (one multiply per element); the scale of the
 * contracted axis pre-scales a copy of the dense operand held by the handle;
 * a mapped g(A) is evaluated into handle scratch once per call.  Scratch
 * grows on first use with a larger operand (stream-ordered).  With the same
 * view and operands the result repeats bit for bit, like vs_spmm.
 * Errors: as vs_spmm; VS_ERR_INVALID for an unknown map.
 */
vs_status vs_spmm_view(vs_handle A, const vs_dense *B, const vs_dense *out, vs_direction dir,
                       vs_variant variant, const vs_view *view, cudaStream_t stream);

/*
 * vs_spmm_host -- vs_spmm with B and out in HOST memory (pinned memory is
 * fastest).  Copies B to device staging owned by the handle, runs vs_spmm on
 * `stream`, copies the result back and synchronises `stream` once before
 * returning, so `out` is ready on return.  Layout rules as for vs_spmm.  The
 * staging buffers grow on first use with a larger operand; a pinned 8-byte
 * status area is allocated on the first call and freed by vs_destroy.
 * A pinned, device-mapped B is staged by a copy kernel reading it through
 * its mapping (loads from every multiprocessor), any other B by the copy
 * engine.  When `out` is pinned host memory mapped into the device's address space
 * (cudaHostAlloc, cudaHostRegister, torch pin_memory) and the product runs as
 * a gather (an aligned product, or VS_DETERMINISTIC / VS_TRANSPOSED over an
 * attached transpose), the kernels store the result straight into it and no
 * copy back is made; elements outside the logical output are never written.
 * Errors: as vs_spmm; VS_ERR_TIMEOUT (and the mark cleared, as by
 * vs_device_status) when a product kernel's bounded wait gave up.
 */
vs_status vs_spmm_host(vs_handle A, const vs_dense *B_host, const vs_dense *out_host,
                       vs_direction dir, vs_variant variant, cudaStream_t stream);

/*
 * vs_attach_transpose -- builds the exact transpose of A from A's own arrays
 * and keeps it in the handle ("Regridder", "API": the exact transpose, kept
 * once built).  For VCSR that is the VCSC of the same matrix (and vice versa);
 * for CSR it is the CSC whose slices list entries in CSR order.  Afterwards
 * VS_TRANSPOSED runs misaligned directions as aligned gathers over it.
 * Synchronises `stream` once.  Idempotent.
 */
vs_status vs_attach_transpose(vs_handle A, cudaStream_t stream);

/*
 * vs_transpose -- a new handle holding the exact transpose of A as a matrix of
 * its own ("Regridder", "API": .T, the exact transpose): same layout and
 * dtype, the other major axis, shape n_cols x n_rows seen from the caller as
 * the transpose (its rows are A's columns).  For CSR, slice j of the result
 * lists the entries of A's column j in A's storage order.  The new handle
 * owns its arrays; A is unchanged.  Synchronises `stream` once.
 *   out   receives the handle (NULL on error); release with vs_destroy
 */
vs_status vs_transpose(vs_handle A, cudaStream_t stream, vs_handle *out);

/*
 * vs_scale_entries -- the hook of the conservative transpose ("Regridder",
 * "API": it scales each entry of the exact transpose by a factor of its own
 * and shares the indices of .T).  Returns a new CSR handle with A's sparsity
 * pattern whose stored value e is A's value e times factors[e], rounded once
 * in A's dtype.  The index arrays and kernel metadata are shared with A (not
 * copied) and stay valid until both handles are destroyed; the new handle
 * owns its values and scratch.  The factors themselves (cell sizes) are the
 * caller's.
 *   factors  device array of nnz values of A's dtype, in A's storage order
 *            (the order of vs_export's values); caller-owned, read before the
 *            call's work on `stream` completes
 *   out      receives the handle (NULL on error); release with vs_destroy
 * Errors: VS_ERR_LAYOUT for a VCS handle (a per-entry factor would split its
 * runs, so no index array could be shared); VS_ERR_INVALID for NULL factors
 * with nnz > 0.
 */
vs_status vs_scale_entries(vs_handle A, const void *factors, cudaStream_t stream,
                           vs_handle *out);

/*
 * vs_force_group_size -- test hook for the group size ("Regridder", "Tests":
 * every group size from 1 to 32 must reproduce the dense product).  From this
 * call on, the gathers over A, and over its exact transpose (attached now or
 * later), give every slice g logical partial sums instead of the g that the
 * matrix rule picks (the largest power of two <= the mean entries per slice,
 * at most 32).  The summation order then follows the forced g: results stay
 * within the tolerance of the exact product, repeat bit for bit, and give a
 * column the same bits alone or in a batch, but their last bits may differ
 * from those under the rule.  g = 0 restores the rule.  Host-side only:
 * call it between products, not while another host thread runs one on A.
 *   g  0, 1, 2, 4, 8, 16 or 32 (VS_ERR_INVALID otherwise)
 */
vs_status vs_force_group_size(vs_handle A, int32_t g);

/* vs_info -- shape, layout and matrix-only kernel parameters of A. */
vs_status vs_info(vs_handle A, vs_info_t *info);

/* vs_export -- read-only device pointers to A's layout arrays (owned by A,
 * valid until vs_destroy). */
vs_status vs_export(vs_handle A, vs_arrays *arrays);

/*
 * vs_handle_bytes -- device bytes held by A: `layout_bytes` counts the layout
 * arrays only (for VCS: major_ptr, values, value_ptr, indices -- no per-nonzero
 * value array exists), `scratch_bytes` counts everything else (chunk tables,
 * partial-sum scratch, staging, an attached transpose).  Either may be NULL.
 */
vs_status vs_handle_bytes(vs_handle A, int64_t *layout_bytes, int64_t *scratch_bytes);

/* vs_destroy -- frees everything A owns.  Synchronises the device first, so
 * work still queued on A finishes before its memory is released.  NULL is OK. */
vs_status vs_destroy(vs_handle A);

/* Static text for a status code. */
const char *vs_status_string(vs_status s);

/* Message of the calling thread's last failed call ("" if none). */
const char *vs_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t vs_version(void);

/* Number of kernels libvs has launched in this process so far (all devices,
 * all handles); a benchmark reads it before and after a timed region. */
int64_t vs_kernel_launches(void);

/*
 * vs_device_status -- synchronises `stream` and reports whether a product
 * kernel on A gave up a bounded wait (every mbarrier wait of the kernels ends
 * after about a second; the kernel then marks the handle, lets its own copies
 * land and exits, leaving its output invalid and the context usable).
 * Returns VS_ERR_TIMEOUT once per such event (the mark is cleared), else
 * VS_OK.  vs_spmm_host calls it before returning.
 */
vs_status vs_device_status(vs_handle A, cudaStream_t stream);

/*
 * vs_test_stall_producers -- test hook for the failure path above: the next
 * `launches` gather launches (process-wide) run with a producer that issues
 * nothing, so their consumers' waits run out and the handle is marked.
 * Nothing faults or hangs; each such launch takes about a second.  0 cancels.
 */
void vs_test_stall_producers(int launches);

/*
 * vs_gather_floor -- a measurement, not a product: the memory-side floor of
 * the gather that vs_spmm(A, B, dir, VS_DETERMINISTIC) runs.  One kernel
 * reads every stored index of the matrix that product walks (the attached
 * transpose for a misaligned direction, when there is one) in storage order,
 * loads the row of B it names through L1 with 16-byte loads and adds the rows
 * into registers; no values, no summation tree, no pipeline, no output rows.
 * Its time is what fetching the operand rows alone costs for this matrix's
 * index stream, the second roof beside HBM.  The sums go to handle scratch.
 * Needs a float32 B whose width is a multiple of 4 and at most 64, with the
 * layout rules of vs_spmm, and for a misaligned direction an attached
 * transpose (VS_ERR_UNSUPPORTED otherwise).
 */
vs_status vs_gather_floor(vs_handle A, const vs_dense *B, vs_direction dir, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VS_H */
