/*
 * vs_oracle.c -- the float64 CPU oracle for sparse x dense products over
 * CSR and the value-grouped VCS layout.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library: every function below is
 * written from the definitions on the pages, plainly and slowly, so that a
 * reader can check it against them by eye.
 *
 * Sources (page title, section):
 *  - "Add CUDA transfer and matmul kernels for the normalized views"
 *    (vsparse PR #61), section "The layout stays compressed": a VCS matrix is
 *    major_ptr -> (values, value_ptr) -> indices; each major slice's nonzeros
 *    are grouped into runs that share one value.
 *  - "Regridder" (regridding PR #70), section "How it is built": assembly is a
 *    counting sort -- one pass counts each row's entries, the next places
 *    them at the rows' cursors, and a row keeps its entries in element order.
 *  - The products are the plain definitions out = A.B and out = B.A.
 *
 * Readings where the pages are open (each is also listed with the design notes):
 *  - VCS run order inside a slice: ascending value, using the IEEE total
 *    order of the float32 bit patterns (so -0.0 and +0.0 are distinct runs);
 *    one run per distinct value.  Indices inside a run: ascending minor
 *    index; exact duplicates keep input order.  NaN values are rejected.
 *  - Explicit zeros and duplicate (i, j) entries are kept as given; products
 *    sum duplicates.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused and the
 * results are the same on every host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_RANGE (-1)
#define OR_ERR_NAN (-2)
#define OR_ERR_ALLOC (-3)
#define OR_ERR_ARG (-4)

/* ------------------------------------------------------------------------ */
/* CSR assembly by counting sort ("Regridder", "How it is built").           */
/* ------------------------------------------------------------------------ */

/*
 * Entries t = 0..nnz-1 are (maj[t], mnr[t], val[t]); val is an opaque record
 * of val_bytes bytes that is moved, never interpreted.  Output: ptr[n_major+1],
 * idx[nnz], vals_out[nnz records].  Returns 0, or OR_ERR_RANGE if an index
 * lies outside [0, n_major) x [0, n_minor).
 */
int or_csr_build(int64_t n_major, int64_t n_minor, int64_t nnz,
                 const int32_t *maj, const int32_t *mnr,
                 const void *val, int64_t val_bytes,
                 int32_t *ptr, int32_t *idx, void *vals_out)
{
    if (n_major < 0 || n_minor < 0 || nnz < 0 || val_bytes < 0) return OR_ERR_ARG;
    for (int64_t t = 0; t < nnz; t++) {
        if (maj[t] < 0 || maj[t] >= n_major || mnr[t] < 0 || mnr[t] >= n_minor)
            return OR_ERR_RANGE;
    }
    /* pass 1: count the entries of each major slice */
    int64_t *count = (int64_t *)calloc((size_t)n_major + 1, sizeof(int64_t));
    if (!count) return OR_ERR_ALLOC;
    for (int64_t t = 0; t < nnz; t++) count[maj[t]] += 1;
    /* exclusive scan of the counts gives the slice starts */
    int64_t running = 0;
    for (int64_t m = 0; m < n_major; m++) {
        ptr[m] = (int32_t)running;
        running += count[m];
    }
    ptr[n_major] = (int32_t)running;
    /* pass 2: place each entry, in input order, at its slice's cursor */
    for (int64_t m = 0; m < n_major; m++) count[m] = ptr[m]; /* cursors */
    const unsigned char *src = (const unsigned char *)val;
    unsigned char *dst = (unsigned char *)vals_out;
    for (int64_t t = 0; t < nnz; t++) {
        int64_t p = count[maj[t]];
        count[maj[t]] = p + 1;
        idx[p] = mnr[t];
        if (val_bytes > 0) memcpy(dst + p * val_bytes, src + t * val_bytes, (size_t)val_bytes);
    }
    free(count);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* VCS assembly ("Add CUDA transfer and matmul kernels ...", "The layout     */
/* stays compressed").                                                       */
/* ------------------------------------------------------------------------ */

/* The IEEE-754 total order of a float32, as an unsigned key: negative values
 * have every bit flipped, non-negative values have the sign bit set. */
static uint32_t float_order_key(float f)
{
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    if (b & 0x80000000u) return ~b;
    return b | 0x80000000u;
}

typedef struct {
    int32_t maj;
    uint32_t vkey;
    int32_t mnr;
    int64_t t; /* input position: makes the order total, hence stable */
    float v;
} or_entry;

static int cmp_entry(const void *pa, const void *pb)
{
    const or_entry *a = (const or_entry *)pa, *b = (const or_entry *)pb;
    if (a->maj != b->maj) return a->maj < b->maj ? -1 : 1;
    if (a->vkey != b->vkey) return a->vkey < b->vkey ? -1 : 1;
    if (a->mnr != b->mnr) return a->mnr < b->mnr ? -1 : 1;
    if (a->t != b->t) return a->t < b->t ? -1 : 1;
    return 0;
}

/*
 * Builds the VCS arrays of the entries (maj, mnr, val):
 *   major_ptr[n_major+1]  run range of each major slice,
 *   values[R]             the value each run shares,
 *   value_ptr[R+1]        index range of each run,
 *   indices[nnz]          minor indices, run by run.
 * values/value_ptr must have room for nnz (resp. nnz+1) entries, since R <= nnz.
 * Returns R >= 0, or a negative error code.
 */
int64_t or_vcs_build(int64_t n_major, int64_t n_minor, int64_t nnz,
                     const int32_t *maj, const int32_t *mnr, const float *val,
                     int32_t *major_ptr, float *values, int32_t *value_ptr, int32_t *indices)
{
    if (n_major < 0 || n_minor < 0 || nnz < 0) return OR_ERR_ARG;
    for (int64_t t = 0; t < nnz; t++) {
        if (maj[t] < 0 || maj[t] >= n_major || mnr[t] < 0 || mnr[t] >= n_minor)
            return OR_ERR_RANGE;
        if (isnan(val[t])) return OR_ERR_NAN;
    }
    or_entry *e = (or_entry *)malloc(sizeof(or_entry) * (size_t)(nnz > 0 ? nnz : 1));
    if (!e) return OR_ERR_ALLOC;
    for (int64_t t = 0; t < nnz; t++) {
        e[t].maj = maj[t];
        e[t].vkey = float_order_key(val[t]);
        e[t].mnr = mnr[t];
        e[t].t = t;
        e[t].v = val[t];
    }
    qsort(e, (size_t)nnz, sizeof(or_entry), cmp_entry);

    /* a run starts wherever (major, value) changes */
    int64_t R = 0;
    int64_t *runs_of = (int64_t *)calloc((size_t)n_major + 1, sizeof(int64_t));
    if (!runs_of) { free(e); return OR_ERR_ALLOC; }
    for (int64_t k = 0; k < nnz; k++) {
        int new_run = (k == 0) || e[k].maj != e[k - 1].maj || e[k].vkey != e[k - 1].vkey;
        if (new_run) {
            value_ptr[R] = (int32_t)k;
            values[R] = e[k].v;
            runs_of[e[k].maj] += 1;
            R++;
        }
        indices[k] = e[k].mnr;
    }
    value_ptr[R] = (int32_t)nnz;
    int64_t running = 0;
    for (int64_t m = 0; m < n_major; m++) {
        major_ptr[m] = (int32_t)running;
        running += runs_of[m];
    }
    major_ptr[n_major] = (int32_t)running;
    free(runs_of);
    free(e);
    return R;
}

/* ------------------------------------------------------------------------ */
/* Expansion of a layout back to (row, col, value) triples, in layout order. */
/* ------------------------------------------------------------------------ */

/* CSR (major_is_row = 1) or CSC (major_is_row = 0) with float64 values. */
void or_csr_triples(int64_t n_major, int major_is_row, const int32_t *ptr, const int32_t *idx,
                    const double *vals, int32_t *ti, int32_t *tj, double *ta)
{
    for (int64_t m = 0; m < n_major; m++) {
        for (int64_t k = ptr[m]; k < ptr[m + 1]; k++) {
            ti[k] = major_is_row ? (int32_t)m : idx[k];
            tj[k] = major_is_row ? idx[k] : (int32_t)m;
            ta[k] = vals[k];
        }
    }
}

/* VCSR (major_is_row = 1) or VCSC (major_is_row = 0): every index of run r
 * carries values[r]. */
void or_vcs_triples(int64_t n_major, int major_is_row, const int32_t *major_ptr,
                    const float *values, const int32_t *value_ptr, const int32_t *indices,
                    int32_t *ti, int32_t *tj, double *ta)
{
    for (int64_t m = 0; m < n_major; m++) {
        for (int64_t r = major_ptr[m]; r < major_ptr[m + 1]; r++) {
            for (int64_t k = value_ptr[r]; k < value_ptr[r + 1]; k++) {
                ti[k] = major_is_row ? (int32_t)m : indices[k];
                tj[k] = major_is_row ? indices[k] : (int32_t)m;
                ta[k] = (double)values[r];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Products: the plain definitions, in float64, over the triples of A.       */
/* D receives sum |a| |b| of every output element (the error scale).         */
/* ------------------------------------------------------------------------ */

/* out = A B.  A: n_rows x n_cols as triples.  B: n_cols x w, row stride ldb.
 * out, D: n_rows x w, row stride ldo. */
void or_spmm_ab(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *ti,
                const int32_t *tj, const double *ta, const double *B, int64_t ldb,
                int64_t w, double *out, double *D, int64_t ldo)
{
    (void)n_cols;
    for (int64_t i = 0; i < n_rows; i++)
        for (int64_t c = 0; c < w; c++) { out[i * ldo + c] = 0.0; D[i * ldo + c] = 0.0; }
    for (int64_t k = 0; k < nnz; k++) {
        int64_t i = ti[k], j = tj[k];
        double a = ta[k];
        for (int64_t c = 0; c < w; c++) {
            double b = B[j * ldb + c];
            out[i * ldo + c] += a * b;
            D[i * ldo + c] += fabs(a) * fabs(b);
        }
    }
}

/* out = B A.  B: w x n_rows, row stride ldb.  out, D: w x n_cols, row stride ldo. */
void or_spmm_ba(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *ti,
                const int32_t *tj, const double *ta, const double *B, int64_t ldb,
                int64_t w, double *out, double *D, int64_t ldo)
{
    (void)n_rows;
    for (int64_t c = 0; c < w; c++)
        for (int64_t j = 0; j < n_cols; j++) { out[c * ldo + j] = 0.0; D[c * ldo + j] = 0.0; }
    for (int64_t k = 0; k < nnz; k++) {
        int64_t i = ti[k], j = tj[k];
        double a = ta[k];
        for (int64_t c = 0; c < w; c++) {
            double b = B[c * ldb + i];
            out[c * ldo + j] += b * a;
            D[c * ldo + j] += fabs(b) * fabs(a);
        }
    }
}

/*
 * Sampled products for matrices too large for a full product: only the
 * output rows (A B) or output columns (B A) listed in `sel` are computed.
 *   or_spmm_ab_rows: out[s, c] = sum over triples with ti == sel[s] of a B[tj, c]
 *                    B: n_cols x w (ldb); out, D: n_sel x w, contiguous.
 *   or_spmm_ba_cols: out[s, c] = sum over triples with tj == sel[s] of B[c, ti] a
 *                    B: w x n_rows (ldb); out, D: n_sel x w, contiguous
 *                    (row s holds output column sel[s]).
 * `slot` is caller scratch of n_out int64 (n_rows resp. n_cols).
 */
void or_spmm_ab_rows(int64_t n_rows, int64_t nnz, const int32_t *ti, const int32_t *tj,
                     const double *ta, const double *B, int64_t ldb, int64_t w,
                     int64_t n_sel, const int64_t *sel, int64_t *slot, double *out, double *D)
{
    for (int64_t i = 0; i < n_rows; i++) slot[i] = -1;
    for (int64_t s = 0; s < n_sel; s++) slot[sel[s]] = s;
    for (int64_t s = 0; s < n_sel * w; s++) { out[s] = 0.0; D[s] = 0.0; }
    for (int64_t k = 0; k < nnz; k++) {
        int64_t s = slot[ti[k]];
        if (s < 0) continue;
        int64_t j = tj[k];
        double a = ta[k];
        for (int64_t c = 0; c < w; c++) {
            double b = B[j * ldb + c];
            out[s * w + c] += a * b;
            D[s * w + c] += fabs(a) * fabs(b);
        }
    }
}

void or_spmm_ba_cols(int64_t n_cols, int64_t nnz, const int32_t *ti, const int32_t *tj,
                     const double *ta, const double *B, int64_t ldb, int64_t w,
                     int64_t n_sel, const int64_t *sel, int64_t *slot, double *out, double *D)
{
    for (int64_t j = 0; j < n_cols; j++) slot[j] = -1;
    for (int64_t s = 0; s < n_sel; s++) slot[sel[s]] = s;
    for (int64_t s = 0; s < n_sel * w; s++) { out[s] = 0.0; D[s] = 0.0; }
    for (int64_t k = 0; k < nnz; k++) {
        int64_t s = slot[tj[k]];
        if (s < 0) continue;
        int64_t i = ti[k];
        double a = ta[k];
        for (int64_t c = 0; c < w; c++) {
            double b = B[c * ldb + i];
            out[s * w + c] += b * a;
            D[s * w + c] += fabs(b) * fabs(a);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Normalized views ("Add CUDA transfer and matmul kernels for the           */
/* normalized views", "The layout stays compressed": a view applies a value  */
/* transform and carries per-row and per-column statistics).  The view of A  */
/* is V = diag(row_scale) . g(A) . diag(col_scale): entry (i, j, a) of A     */
/* becomes (i, j, row_scale[i] * g(a) * col_scale[j]).                       */
/*   map 0: g(a) = a;  map 1: g(a) = log(1 + a);  map 2: g(a) = sqrt(a).     */
/* row_scale / col_scale may be NULL (all ones).  Returns OR_ERR_ARG for an  */
/* unknown map.                                                              */
/* ------------------------------------------------------------------------ */
int or_view_triples(int64_t nnz, const int32_t *ti, const int32_t *tj, const double *ta,
                    int map, const double *row_scale, const double *col_scale, double *out)
{
    if (map < 0 || map > 2) return OR_ERR_ARG;
    for (int64_t k = 0; k < nnz; k++) {
        double v = ta[k];
        if (map == 1) v = log1p(v);
        if (map == 2) v = sqrt(v);
        if (row_scale) v = row_scale[ti[k]] * v;
        if (col_scale) v = v * col_scale[tj[k]];
        out[k] = v;
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* The same products over a stored layout, on several host threads (the     */
/* pages' host kernels: "Add CUDA transfer and matmul kernels ...", "The     */
/* kernels" -- aligned directions take whole slices per thread, misaligned   */
/* ones accumulate into per-thread private outputs that are then merged).    */
/*                                                                          */
/* Slice frame: a slice s is a stored major index; its entries (t, a) carry  */
/* the minor index t.  `ptr` gives each slice's entry range (CSR), or its    */
/* run range when `vptr` is given (VCS: run r holds entries vptr[r] ..       */
/* vptr[r+1]-1, all with value vals[r]; otherwise vals[k] is entry k's).     */
/*   aligned = 1:  Y[s, :] = sum over entries (t, a) of s of a * X[t, :]     */
/*                 (X: n_minor x w, Y: n_major x w)                          */
/*   aligned = 0:  Y[t, :] = sum over slices s, entries (t, a) of a * X[s, :] */
/*                 (X: n_major x w, Y: n_minor x w)                          */
/* Both row-major with row stride w.  D receives sum |a| |x| per element.    */
/* Aligned: each output row is summed in entry order by one thread, exactly  */
/* as the serial products above add it.  Misaligned: thread k of T takes the */
/* consecutive slices whose first entry lies in [nnz k / T, nnz (k+1) / T)   */
/* into a private Y_k (whole slices, balanced by entries); then              */
/* Y = Y_0 + Y_1 + ... in thread order, so the result depends on T only.     */
/* n_threads <= 0 means every thread OpenMP offers.  Returns OR_ERR_ALLOC    */
/* when the private outputs cannot be allocated.                             */
/* ------------------------------------------------------------------------ */
int or_threads_available(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* First entry of slice s, and the entry count. */
static int64_t slice_entry(const int32_t *ptr, const int32_t *vptr, int64_t s)
{
    return vptr ? vptr[ptr[s]] : ptr[s];
}

static int64_t nnz_of(int64_t n_major, const int32_t *ptr, const int32_t *vptr)
{
    return slice_entry(ptr, vptr, n_major);
}

/* The first slice s whose first entry is >= e (n_major if none). */
static int64_t first_slice_at(int64_t n_major, const int32_t *ptr, const int32_t *vptr, int64_t e)
{
    int64_t lo = 0, hi = n_major;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (slice_entry(ptr, vptr, mid) < e) lo = mid + 1; else hi = mid;
    }
    return lo;
}

int or_spmm_slices(int64_t n_major, int64_t n_minor, const int32_t *ptr, const int32_t *vptr,
                   const int32_t *idx, const double *vals, int aligned, const double *X,
                   int64_t w, double *Y, double *D, int n_threads)
{
    if (n_major < 0 || n_minor < 0 || w < 0) return OR_ERR_ARG;
    int T = n_threads > 0 ? n_threads : or_threads_available();
    if (T < 1) T = 1;
    if (aligned) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64) num_threads(T)
#endif
        for (int64_t s = 0; s < n_major; s++) {
            double *y = Y + s * w, *d = D + s * w;
            for (int64_t c = 0; c < w; c++) { y[c] = 0.0; d[c] = 0.0; }
            int64_t lo = ptr[s], hi = ptr[s + 1];
            for (int64_t q = lo; q < hi; q++) {
                /* CSR: q is an entry; VCS: q is a run covering vptr[q] .. vptr[q+1]-1 */
                int64_t k0 = vptr ? vptr[q] : q, k1 = vptr ? vptr[q + 1] : q + 1;
                double a = vals[q];
                for (int64_t k = k0; k < k1; k++) {
                    const double *x = X + (int64_t)idx[k] * w;
                    for (int64_t c = 0; c < w; c++) {
                        y[c] += a * x[c];
                        d[c] += fabs(a) * fabs(x[c]);
                    }
                }
            }
        }
        return OR_OK;
    }
    /* misaligned: private outputs per thread, merged in thread order */
    size_t per = (size_t)(n_minor > 0 ? n_minor : 1) * (size_t)(w > 0 ? w : 1);
    double *priv = (double *)calloc((size_t)T * per * 2, sizeof(double));
    if (!priv) return OR_ERR_ALLOC;
#ifdef _OPENMP
#pragma omp parallel for schedule(static, 1) num_threads(T)
#endif
    for (int k = 0; k < T; k++) {
        double *y = priv + (size_t)k * per * 2, *d = y + per;
        int64_t s0 = first_slice_at(n_major, ptr, vptr, nnz_of(n_major, ptr, vptr) * k / T);
        int64_t s1 = first_slice_at(n_major, ptr, vptr, nnz_of(n_major, ptr, vptr) * (k + 1) / T);
        if (k == T - 1) s1 = n_major;
        for (int64_t s = s0; s < s1; s++) {
            const double *x = X + s * w;
            for (int64_t q = ptr[s]; q < ptr[s + 1]; q++) {
                int64_t k0 = vptr ? vptr[q] : q, k1 = vptr ? vptr[q + 1] : q + 1;
                double a = vals[q];
                for (int64_t e = k0; e < k1; e++) {
                    double *yt = y + (int64_t)idx[e] * w, *dt = d + (int64_t)idx[e] * w;
                    for (int64_t c = 0; c < w; c++) {
                        yt[c] += a * x[c];
                        dt[c] += fabs(a) * fabs(x[c]);
                    }
                }
            }
        }
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(T)
#endif
    for (int64_t t = 0; t < n_minor; t++) {
        for (int64_t c = 0; c < w; c++) {
            double ys = 0.0, ds = 0.0;
            for (int k = 0; k < T; k++) {
                const double *y = priv + (size_t)k * per * 2;
                ys += y[t * w + c];
                ds += y[per + t * w + c];
            }
            Y[t * w + c] = ys;
            D[t * w + c] = ds;
        }
    }
    free(priv);
    return OR_OK;
}
