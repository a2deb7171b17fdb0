// assembly.cu -- device construction of CSR/CSC and VCSR/VCSC from COO.
//
// "Regridder" (regridding PR #70), "How it is built": assembly is a counting
// sort.  One pass counts each slice's entries, an exclusive scan turns the
// counts into slice starts, and a placement pass puts every entry at its
// slice's cursor so that a slice keeps its entries in input order.
//
// The placement must be stable and bit-identical on every run, so it is done
// as an LSD radix sort of a permutation with 8-bit digits: each pass counts
// digits per tile of 2048 entries, scans the (digit, tile) counts, and scatters
// with ranks that follow input order inside a tile (warp match + per-warp
// digit counters, then a prefix over warps).  Every count is an integer, so
// the result does not depend on scheduling.  No kernel waits on another
// block: scans are reduce-then-scan with separate launches.
//
// VCS ("Add CUDA transfer and matmul kernels for the normalized views", "The
// layout stays compressed") sorts by the key (major, value, minor), LSD order:
// minor first, then the value's total-order bits, then major.  Passes whose
// bits never vary, or whose order the input already has, are skipped.
#include <algorithm>
#include <vector>

#include "device_utils.cuh"
#include "vs_internal.h"

namespace vs {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;  // 2048 entries per tile

// ------------------------------------------------------------------ temporaries

// Stream-ordered temporary device memory, released when it goes out of scope.
struct Temp {
  void *p = nullptr;
  cudaStream_t s;
  explicit Temp(cudaStream_t st) : s(st) {}
  vs_status alloc(size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMallocAsync(&p, bytes, s);
    if (e != cudaSuccess) {
      p = nullptr;
      return cuda_status(e, "cudaMallocAsync (assembly temporary)");
    }
    return VS_OK;
  }
  ~Temp() {
    if (p) cudaFreeAsync(p, s);
  }
  template <typename T>
  T *as() const {
    return static_cast<T *>(p);
  }
};

}  // namespace

vs_status dev_alloc(void **p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    *p = nullptr;
    return e == cudaErrorMemoryAllocation ? (set_error("device allocation failed"), VS_ERR_ALLOC)
                                          : cuda_status(e, "cudaMalloc");
  }
  return VS_OK;
}

namespace {

inline unsigned grid_for(int64_t n, int per_block) {
  return (unsigned)std::max<int64_t>(1, (n + per_block - 1) / per_block);
}

inline int bit_length(uint64_t x) {
  int b = 0;
  while (x) {
    ++b;
    x >>= 1;
  }
  return b;
}

// ------------------------------------------------------------------ scan

// sums[b] = sum of in[b*kTile .. (b+1)*kTile)
__global__ void scan_reduce_kernel(const int32_t *__restrict__ in, int64_t n,
                                   int32_t *__restrict__ sums) {
  const int64_t base = (int64_t)blockIdx.x * kTile;
  int local = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    int64_t i = base + k * kThreads + threadIdx.x;
    if (i < n) local += in[i];
  }
  int total;
  block_exclusive_scan<kThreads>(local, total);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// out[i] = offsets[b] + exclusive prefix of in inside tile b; out[n] = grand total.
__global__ void scan_apply_kernel(const int32_t *__restrict__ in, int64_t n,
                                  const int32_t *__restrict__ offsets, int32_t *__restrict__ out) {
  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
  int v[kItems];
  int local = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    int64_t i = base + k;
    v[k] = i < n ? in[i] : 0;
    local += v[k];
  }
  int total;
  int run = block_exclusive_scan<kThreads>(local, total) + (offsets ? offsets[blockIdx.x] : 0);
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    int64_t i = base + k;
    if (i < n) out[i] = run;
    run += v[k];
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == kThreads - 1) out[n] = run;
}

// Exclusive scan of in[0..n) into out[0..n], out[n] = total.  Integer-exact.
vs_status exclusive_scan(const int32_t *in, int32_t *out, int64_t n, cudaStream_t s) {
  const int64_t nb = (n + kTile - 1) / kTile;
  if (nb <= 1) {
    scan_apply_kernel<<<1, kThreads, 0, s>>>(in, n, nullptr, out);
    VS_LAUNCH_CHECK();
    return VS_OK;
  }
  Temp sums(s), offs(s);
  VS_TRY(sums.alloc(sizeof(int32_t) * nb));
  VS_TRY(offs.alloc(sizeof(int32_t) * (nb + 1)));
  scan_reduce_kernel<<<(unsigned)nb, kThreads, 0, s>>>(in, n, sums.as<int32_t>());
  VS_LAUNCH_CHECK();
  VS_TRY(exclusive_scan(sums.as<int32_t>(), offs.as<int32_t>(), nb, s));
  scan_apply_kernel<<<(unsigned)nb, kThreads, 0, s>>>(in, n, offs.as<int32_t>(), out);
  VS_LAUNCH_CHECK();
  return VS_OK;
}

// ------------------------------------------------------------------ radix sort of a permutation

__device__ __forceinline__ int digit_of(const int32_t *perm, const uint32_t *key, int64_t i,
                                        int shift) {
  int64_t e = perm ? perm[i] : i;
  return (int)((key[e] >> shift) & 0xFFu);
}

__global__ void radix_hist_kernel(const int32_t *__restrict__ perm, const uint32_t *__restrict__ key,
                                  int64_t n, int shift, int32_t *__restrict__ hist, int64_t ntiles) {
  __shared__ int h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kTile;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    int64_t i = base + k * kThreads + threadIdx.x;
    if (i < n) atomicAdd(&h[digit_of(perm, key, i, shift)], 1);
  }
  __syncthreads();
  hist[(int64_t)threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter: inside a tile, warp w owns entries [w*256, (w+1)*256) and
// walks them 32 at a time in order; equal digits are ranked by lane order.
__global__ void radix_scatter_kernel(const int32_t *__restrict__ perm_in,
                                     const uint32_t *__restrict__ key, int64_t n, int shift,
                                     const int32_t *__restrict__ offsets, int64_t ntiles,
                                     int32_t *__restrict__ perm_out) {
  __shared__ int wcount[kThreads / 32][256];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int d = threadIdx.x; d < (kThreads / 32) * 256; d += kThreads) (&wcount[0][0])[d] = 0;
  __syncthreads();
  int dig[kItems], rank[kItems], elem[kItems];
  const int64_t wbase = (int64_t)blockIdx.x * kTile + (int64_t)w * (kItems * 32);
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const int64_t i = wbase + it * 32 + lane;
    const bool valid = i < n;
    const int e = valid ? (perm_in ? perm_in[i] : (int)i) : -1;
    const int d = valid ? (int)((key[e] >> shift) & 0xFFu) : 256;
    const unsigned peers = __match_any_sync(kFullMask, d);
    const int before = __popc(peers & lt);
    const int base = valid ? wcount[w][d] : 0;
    __syncwarp();
    if (valid && before == 0) wcount[w][d] = base + __popc(peers);
    __syncwarp();
    dig[it] = d;
    rank[it] = base + before;
    elem[it] = e;
  }
  __syncthreads();
  {  // exclusive prefix over warps, per digit (thread = digit)
    const int d = threadIdx.x;
    int run = 0;
#pragma unroll
    for (int ww = 0; ww < kThreads / 32; ++ww) {
      int c = wcount[ww][d];
      wcount[ww][d] = run;
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    if (dig[it] < 256) {
      const int64_t pos =
          (int64_t)offsets[(int64_t)dig[it] * ntiles + blockIdx.x] + wcount[w][dig[it]] + rank[it];
      perm_out[pos] = elem[it];
    }
  }
}

// Sorts the permutation *perm (nullptr = identity) stably by key bits
// [bit_lo, bit_hi) in 8-bit digits.  buf0/buf1 are int32[n] ping-pong buffers;
// on return *perm points at the one holding the result.
vs_status radix_passes(const int32_t **perm, const uint32_t *key, int64_t n, int bit_lo,
                       int bit_hi, int32_t *buf0, int32_t *buf1, cudaStream_t s) {
  if (bit_hi <= bit_lo || n <= 1) return VS_OK;
  const int64_t ntiles = (n + kTile - 1) / kTile;
  Temp hist(s), offs(s);
  VS_TRY(hist.alloc(sizeof(int32_t) * 256 * ntiles));
  VS_TRY(offs.alloc(sizeof(int32_t) * (256 * ntiles + 1)));
  for (int shift = bit_lo; shift < bit_hi; shift += 8) {
    int32_t *dst = (*perm == buf0) ? buf1 : buf0;
    radix_hist_kernel<<<(unsigned)ntiles, kThreads, 0, s>>>(*perm, key, n, shift,
                                                            hist.as<int32_t>(), ntiles);
    VS_LAUNCH_CHECK();
    VS_TRY(exclusive_scan(hist.as<int32_t>(), offs.as<int32_t>(), 256 * ntiles, s));
    radix_scatter_kernel<<<(unsigned)ntiles, kThreads, 0, s>>>(*perm, key, n, shift,
                                                               offs.as<int32_t>(), ntiles, dst);
    VS_LAUNCH_CHECK();
    *perm = dst;
  }
  return VS_OK;
}

// ------------------------------------------------------------------ checks and keys

struct Checks {
  int range_error;     // a coordinate outside the matrix
  int nan_error;       // a NaN value (VCS only)
  int major_unsorted;  // major[t] < major[t-1] somewhere
  int minor_unsorted;  // minor[t] < minor[t-1] somewhere
  int lex_unsorted;    // (major, minor)[t] < (major, minor)[t-1] somewhere
  unsigned key_or;     // OR of the value keys
  unsigned key_and;    // AND of the value keys
  int pad;
};

// Total-order key of a float32: negative values flip every bit, others set the sign bit.
__device__ __forceinline__ uint32_t order_key(uint32_t b) {
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void check_kernel(const int32_t *__restrict__ maj, const int32_t *__restrict__ mnr,
                             const float *__restrict__ val, int64_t nnz, int64_t n_major,
                             int64_t n_minor, uint32_t *__restrict__ vkey, Checks *out) {
  int range = 0, nan = 0, mu = 0, nu = 0, lu = 0;
  unsigned kor = 0, kand = 0xffffffffu;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nnz;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int a = maj[t], b = mnr[t];
    if (a < 0 || a >= n_major || b < 0 || b >= n_minor) range = 1;
    if (t > 0) {
      const int pa = maj[t - 1], pb = mnr[t - 1];
      if (a < pa) mu = 1;
      if (b < pb) nu = 1;
      if (a < pa || (a == pa && b < pb)) lu = 1;
    }
    if (val) {
      const uint32_t bits = __float_as_uint(val[t]);
      if ((bits & 0x7fffffffu) > 0x7f800000u) nan = 1;
      const uint32_t k = order_key(bits);
      vkey[t] = k;
      kor |= k;
      kand &= k;
    }
  }
  range = __syncthreads_or(range);
  nan = __syncthreads_or(nan);
  mu = __syncthreads_or(mu);
  nu = __syncthreads_or(nu);
  lu = __syncthreads_or(lu);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    kor |= __shfl_xor_sync(kFullMask, kor, d);
    kand &= __shfl_xor_sync(kFullMask, kand, d);
  }
  if (threadIdx.x == 0) {
    if (range) atomicOr(&out->range_error, 1);
    if (nan) atomicOr(&out->nan_error, 1);
    if (mu) atomicOr(&out->major_unsorted, 1);
    if (nu) atomicOr(&out->minor_unsorted, 1);
    if (lu) atomicOr(&out->lex_unsorted, 1);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicOr(&out->key_or, kor);
    atomicAnd(&out->key_and, kand);
  }
}

__global__ void copy_key_kernel(const int32_t *__restrict__ src, uint32_t *__restrict__ dst,
                                int64_t n) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x)
    dst[t] = (uint32_t)src[t];
}

__global__ void count_kernel(const int32_t *__restrict__ maj, int64_t n, int32_t *__restrict__ cnt) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x)
    atomicAdd(&cnt[maj[t]], 1);
}

// dst_idx[i] = mnr[perm[i]]; dst_val[i] = val[perm[i]] (raw `words` 32-bit words each).
__global__ void gather_entries_kernel(const int32_t *__restrict__ perm,
                                      const int32_t *__restrict__ mnr,
                                      const uint32_t *__restrict__ val, int words, int64_t n,
                                      int32_t *__restrict__ dst_idx, uint32_t *__restrict__ dst_val) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = perm ? perm[i] : i;
    dst_idx[i] = mnr[e];
    if (dst_val)
      for (int k = 0; k < words; ++k) dst_val[i * words + k] = val[e * words + k];
  }
}

// Run starts of the sorted VCS entries: flag[i] = 1 where (major, value) changes.
__global__ void run_flag_kernel(const int32_t *__restrict__ perm, const int32_t *__restrict__ maj,
                                const uint32_t *__restrict__ vkey, int64_t n,
                                int32_t *__restrict__ flag) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = perm ? perm[i] : i;
    int f = 1;
    if (i > 0) {
      const int64_t p = perm ? perm[i - 1] : i - 1;
      f = (maj[e] != maj[p]) || (vkey[e] != vkey[p]);
    }
    flag[i] = f;
  }
}

__global__ void run_fill_kernel(const int32_t *__restrict__ perm, const int32_t *__restrict__ maj,
                                const float *__restrict__ val, const int32_t *__restrict__ flag,
                                const int32_t *__restrict__ run_id, int64_t n,
                                int32_t *__restrict__ vptr, float *__restrict__ values,
                                int32_t *__restrict__ runs_per_major) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (!flag[i]) continue;
    const int64_t e = perm ? perm[i] : i;
    const int r = run_id[i];
    vptr[r] = (int32_t)i;
    values[r] = val[e];
    atomicAdd(&runs_per_major[maj[e]], 1);
  }
}

__global__ void set_int_kernel(int32_t *p, int32_t v) { *p = v; }

constexpr unsigned kGridCap = 152 * 16;

}  // namespace

// ------------------------------------------------------------------ build_matrix

vs_status build_matrix(Matrix &m, vs_layout layout, vs_major major, vs_dtype dtype, int64_t n_rows,
                       int64_t n_cols, int64_t nnz, const int32_t *d_row, const int32_t *d_col,
                       const void *d_val, cudaStream_t s) {
  m.layout = layout;
  m.major = major;
  m.dtype = dtype;
  m.n_rows = n_rows;
  m.n_cols = n_cols;
  m.n_major = major == VS_MAJOR_ROW ? n_rows : n_cols;
  m.n_minor = major == VS_MAJOR_ROW ? n_cols : n_rows;
  m.nnz = nnz;
  const int32_t *maj = major == VS_MAJOR_ROW ? d_row : d_col;
  const int32_t *mnr = major == VS_MAJOR_ROW ? d_col : d_row;
  const bool vcs = layout == VS_LAYOUT_VCS;
  const size_t dsize = m.dsize();

  // ---- checks (and value keys for VCS)
  Temp checks(s), vkey(s);
  VS_TRY(checks.alloc(sizeof(Checks)));
  Checks init{};
  init.key_and = 0xffffffffu;
  VS_CUDA(cudaMemcpyAsync(checks.p, &init, sizeof init, cudaMemcpyHostToDevice, s));
  if (vcs) VS_TRY(vkey.alloc(sizeof(uint32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  if (nnz > 0) {
    check_kernel<<<std::min<unsigned>(kGridCap, grid_for(nnz, 256)), 256, 0, s>>>(
        maj, mnr, vcs ? static_cast<const float *>(d_val) : nullptr, nnz, m.n_major, m.n_minor,
        vkey.as<uint32_t>(), checks.as<Checks>());
    VS_LAUNCH_CHECK();
  }
  Checks ck{};
  VS_CUDA(cudaMemcpyAsync(&ck, checks.p, sizeof ck, cudaMemcpyDeviceToHost, s));
  VS_CUDA(cudaStreamSynchronize(s));
  if (ck.range_error) {
    set_error("a COO coordinate lies outside the matrix");
    return VS_ERR_RANGE;
  }
  if (ck.nan_error) {
    set_error("NaN value: VCS runs need an ordered value key");
    return VS_ERR_NAN;
  }

  // ---- the permutation that orders the entries
  Temp b0(s), b1(s), keybuf(s);
  VS_TRY(b0.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  VS_TRY(b1.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  VS_TRY(keybuf.alloc(sizeof(uint32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  const int32_t *perm = nullptr;  // identity
  const unsigned eg = std::min<unsigned>(kGridCap, grid_for(nnz, 256));
  if (vcs) {
    // minor first (unless the input already orders it), then value bits, then major
    if (ck.minor_unsorted && ck.lex_unsorted && nnz > 1) {
      copy_key_kernel<<<eg, 256, 0, s>>>(mnr, keybuf.as<uint32_t>(), nnz);
      VS_LAUNCH_CHECK();
      VS_TRY(radix_passes(&perm, keybuf.as<uint32_t>(), nnz, 0,
                          bit_length((uint64_t)std::max<int64_t>(m.n_minor - 1, 0)),
                          b0.as<int32_t>(), b1.as<int32_t>(), s));
    }
    const unsigned diff = ck.key_or ^ ck.key_and;
    if (diff && nnz > 1) {
      const int lo = __builtin_ctz(diff), hi = 32 - __builtin_clz(diff);
      VS_TRY(radix_passes(&perm, vkey.as<uint32_t>(), nnz, lo, hi, b0.as<int32_t>(),
                          b1.as<int32_t>(), s));
    }
    if (nnz > 1 && (ck.major_unsorted || diff || (ck.minor_unsorted && ck.lex_unsorted))) {
      copy_key_kernel<<<eg, 256, 0, s>>>(maj, keybuf.as<uint32_t>(), nnz);
      VS_LAUNCH_CHECK();
      VS_TRY(radix_passes(&perm, keybuf.as<uint32_t>(), nnz, 0,
                          bit_length((uint64_t)std::max<int64_t>(m.n_major - 1, 0)),
                          b0.as<int32_t>(), b1.as<int32_t>(), s));
    }
  } else if (ck.major_unsorted && nnz > 1) {
    copy_key_kernel<<<eg, 256, 0, s>>>(maj, keybuf.as<uint32_t>(), nnz);
    VS_LAUNCH_CHECK();
    VS_TRY(radix_passes(&perm, keybuf.as<uint32_t>(), nnz, 0,
                        bit_length((uint64_t)std::max<int64_t>(m.n_major - 1, 0)),
                        b0.as<int32_t>(), b1.as<int32_t>(), s));
  }

  // ---- owned arrays: slice pointer and indices (padded for vector over-reads)
  VS_TRY(dev_alloc((void **)&m.ptr, sizeof(int32_t) * (m.n_major + 1 + 16)));
  VS_CUDA(cudaMemsetAsync(m.ptr, 0, sizeof(int32_t) * (m.n_major + 1 + 16), s));
  VS_TRY(dev_alloc((void **)&m.idx, sizeof(int32_t) * (nnz + 16)));
  VS_CUDA(cudaMemsetAsync(m.idx, 0, sizeof(int32_t) * (nnz + 16), s));
  Temp cnt(s);
  VS_TRY(cnt.alloc(sizeof(int32_t) * (m.n_major + 1)));
  VS_CUDA(cudaMemsetAsync(cnt.p, 0, sizeof(int32_t) * (m.n_major + 1), s));

  if (!vcs) {
    VS_TRY(dev_alloc(&m.vals, dsize * (nnz + 16)));
    VS_CUDA(cudaMemsetAsync(m.vals, 0, dsize * (nnz + 16), s));
    if (nnz > 0) {
      gather_entries_kernel<<<eg, 256, 0, s>>>(perm, mnr, static_cast<const uint32_t *>(d_val),
                                               (int)(dsize / 4), nnz, m.idx,
                                               static_cast<uint32_t *>(m.vals));
      VS_LAUNCH_CHECK();
      count_kernel<<<eg, 256, 0, s>>>(maj, nnz, cnt.as<int32_t>());
      VS_LAUNCH_CHECK();
    }
    VS_TRY(exclusive_scan(cnt.as<int32_t>(), m.ptr, m.n_major, s));
    m.R = nnz;
    VS_CUDA(cudaStreamSynchronize(s));
    return VS_OK;
  }

  // ---- VCS: runs
  Temp flag(s), run_id(s);
  VS_TRY(flag.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  VS_TRY(run_id.alloc(sizeof(int32_t) * (nnz + 1)));
  int32_t R = 0;
  if (nnz > 0) {
    gather_entries_kernel<<<eg, 256, 0, s>>>(perm, mnr, nullptr, 0, nnz, m.idx, nullptr);
    VS_LAUNCH_CHECK();
    run_flag_kernel<<<eg, 256, 0, s>>>(perm, maj, vkey.as<uint32_t>(), nnz, flag.as<int32_t>());
    VS_LAUNCH_CHECK();
    VS_TRY(exclusive_scan(flag.as<int32_t>(), run_id.as<int32_t>(), nnz, s));
    VS_CUDA(cudaMemcpyAsync(&R, run_id.as<int32_t>() + nnz, sizeof R, cudaMemcpyDeviceToHost, s));
    VS_CUDA(cudaStreamSynchronize(s));
  }
  m.R = R;
  VS_TRY(dev_alloc(&m.vals, sizeof(float) * (R + 16)));
  VS_TRY(dev_alloc((void **)&m.vptr, sizeof(int32_t) * (R + 16)));
  VS_CUDA(cudaMemsetAsync(m.vals, 0, sizeof(float) * (R + 16), s));
  VS_CUDA(cudaMemsetAsync(m.vptr, 0, sizeof(int32_t) * (R + 16), s));
  if (nnz > 0) {
    run_fill_kernel<<<eg, 256, 0, s>>>(perm, maj, static_cast<const float *>(d_val),
                                       flag.as<int32_t>(), run_id.as<int32_t>(), nnz, m.vptr,
                                       static_cast<float *>(m.vals), cnt.as<int32_t>());
    VS_LAUNCH_CHECK();
  }
  set_int_kernel<<<1, 1, 0, s>>>(m.vptr + R, (int32_t)nnz);
  VS_LAUNCH_CHECK();
  VS_TRY(exclusive_scan(cnt.as<int32_t>(), m.ptr, m.n_major, s));
  VS_CUDA(cudaStreamSynchronize(s));
  return VS_OK;
}

// ------------------------------------------------------------------ wide matrices

namespace {

// flags[0]: a coordinate outside the matrix; flags[1]: a NaN value (VCS keys)
__global__ void wide_check_kernel(const int32_t *__restrict__ maj, const int32_t *__restrict__ mnr,
                                  const float *__restrict__ val, int64_t nnz, int64_t n_major,
                                  int64_t n_minor, int *flags) {
  int range = 0, nan = 0;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nnz;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int a = maj[t], b = mnr[t];
    if (a < 0 || a >= n_major || b < 0 || b >= n_minor) range = 1;
    if (val && (__float_as_uint(val[t]) & 0x7fffffffu) > 0x7f800000u) nan = 1;
  }
  range = __syncthreads_or(range);
  nan = __syncthreads_or(nan);
  if (threadIdx.x == 0) {
    if (range) atomicOr(&flags[0], 1);
    if (nan) atomicOr(&flags[1], 1);
  }
}

__global__ void count64_kernel(const int32_t *__restrict__ maj, int64_t n,
                               unsigned long long *__restrict__ cnt) {
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x)
    atomicAdd(&cnt[maj[t]], 1ull);
}

// Selection of the entries whose major index lies in [s0, s1), in input
// order: tile b (kTile entries) counts its matches, an exclusive scan of the
// counts gives each tile's first output position, and the tile writes its
// matches in order (thread k holds entries k*kItems .. k*kItems+kItems-1 of
// the tile; a block scan orders the threads).
__global__ void select_count_kernel(const int32_t *__restrict__ maj, int64_t n, int s0, int s1,
                                    int64_t *__restrict__ tile_count) {
  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
  int c = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int64_t i = base + k;
    if (i < n && maj[i] >= s0 && maj[i] < s1) ++c;
  }
  int total;
  block_exclusive_scan<kThreads>(c, total);
  if (threadIdx.x == 0) tile_count[blockIdx.x] = total;
}

__global__ void select_write_kernel(const int32_t *__restrict__ maj, const int32_t *__restrict__ mnr,
                                    const uint32_t *__restrict__ val, int words, int64_t n, int s0,
                                    int s1, const int64_t *__restrict__ tile_first,
                                    int32_t *__restrict__ out_maj, int32_t *__restrict__ out_mnr,
                                    uint32_t *__restrict__ out_val) {
  const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)threadIdx.x * kItems;
  bool keep[kItems];
  int c = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int64_t i = base + k;
    keep[k] = i < n && maj[i] >= s0 && maj[i] < s1;
    c += keep[k];
  }
  int total;
  int64_t pos = tile_first[blockIdx.x] + block_exclusive_scan<kThreads>(c, total);
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    if (!keep[k]) continue;
    const int64_t i = base + k;
    out_maj[pos] = maj[i] - s0;
    out_mnr[pos] = mnr[i];
    for (int q = 0; q < words; ++q) out_val[pos * words + q] = val[i * words + q];
    ++pos;
  }
}

// p[i] += d, i < n
__global__ void shift_kernel(int32_t *__restrict__ p, int64_t n, int32_t d) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] += d;
}

// out[i] = d for i < lead; out[lead + i] = d + src[i] for i < n
__global__ void lead_shift_kernel(const int32_t *__restrict__ src, int64_t n, int lead, int32_t d,
                                  int32_t *__restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n + lead;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = i < lead ? d : d + src[i - lead];
}

// dst[i] = add + src[i], i < n
__global__ void widen_kernel(const int32_t *__restrict__ src, int64_t n, int64_t add,
                             int64_t *__restrict__ dst) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = add + (int64_t)src[i];
}

}  // namespace

vs_status build_wide(Matrix &m, vs_layout layout, vs_major major, vs_dtype dtype, int64_t n_rows,
                     int64_t n_cols, int64_t nnz, const int32_t *d_row, const int32_t *d_col,
                     const void *d_val, int64_t seg_entries, cudaStream_t s) {
  m.layout = layout;
  m.major = major;
  m.dtype = dtype;
  m.n_rows = n_rows;
  m.n_cols = n_cols;
  m.n_major = major == VS_MAJOR_ROW ? n_rows : n_cols;
  m.n_minor = major == VS_MAJOR_ROW ? n_cols : n_rows;
  m.nnz = nnz;
  m.wide = true;
  m.seg_entries = seg_entries > 0 ? std::min(seg_entries, kMaxSegmentEntries) : kMaxSegmentEntries;
  const int32_t *maj = major == VS_MAJOR_ROW ? d_row : d_col;
  const int32_t *mnr = major == VS_MAJOR_ROW ? d_col : d_row;
  const bool vcs = layout == VS_LAYOUT_VCS;
  const size_t dsize = m.dsize();
  const unsigned eg = std::min<unsigned>(kGridCap, grid_for(nnz, 256));

  // ---- checks over every entry, and the entries of each slice
  Temp flags(s), cnt(s);
  VS_TRY(flags.alloc(2 * sizeof(int)));
  VS_CUDA(cudaMemsetAsync(flags.p, 0, 2 * sizeof(int), s));
  VS_TRY(cnt.alloc(sizeof(unsigned long long) * (size_t)std::max<int64_t>(m.n_major, 1)));
  VS_CUDA(cudaMemsetAsync(cnt.p, 0, sizeof(unsigned long long) * (size_t)std::max<int64_t>(m.n_major, 1), s));
  int hflags[2] = {0, 0};
  if (nnz > 0) {
    wide_check_kernel<<<eg, 256, 0, s>>>(maj, mnr, vcs ? static_cast<const float *>(d_val) : nullptr,
                                         nnz, m.n_major, m.n_minor, flags.as<int>());
    VS_LAUNCH_CHECK();
    VS_CUDA(cudaMemcpyAsync(hflags, flags.p, sizeof hflags, cudaMemcpyDeviceToHost, s));
    VS_CUDA(cudaStreamSynchronize(s));
    if (hflags[0]) {
      set_error("a COO coordinate lies outside the matrix");
      return VS_ERR_RANGE;
    }
    if (hflags[1]) {
      set_error("NaN value: VCS runs need an ordered value key");
      return VS_ERR_NAN;
    }
    count64_kernel<<<eg, 256, 0, s>>>(maj, nnz, cnt.as<unsigned long long>());
    VS_LAUNCH_CHECK();
  }
  std::vector<unsigned long long> counts((size_t)m.n_major);
  if (m.n_major > 0)
    VS_CUDA(cudaMemcpyAsync(counts.data(), cnt.p, sizeof(unsigned long long) * counts.size(),
                            cudaMemcpyDeviceToHost, s));
  VS_CUDA(cudaStreamSynchronize(s));
  std::vector<int64_t> start((size_t)m.n_major + 1, 0);  // entry start of each slice
  for (int64_t k = 0; k < m.n_major; ++k) {
    if ((int64_t)counts[k] > kMaxSegmentEntries) {
      set_error("a slice holds more entries than one kernel segment takes (about 2^31)");
      return VS_ERR_UNSUPPORTED;
    }
    start[k + 1] = start[k] + (int64_t)counts[k];
  }

  // ---- segments: consecutive slices with at most seg_entries entries (a
  // longer slice alone)
  std::vector<std::pair<int64_t, int64_t>> cuts;  // [s0, s1)
  for (int64_t s0 = 0; s0 < m.n_major;) {
    int64_t s1 = std::upper_bound(start.begin() + s0 + 1, start.end(), start[s0] + m.seg_entries) -
                 start.begin() - 1;
    s1 = std::max(s1, s0 + 1);
    cuts.emplace_back(s0, s1);
    s0 = s1;
  }
  VS_TRY(dev_alloc((void **)&m.ptr64, sizeof(int64_t) * (size_t)(m.n_major + 1 + 16)));
  VS_CUDA(cudaMemsetAsync(m.ptr64, 0, sizeof(int64_t) * (size_t)(m.n_major + 1 + 16), s));
  VS_TRY(dev_alloc((void **)&m.idx, sizeof(int32_t) * (size_t)(nnz + 16)));
  VS_CUDA(cudaMemsetAsync(m.idx, 0, sizeof(int32_t) * (size_t)(nnz + 16), s));
  if (!vcs) {
    VS_TRY(dev_alloc(&m.vals, dsize * (size_t)(nnz + 16)));
    VS_CUDA(cudaMemsetAsync(m.vals, 0, dsize * (size_t)(nnz + 16), s));
  }
  m.segs.resize(cuts.size());
  const int64_t ntiles = std::max<int64_t>(1, (nnz + kTile - 1) / kTile);
  Temp tile_count(s), tile_first(s);
  VS_TRY(tile_count.alloc(sizeof(int64_t) * (size_t)ntiles));
  VS_TRY(tile_first.alloc(sizeof(int64_t) * (size_t)ntiles));
  std::vector<int64_t> htc((size_t)ntiles);
  const int words = (int)((vcs ? sizeof(float) : dsize) / 4);
  int64_t r_base = 0;
  for (size_t k = 0; k < cuts.size(); ++k) {
    Matrix &g = m.segs[k];
    const int64_t s0 = cuts[k].first, s1 = cuts[k].second;
    const int64_t e0 = start[s0], ne = start[s1] - start[s0];
    // this segment's entries, in input order, with slice indices relative to s0
    Temp smaj(s), smnr(s), sval(s);
    VS_TRY(smaj.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(ne, 1)));
    VS_TRY(smnr.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(ne, 1)));
    VS_TRY(sval.alloc(sizeof(uint32_t) * words * (size_t)std::max<int64_t>(ne, 1)));
    if (nnz > 0) {
      select_count_kernel<<<(unsigned)ntiles, kThreads, 0, s>>>(maj, nnz, (int)s0, (int)s1,
                                                                tile_count.as<int64_t>());
      VS_LAUNCH_CHECK();
      VS_CUDA(cudaMemcpyAsync(htc.data(), tile_count.p, sizeof(int64_t) * htc.size(),
                              cudaMemcpyDeviceToHost, s));
      VS_CUDA(cudaStreamSynchronize(s));
      int64_t run = 0;
      for (auto &c : htc) {
        const int64_t v = c;
        c = run;
        run += v;
      }
      if (run != ne) {
        set_error("internal: segment selection count mismatch");
        return VS_ERR_CUDA;
      }
      VS_CUDA(cudaMemcpyAsync(tile_first.p, htc.data(), sizeof(int64_t) * htc.size(),
                              cudaMemcpyHostToDevice, s));
      select_write_kernel<<<(unsigned)ntiles, kThreads, 0, s>>>(
          maj, mnr, static_cast<const uint32_t *>(d_val), words, nnz, (int)s0, (int)s1,
          tile_first.as<int64_t>(), smaj.as<int32_t>(), smnr.as<int32_t>(), sval.as<uint32_t>());
      VS_LAUNCH_CHECK();
    }
    // assembled like any int32 matrix (rows = the segment's slices)
    VS_TRY(build_matrix(g, layout, VS_MAJOR_ROW, dtype, s1 - s0, m.n_minor, ne, smaj.as<int32_t>(),
                        smnr.as<int32_t>(), sval.p, s));
    g.major = major;
    g.n_rows = major == VS_MAJOR_ROW ? s1 - s0 : m.n_minor;
    g.n_cols = major == VS_MAJOR_ROW ? m.n_minor : s1 - s0;
    g.seg_slice0 = s0;
    const int64_t r0 = vcs ? r_base : e0, R_seg = g.R;
    // the whole matrix's indices (and CSR values) take the segment's; the
    // segment keeps views of them
    if (ne > 0) {
      VS_CUDA(cudaMemcpyAsync(m.idx + e0, g.idx, sizeof(int32_t) * (size_t)ne,
                              cudaMemcpyDeviceToDevice, s));
      if (!vcs)
        VS_CUDA(cudaMemcpyAsync(static_cast<char *>(m.vals) + (size_t)e0 * dsize, g.vals,
                                dsize * (size_t)ne, cudaMemcpyDeviceToDevice, s));
    }
    // 64-bit slice pointers: entry starts (CSR) or run starts (VCS)
    const unsigned pg = std::min<unsigned>(kGridCap, grid_for(s1 - s0 + 1, 256));
    widen_kernel<<<pg, 256, 0, s>>>(g.ptr, s1 - s0 + 1, r0, m.ptr64 + s0);
    VS_LAUNCH_CHECK();
    // The segment's views start at the 16-byte boundary at or before its first
    // entry (and run), as the bulk copies of its blocks need: its slice
    // pointers count from there, past `lead` entries (runs) of the previous
    // segment that none of its slices names.
    const int lead_e = (int)(e0 & 3), lead_r = vcs ? (int)(r0 & 3) : lead_e;
    g.seg_entry0 = e0 - lead_e;
    g.seg_run0 = r0 - lead_r;
    g.seg_lead_e = lead_e;
    g.seg_lead_r = lead_r;
    if (lead_r) {
      shift_kernel<<<pg, 256, 0, s>>>(g.ptr, s1 - s0 + 1, lead_r);
      VS_LAUNCH_CHECK();
    }
    if (vcs) {
      // run starts: lead_r leading runs (never named), the rest shifted by lead_e
      int32_t *vp = nullptr;
      VS_TRY(dev_alloc((void **)&vp, sizeof(int32_t) * (size_t)(R_seg + lead_r + 1 + 16)));
      VS_CUDA(cudaMemsetAsync(vp, 0, sizeof(int32_t) * (size_t)(R_seg + lead_r + 1 + 16), s));
      lead_shift_kernel<<<std::min<unsigned>(kGridCap, grid_for(R_seg + 1 + lead_r, 256)), 256, 0,
                          s>>>(g.vptr, R_seg + 1, lead_r, lead_e, vp);
      VS_LAUNCH_CHECK();
      VS_CUDA(cudaStreamSynchronize(s));
      cudaFree(g.vptr);
      g.vptr = vp;
      g.R = R_seg + lead_r;
    } else {
      g.R = ne + lead_e;
    }
    g.nnz = ne + lead_e;
    VS_CUDA(cudaStreamSynchronize(s));
    cudaFree(g.idx);
    g.idx = m.idx + g.seg_entry0;
    g.borrowed_idx = true;
    if (!vcs) {
      cudaFree(g.vals);
      g.vals = static_cast<char *>(m.vals) + (size_t)g.seg_entry0 * dsize;
      g.borrowed_vals = true;
    }
    r_base += R_seg;
  }
  m.R = vcs ? r_base : nnz;
  if (vcs) {
    // run values and 64-bit run starts of the whole matrix
    VS_TRY(dev_alloc(&m.vals, sizeof(float) * (size_t)(m.R + 16)));
    VS_CUDA(cudaMemsetAsync(m.vals, 0, sizeof(float) * (size_t)(m.R + 16), s));
    VS_TRY(dev_alloc((void **)&m.vptr64, sizeof(int64_t) * (size_t)(m.R + 1 + 16)));
    VS_CUDA(cudaMemsetAsync(m.vptr64, 0, sizeof(int64_t) * (size_t)(m.R + 1 + 16), s));
    for (Matrix &g : m.segs) {
      // the segment's own runs (after its lead): values and 64-bit run starts
      const int64_t r0 = g.seg_run0 + g.seg_lead_r, R_seg = g.R - g.seg_lead_r;
      if (R_seg > 0)
        VS_CUDA(cudaMemcpyAsync(static_cast<float *>(m.vals) + r0, g.vals,
                                sizeof(float) * (size_t)R_seg, cudaMemcpyDeviceToDevice, s));
      widen_kernel<<<std::min<unsigned>(kGridCap, grid_for(R_seg + 1, 256)), 256, 0, s>>>(
          g.vptr + (r0 - g.seg_run0), R_seg + 1, g.seg_entry0, m.vptr64 + r0);
      VS_LAUNCH_CHECK();
    }
    VS_CUDA(cudaStreamSynchronize(s));
    for (Matrix &g : m.segs) {
      cudaFree(g.vals);
      g.vals = static_cast<float *>(m.vals) + g.seg_run0;
      g.borrowed_vals = true;
    }
  }
  // kernel parameters of every segment, with the whole matrix's group size
  m.g = group_size_rule(m.nnz, m.n_major);
  m.sorted_segments = true;
  for (Matrix &g : m.segs) {
    g.tt_req_rows = m.tt_req_rows;
    VS_TRY(prepare_matrix(g, s));
    g.g = m.g;
    m.n_sm = g.n_sm;
    m.sorted_segments = m.sorted_segments && g.sorted_segments;
    m.n_blocks += g.n_blocks;
    m.n_long += g.n_long;
    m.n_chunks += g.n_chunks;
  }
  if (m.segs.empty()) {
    int dev = 0;
    VS_CUDA(cudaGetDevice(&dev));
    VS_CUDA(cudaDeviceGetAttribute(&m.n_sm, cudaDevAttrMultiProcessorCount, dev));
  }
  return VS_OK;
}

// ------------------------------------------------------------------ transpose

namespace {

// COO of a stored layout, in layout order: (major, minor, value bits).  The
// major index written is slice0 + s (a segment of a wide matrix passes its
// first slice, and output pointers already offset to its first entry).
__global__ void expand_csr_kernel(const int32_t *__restrict__ ptr, int64_t n_major,
                                  int32_t *__restrict__ out_major, int64_t slice0 = 0) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n_major;
       s += (int64_t)gridDim.x * blockDim.x)
    for (int32_t k = ptr[s]; k < ptr[s + 1]; ++k) out_major[k] = (int32_t)(slice0 + s);
}

__global__ void expand_vcs_kernel(const int32_t *__restrict__ major_ptr,
                                  const int32_t *__restrict__ vptr, const float *__restrict__ values,
                                  int64_t n_major, int32_t *__restrict__ out_major,
                                  float *__restrict__ out_val, int64_t slice0 = 0) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n_major;
       s += (int64_t)gridDim.x * blockDim.x)
    for (int32_t r = major_ptr[s]; r < major_ptr[s + 1]; ++r)
      for (int32_t k = vptr[r]; k < vptr[r + 1]; ++k) {
        out_major[k] = (int32_t)(slice0 + s);
        out_val[k] = values[r];
      }
}

}  // namespace

vs_status build_transpose(const Matrix &src, Matrix &dst, cudaStream_t s) {
  const int64_t nnz = src.nnz;
  Temp maj(s), vals(s);
  if (src.wide) {
    // the COO of every segment into the whole matrix's positions, then a wide build
    VS_TRY(maj.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1)));
    const bool vcs = src.layout == VS_LAYOUT_VCS;
    if (vcs) VS_TRY(vals.alloc(sizeof(float) * (size_t)std::max<int64_t>(nnz, 1)));
    for (const Matrix &g : src.segs) {
      if (g.n_major == 0) continue;
      const unsigned gg = std::min<unsigned>(kGridCap, grid_for(g.n_major, 256));
      if (vcs)
        expand_vcs_kernel<<<gg, 256, 0, s>>>(g.ptr, g.vptr, static_cast<const float *>(g.vals),
                                             g.n_major, maj.as<int32_t>() + g.seg_entry0,
                                             vals.as<float>() + g.seg_entry0, g.seg_slice0);
      else
        expand_csr_kernel<<<gg, 256, 0, s>>>(g.ptr, g.n_major, maj.as<int32_t>() + g.seg_entry0,
                                             g.seg_slice0);
      VS_LAUNCH_CHECK();
    }
    const vs_major other = src.major == VS_MAJOR_ROW ? VS_MAJOR_COL : VS_MAJOR_ROW;
    const int32_t *rows = src.major == VS_MAJOR_ROW ? maj.as<int32_t>() : src.idx;
    const int32_t *cols = src.major == VS_MAJOR_ROW ? src.idx : maj.as<int32_t>();
    return build_wide(dst, src.layout, other, src.dtype, src.n_rows, src.n_cols, nnz, rows, cols,
                      vcs ? vals.p : src.vals, src.seg_entries, s);
  }
  VS_TRY(maj.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(nnz, 1)));
  const unsigned g = std::min<unsigned>(kGridCap, grid_for(src.n_major, 256));
  const void *val_ptr = src.vals;
  if (src.layout == VS_LAYOUT_CSR) {
    if (src.n_major > 0) {
      expand_csr_kernel<<<g, 256, 0, s>>>(src.ptr, src.n_major, maj.as<int32_t>());
      VS_LAUNCH_CHECK();
    }
  } else {
    VS_TRY(vals.alloc(sizeof(float) * (size_t)std::max<int64_t>(nnz, 1)));
    if (src.n_major > 0) {
      expand_vcs_kernel<<<g, 256, 0, s>>>(src.ptr, src.vptr, static_cast<const float *>(src.vals),
                                          src.n_major, maj.as<int32_t>(), vals.as<float>());
      VS_LAUNCH_CHECK();
    }
    val_ptr = vals.p;
  }
  // the stored major axis becomes the minor axis of the transpose
  const vs_major other = src.major == VS_MAJOR_ROW ? VS_MAJOR_COL : VS_MAJOR_ROW;
  const int32_t *rows = src.major == VS_MAJOR_ROW ? maj.as<int32_t>() : src.idx;
  const int32_t *cols = src.major == VS_MAJOR_ROW ? src.idx : maj.as<int32_t>();
  return build_matrix(dst, src.layout, other, src.dtype, src.n_rows, src.n_cols, nnz, rows, cols,
                      val_ptr, s);
}

// ------------------------------------------------------------------ matrix-only parameters

namespace {
__global__ void mark_starts_kernel(const int32_t *__restrict__ seg_ptr, int64_t n_seg,
                                   uint8_t *__restrict__ start) {
  for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n_seg;
       s += (int64_t)gridDim.x * blockDim.x)
    start[seg_ptr[s]] = 1;
}
__global__ void unsorted_kernel(const int32_t *__restrict__ idx, const uint8_t *__restrict__ start,
                                int64_t n, int *flag) {
  int bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x + 1; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    if (!start[i] && idx[i] < idx[i - 1]) bad = 1;
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(flag, 1);
}
}  // namespace

vs_status prepare_matrix(Matrix &m, cudaStream_t s) {
  if (m.wide) return VS_OK;  // build_wide prepared every segment
  // slice entry ranges on the host
  std::vector<int32_t> ptr(m.n_major + 1), vptr;
  VS_CUDA(cudaMemcpyAsync(ptr.data(), m.ptr, sizeof(int32_t) * (m.n_major + 1),
                          cudaMemcpyDeviceToHost, s));
  if (m.layout == VS_LAYOUT_VCS) {
    vptr.resize(m.R + 1);
    VS_CUDA(cudaMemcpyAsync(vptr.data(), m.vptr, sizeof(int32_t) * (m.R + 1),
                            cudaMemcpyDeviceToHost, s));
  }
  // are the minor indices ascending inside every segment (row or run)?
  int unsorted = 0;
  if (m.layout == VS_LAYOUT_VCS) {
    m.sorted_segments = true;  // by construction
  } else if (m.nnz > 1) {
    Temp start(s), flag(s);
    VS_TRY(start.alloc(m.nnz + 1));
    VS_TRY(flag.alloc(sizeof(int)));
    VS_CUDA(cudaMemsetAsync(start.p, 0, m.nnz + 1, s));
    VS_CUDA(cudaMemsetAsync(flag.p, 0, sizeof(int), s));
    mark_starts_kernel<<<std::min<unsigned>(kGridCap, grid_for(m.n_major, 256)), 256, 0, s>>>(
        m.ptr, m.n_major, start.as<uint8_t>());
    VS_LAUNCH_CHECK();
    unsorted_kernel<<<std::min<unsigned>(kGridCap, grid_for(m.nnz, 256)), 256, 0, s>>>(
        m.idx, start.as<uint8_t>(), m.nnz, flag.as<int>());
    VS_LAUNCH_CHECK();
    VS_CUDA(cudaMemcpyAsync(&unsorted, flag.p, sizeof(int), cudaMemcpyDeviceToHost, s));
    VS_CUDA(cudaStreamSynchronize(s));
    m.sorted_segments = !unsorted;
  } else {
    m.sorted_segments = true;
  }
  VS_CUDA(cudaStreamSynchronize(s));
  auto entry = [&](int64_t sl) -> int64_t {
    return m.layout == VS_LAYOUT_VCS ? vptr[ptr[sl]] : ptr[sl];
  };

  m.g = group_size_rule(m.nnz, m.n_major);
  {
    int dev = 0;
    VS_CUDA(cudaGetDevice(&dev));
    VS_CUDA(cudaDeviceGetAttribute(&m.n_sm, cudaDevAttrMultiProcessorCount, dev));
  }

  // ---- blocks: runs of short slices, and chunks of long slices
  const bool vcs = m.layout == VS_LAYOUT_VCS;
  auto runs_of = [&](int64_t sl) -> int64_t { return vcs ? ptr[sl + 1] - ptr[sl] : 0; };
  std::vector<int4> desc;
  auto push = [&](int4 x, int4 y, int4 z) {
    desc.push_back(x);
    desc.push_back(y);
    desc.push_back(z);
  };
  int64_t n_long = 0, n_chunks = 0, n_shares = 0;
  std::vector<int4> longs;  // {slice, first share, shares, 0} per long slice
  int64_t bs0 = -1, be = 0, br = 0;  // open slice block: first slice, entries, runs
  auto close_slices = [&](int64_t s_end) {
    if (bs0 < 0) return;
    push(make_int4((int)bs0, (int)s_end, (int)entry(bs0), (int)entry(s_end)),
         make_int4(vcs ? ptr[bs0] : 0, vcs ? ptr[s_end] : 0, 0, -1), make_int4(0, 0, 0, 0));
    bs0 = -1;
  };
  for (int64_t sl = 0; sl < m.n_major; ++sl) {
    const int64_t len = entry(sl + 1) - entry(sl), nr = runs_of(sl);
    const bool is_long = len > kBlockEntries || nr > kBlockRuns;
    if (!is_long) {
      if (bs0 >= 0 && (be + len > kBlockEntries || br + nr > kBlockRuns ||
                       sl - bs0 + 1 > kBlockSlices))
        close_slices(sl);
      if (bs0 < 0) {
        bs0 = sl;
        be = br = 0;
      }
      be += len;
      br += nr;
      continue;
    }
    close_slices(sl);
    // cut the long slice into chunks of at most kBlockEntries entries and kBlockRuns runs
    std::vector<int4> ch;  // {e0, e1, r0, r1}
    int64_t pos = entry(sl), r = vcs ? ptr[sl] : 0;
    const int64_t end = entry(sl + 1);
    while (pos < end) {
      int64_t e1 = std::min<int64_t>(end, pos + kBlockEntries);
      int64_t r_first = r, r_last = r;
      if (vcs) {
        while (r_first < ptr[sl + 1] - 1 && vptr[r_first + 1] <= pos) ++r_first;
        r_last = r_first;
        while (r_last + 1 < ptr[sl + 1] && vptr[r_last + 1] < e1) ++r_last;
        if (r_last - r_first + 1 > kBlockRuns) {
          r_last = r_first + kBlockRuns - 1;
          e1 = vptr[r_last + 1];
        }
        r = r_last;
      }
      ch.push_back(make_int4((int)pos, (int)e1, (int)r_first, (int)(r_last + 1)));
      pos = e1;
    }
    int64_t sh = n_shares;  // first share of this slice
    int64_t slice_shares = 0;
    for (size_t k2 = 0; k2 < ch.size(); ++k2)
      slice_shares += (ch[k2].y - ch[k2].x + kShareEntries - 1) / kShareEntries;
    for (size_t k2 = 0; k2 < ch.size(); ++k2) {
      push(make_int4((int)sl, (int)k2, ch[k2].x, ch[k2].y),
           make_int4(vcs ? ch[k2].z : 0, vcs ? ch[k2].w : 0, 1, (int)n_long),
           make_int4((int)sh, (int)n_shares, (int)slice_shares, 0));
      sh += (ch[k2].y - ch[k2].x + kShareEntries - 1) / kShareEntries;
    }
    n_chunks += (int64_t)ch.size();
    longs.push_back(make_int4((int)sl, (int)n_shares, (int)slice_shares, 0));
    n_shares += slice_shares;
    ++n_long;
  }
  close_slices(m.n_major);
  m.n_blocks = (int64_t)desc.size() / 3;
  m.n_long = n_long;
  m.n_chunks = n_chunks;
  m.n_shares = n_shares;
  if (m.n_blocks > 0) {
    VS_TRY(dev_alloc((void **)&m.blocks, sizeof(int4) * desc.size()));
    VS_CUDA(cudaMemcpyAsync(m.blocks, desc.data(), sizeof(int4) * desc.size(),
                            cudaMemcpyHostToDevice, s));
  }
  if (n_long > 0) {
    VS_TRY(dev_alloc((void **)&m.longs, sizeof(int4) * n_long));
    VS_CUDA(cudaMemcpyAsync(m.longs, longs.data(), sizeof(int4) * n_long, cudaMemcpyHostToDevice, s));
    // share partials hold sums of the operand type: float64 covers every product
    VS_TRY(dev_alloc(&m.partials, sizeof(double) * kMaxBlockWidth * n_shares));
  }
  VS_TRY(dev_alloc((void **)&m.err, sizeof(int)));
  VS_CUDA(cudaMemsetAsync(m.err, 0, sizeof(int), s));

  // ---- two-phase groups: C groups of consecutive blocks, balanced by entries.
  // C depends on the matrix only; it is kept small when the scattered output
  // is large, so that C partial copies of it stay bounded (64 MiB at width 64).
  {
    const int64_t c_nnz = std::max<int64_t>(1, (m.nnz + 32767) / 32768);
    const int64_t out_row_bytes = (int64_t)m.dsize() * kMaxBlockWidth;
    const int64_t c_mem =
        std::max<int64_t>(1, (int64_t(1) << 26) / std::max<int64_t>(1, m.n_minor * out_row_bytes));
    int64_t C = std::min<int64_t>(std::min(c_nnz, c_mem), 256);
    C = std::max<int64_t>(1, std::min<int64_t>(C, std::max<int64_t>(m.n_blocks, 1)));
    std::vector<int32_t> bounds(C + 1);
    bounds[0] = 0;
    int64_t b = 0;
    for (int64_t c = 1; c < C; ++c) {
      const int64_t target = m.nnz * c / C;
      while (b < m.n_blocks && desc[3 * b].z < target) ++b;
      bounds[c] = (int32_t)b;
    }
    bounds[C] = (int32_t)m.n_blocks;
    m.tp_chunks = (int)C;
    VS_TRY(dev_alloc((void **)&m.tp_bounds, sizeof(int32_t) * (C + 1)));
    VS_CUDA(cudaMemcpyAsync(m.tp_bounds, bounds.data(), sizeof(int32_t) * (C + 1),
                            cudaMemcpyHostToDevice, s));
  }
  // ---- the tiled two-phase scheme's per-(run, tile) entry offsets
  VS_TRY(build_tiled_two_phase(m, ptr, vptr, s));
  VS_CUDA(cudaStreamSynchronize(s));
  return VS_OK;
}

}  // namespace vs
