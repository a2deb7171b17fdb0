// device_utils.cuh -- small device helpers shared by the libvs kernels:
// vector types, shared and gather loads, vector reductions, scans, mbarrier
// and bulk-copy wrappers, and the programmatic-dependent-launch helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vs {

constexpr unsigned kFullMask = 0xffffffffu;

template <typename T, int VEC>
struct VecT;
template <>
struct VecT<float, 4> {
  using type = float4;
};
template <>
struct VecT<float, 2> {
  using type = float2;
};
template <>
struct VecT<float, 1> {
  using type = float;
};
template <>
struct VecT<double, 2> {
  using type = double2;
};
template <>
struct VecT<double, 1> {
  using type = double;
};

// Element e of a vector value, and the reverse.
template <typename T, int VEC>
struct VecOps {
  using V = typename VecT<T, VEC>::type;
  __device__ __forceinline__ static void unpack(const V &v, T (&o)[VEC]) {
    const T *p = reinterpret_cast<const T *>(&v);
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[e] = p[e];
  }
  __device__ __forceinline__ static V pack(const T (&o)[VEC]) {
    V v;
    T *p = reinterpret_cast<T *>(&v);
#pragma unroll
    for (int e = 0; e < VEC; ++e) p[e] = o[e];
    return v;
  }
};

// Gathered dense rows: read-only, cached in L1.
template <typename V>
__device__ __forceinline__ V ld_gather(const V *p) {
  return __ldg(p);
}

// Shared-memory vector loads at a 32-bit shared address.
template <typename V>
__device__ __forceinline__ V ld_shared(uint32_t addr);
template <>
__device__ __forceinline__ float4 ld_shared<float4>(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
template <>
__device__ __forceinline__ float2 ld_shared<float2>(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
template <>
__device__ __forceinline__ float ld_shared<float>(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
template <>
__device__ __forceinline__ double2 ld_shared<double2>(uint32_t addr) {
  double2 v;
  asm volatile("ld.shared.v2.f64 {%0, %1}, [%2];" : "=d"(v.x), "=d"(v.y) : "r"(addr));
  return v;
}
template <>
__device__ __forceinline__ double ld_shared<double>(uint32_t addr) {
  double v;
  asm volatile("ld.shared.f64 %0, [%1];" : "=d"(v) : "r"(addr));
  return v;
}

// Programmatic dependent launch: a kernel launched with launch_early may be
// resident before the previous kernel of its stream has finished; this waits
// until that kernel has completed and its memory is visible (a no-op when
// there is no such dependency).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launches `kernel` allowing it to start while the previous kernel of the
// stream drains (the kernel must call grid_dependency_wait before it reads
// or writes memory that kernel may touch).
template <typename... KArgs, typename... Args>
cudaError_t launch_early(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Barrier over the first `threads` threads of the block (named barrier `id`).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Atomic accumulation (no return value) of a vector into global memory.
__device__ __forceinline__ void red_add(float *p, const float (&v)[4]) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3])
               : "memory");
}
__device__ __forceinline__ void red_add(float *p, const float (&v)[2]) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(v[0]), "f"(v[1]) : "memory");
}
__device__ __forceinline__ void red_add(float *p, const float (&v)[1]) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v[0]) : "memory");
}
__device__ __forceinline__ void red_add(double *p, const double (&v)[2]) {
  asm volatile("red.global.add.f64 [%0], %1;" ::"l"(p), "d"(v[0]) : "memory");
  asm volatile("red.global.add.f64 [%0], %1;" ::"l"(p + 1), "d"(v[1]) : "memory");
}
__device__ __forceinline__ void red_add(double *p, const double (&v)[1]) {
  asm volatile("red.global.add.f64 [%0], %1;" ::"l"(p), "d"(v[0]) : "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Inclusive warp scan of ints.
__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int u = __shfl_up_sync(kFullMask, v, d);
    if (lane >= d) v += u;
  }
  return v;
}

// Exclusive scan of one int per thread over a block of NT threads (NT % 32 == 0).
// Returns the thread's exclusive prefix; *total receives the block sum.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int &total) {
  __shared__ int warp_sums[NT / 32];
  __shared__ int block_total;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int inc = warp_inclusive_scan(v);
  if (lane == 31) warp_sums[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    int s = lane < NT / 32 ? warp_sums[lane] : 0;
    int si = warp_inclusive_scan(s);
    if (lane < NT / 32) warp_sums[lane] = si - s;
    if (lane == 31) block_total = si;
  }
  __syncthreads();
  int r = warp_sums[wid] + inc - v;
  total = block_total;
  __syncthreads();
  return r;
}

}  // namespace vs

namespace vs {

// ------------------------------------------------------------------ bulk copies and mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the asynchronous (bulk copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One non-tensor bulk copy global -> shared that signals `bar` with its byte count.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking: whether phase `parity` of `bar` has completed.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar` for at most about `limit_ns`; false if it
// gave up.  try_wait itself suspends the thread for a while when the phase is
// not complete; the clock is read only every 64 tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 64; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

}  // namespace vs
