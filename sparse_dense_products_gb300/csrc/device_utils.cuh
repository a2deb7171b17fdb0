// device_utils.cuh -- small device helpers shared by the libvs kernels:
// vector types, cache-hinted loads, vector reductions and a block scan.
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

// Read-only, read-once streams (indices, values): no L1 allocation.
__device__ __forceinline__ int ld_stream(const int *p) {
  int v;
  asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_stream(const float *p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ double ld_stream(const double *p) {
  double v;
  asm("ld.global.nc.L1::no_allocate.f64 %0, [%1];" : "=d"(v) : "l"(p));
  return v;
}

// Gathered dense rows: read-only, cached in L1.
template <typename V>
__device__ __forceinline__ V ld_gather(const V *p) {
  return __ldg(p);
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
