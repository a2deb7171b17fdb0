// stage.cuh -- streaming of matrix blocks through shared memory.
//
// The stored entries of a matrix are cut (once, at build time, from the matrix
// alone) into blocks of at most kBlockEntries entries, kBlockRuns runs and
// kBlockSlices slices.  A block is either
//   * a slice block: consecutive slices [s0, s1), each short enough for one
//     warp, or
//   * a chunk block: chunk k, entries [e0, e1), of a long slice s0; the chunk
//     is further cut into shares of kShareEntries entries.
//
// Each CTA runs a producer/consumer pipeline over its blocks.  A producer warp
// brings a block's index, value, slice-pointer and run arrays, and its
// descriptor, into one of the stage buffers with bulk copies (cp.async.bulk),
// signalled on the buffer's "full" mbarrier.  For VCS the run values are then
// expanded to one value per entry in shared memory (by the same warp, or by
// dedicated expanding warps) and the buffer's "ready" mbarrier is signalled.
// The consumer warps (kWarpsPerCta, or the count the kernel passes to
// Pipe::init) take the block's work units (groups of slices, or shares) in a
// round-robin the kernel fixes, and when done arrive on the buffer's "empty"
// mbarrier, which lets the producer refill it.  Warps never wait for one
// another except through these barriers, and every wait is bounded in time.
#pragma once

#include "device_utils.cuh"
#include "vs_internal.h"

namespace vs {

constexpr int kStages = 4;
constexpr int kConsumerThreads = kWarpsPerCta * 32;
constexpr int kPipeThreads = kConsumerThreads + 32;  // plus the producer warp
constexpr uint64_t kWaitLimitNs = 1000000000ull;     // 1 s
constexpr int kFillRuns = 16;  // VCS expansion: blocks with at most this many runs fill run by run

// Element capacity of each staged array, with room for 16-byte alignment slack.
constexpr int kCapEntries = kBlockEntries + 8;
constexpr int kCapSlices = kBlockSlices + 8;
constexpr int kCapRuns = kBlockRuns + 8;

struct StageArrays {
  const int32_t *ptr;   // slice pointer (CSR entry starts / VCS run starts), padded
  const int32_t *idx;   // minor indices, padded
  const void *vals;     // CSR: entry values of T; VCS: run values (float), padded
  const int32_t *vptr;  // VCS: run entry starts, padded
  const int4 *blocks;   // [n_blocks][3]
  int n_blocks;
  int *err;             // set to 1 when a bounded wait gives up
  // Optional L2 prefetch of the dense rows X[s0:s1) of each slice block
  // (misaligned products read X by slice): base, row stride, element size,
  // valid elements per row; nullptr disables it.
  const void *xrows;
  int64_t xld;
  int xes, xw;
};

// Byte layout of one stage buffer for value type T.
template <typename T, bool VCS>
struct StageLayout {
  static constexpr int kIdx = 0;
  static constexpr int kVals = kIdx + kCapEntries * 4;                              // CSR only
  static constexpr int kPtr = kVals + (VCS ? 0 : kCapEntries * (int)sizeof(T));
  static constexpr int kVptr = kPtr + kCapSlices * 4;                               // VCS only
  static constexpr int kRvals = kVptr + (VCS ? kCapRuns * 4 : 0);                   // VCS only
  static constexpr int kEvals = kRvals + (VCS ? kCapRuns * 4 : 0);                  // VCS only
  static constexpr int kBitmap = kEvals + (VCS ? kCapEntries * 4 : 0);              // VCS only
  static constexpr int kWords = (kCapEntries + 31) / 32;                           // bitmap words
  static constexpr int kDesc = kBitmap + (VCS ? (kWords * 4 + 15) / 16 * 16 : 0);
  static constexpr int kBytes = kDesc + 3 * 16;  // the block's descriptor, copied by the producer
  static_assert(kVals % 16 == 0 && kPtr % 16 == 0 && kVptr % 16 == 0 && kRvals % 16 == 0 &&
                    kEvals % 16 == 0 && kBitmap % 16 == 0 && kDesc % 16 == 0 &&
                    kBytes % 16 == 0,
                "stage arrays must start on 16-byte boundaries");
};

// Shared memory of a pipelined kernel with NS stage buffers: the buffers,
// then the control words (full, empty and ready barriers, failure flag,
// slab barrier), then `extra`.
template <typename T, bool VCS, int NS = kStages>
struct PipeLayout {
  static constexpr int kBufs = 0;
  static constexpr int kFull = NS * StageLayout<T, VCS>::kBytes;
  static constexpr int kEmpty = kFull + 8 * NS;
  static constexpr int kReady = kEmpty + 8 * NS;  // VCS: run values expanded
  static constexpr int kFail = kReady + 8 * NS;
  static constexpr int kSlab = kFail + 8;  // gather: the shared-memory copy of X landed
  static constexpr int kExtra = (kSlab + 8 + 127) / 128 * 128;
};

template <typename T, bool VCS, int NS = kStages>
constexpr int pipe_smem_bytes(int extra) {
  return PipeLayout<T, VCS, NS>::kExtra + extra;
}

// A block's descriptor, decoded.
struct Block {
  int s0, s1, e0, e1;     // slice range, or (slice, chunk index); entry range
  int r0, r1, type, lid;  // run range (VCS); 0 = slices, 1 = chunk; long-slice id
  int first;              // chunk blocks: global index of this chunk's first share
  int sfirst, nsh;        // chunk blocks: first share of the slice, shares of the slice
};

__device__ __forceinline__ Block decode_block(const int4 x, const int4 y, const int4 z) {
  return Block{x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w, z.x, z.y, z.z};
}

__device__ __forceinline__ Block load_block(const int4 *blocks, int b) {
  return decode_block(blocks[3 * b], blocks[3 * b + 1], blocks[3 * b + 2]);
}

// The descriptor of the block held by a stage buffer (written at issue).
template <typename T, bool VCS>
__device__ __forceinline__ Block stage_desc(const unsigned char *buf) {
  const int4 *d = reinterpret_cast<const int4 *>(buf + StageLayout<T, VCS>::kDesc);
  return decode_block(d[0], d[1], d[2]);
}

// A producer warp's window of 32 block descriptors, one per lane, so that the
// global loads of descriptors are not on the issue path of every block.
struct DescWindow {
  int4 x, y, z;
  int first = -1;  // position (in the warp's block sequence) of lane 0's block
  // Descriptor of the i-th block of the sequence b_begin + i * step (all lanes).
  __device__ __forceinline__ void get(const int4 *blocks, int b_begin, int step, int b_end, int i,
                                      int4 (&d)[3]) {
    const int lane = threadIdx.x & 31;
    if (first < 0 || i >= first + 32) {
      first = i - i % 32;
      const int b = b_begin + (first + lane) * step;
      if (b < b_end) {
        x = blocks[3 * b];
        y = blocks[3 * b + 1];
        z = blocks[3 * b + 2];
      }
    }
    const int src = i - first;
    d[0] = make_int4(__shfl_sync(kFullMask, x.x, src), __shfl_sync(kFullMask, x.y, src),
                     __shfl_sync(kFullMask, x.z, src), __shfl_sync(kFullMask, x.w, src));
    d[1] = make_int4(__shfl_sync(kFullMask, y.x, src), __shfl_sync(kFullMask, y.y, src),
                     __shfl_sync(kFullMask, y.z, src), __shfl_sync(kFullMask, y.w, src));
    d[2] = make_int4(__shfl_sync(kFullMask, z.x, src), __shfl_sync(kFullMask, z.y, src),
                     __shfl_sync(kFullMask, z.z, src), __shfl_sync(kFullMask, z.w, src));
  }
};

// Work units of a block: groups of S slices, or shares of a chunk.
__device__ __forceinline__ int block_units(const Block &k, int S) {
  return k.type == 0 ? (k.s1 - k.s0 + S - 1) / S
                     : (k.e1 - k.e0 + kShareEntries - 1) / kShareEntries;
}

// Views of the staged arrays of one block, indexed by global positions.
template <typename T, bool VCS>
struct Staged {
  const int32_t *idx;   // idx[n] for n in [e0, e1)
  const T *vals;        // vals[n]: CSR the stored values, VCS the run values expanded on chip
  const int32_t *ptr;   // ptr[s] for s in [s0, s1]
  const int32_t *vptr;  // VCS: vptr[r] for r in [r0, r1]
  const float *rvals;   // VCS: rvals[r] for r in [r0, r1)
};

template <int E>
__device__ __forceinline__ int align_down(int x) {
  return x & ~(E - 1);
}
template <int E>
__device__ __forceinline__ int align_up(int x) {
  return (x + E - 1) & ~(E - 1);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Producer (one thread): copy the descriptor d of a block into `buf`, issue
// the bulk copies of the block's arrays and arm `bar`.
template <typename T, bool VCS>
__device__ __forceinline__ void stage_issue(const StageArrays &a, const int4 (&d)[3],
                                            unsigned char *buf, uint64_t *bar) {
  using LY = StageLayout<T, VCS>;
  constexpr int VPE = 16 / (int)sizeof(T);  // values per 16 bytes
  int4 *dst = reinterpret_cast<int4 *>(buf + LY::kDesc);
  dst[0] = d[0];
  dst[1] = d[1];
  dst[2] = d[2];
  const Block k = decode_block(d[0], d[1], d[2]);
  uint32_t bytes = 0;
  int n_idx = 0, n_val = 0, n_ptr = 0, n_vp = 0, n_rv = 0;
  const int ei = align_down<4>(k.e0);
  if (k.e1 > k.e0) {
    n_idx = align_up<4>(k.e1) - ei;
    bytes += n_idx * 4;
    if (!VCS) {
      n_val = align_up<VPE>(k.e1) - align_down<VPE>(k.e0);
      bytes += n_val * (int)sizeof(T);
    }
  }
  const int pi = align_down<4>(k.s0);
  if (k.type == 0) {
    n_ptr = align_up<4>(k.s1 + 1) - pi;
    bytes += n_ptr * 4;
  }
  const int ri = align_down<4>(k.r0);
  if (VCS) {  // run starts [r0, r1] always (empty slices read vptr[r0]); values [r0, r1)
    n_vp = align_up<4>(k.r1 + 1) - ri;
    n_rv = k.r1 > k.r0 ? align_up<4>(k.r1) - ri : 0;
    bytes += (n_vp + n_rv) * 4;
  }
  mbar_arrive_expect_tx(bar, bytes);
  if (n_idx) bulk_load(buf + LY::kIdx, a.idx + ei, n_idx * 4, bar);
  if (!VCS && n_val)
    bulk_load(buf + LY::kVals, static_cast<const T *>(a.vals) + align_down<VPE>(k.e0),
              n_val * (int)sizeof(T), bar);
  if (n_ptr) bulk_load(buf + LY::kPtr, a.ptr + pi, n_ptr * 4, bar);
  if (VCS && n_vp) bulk_load(buf + LY::kVptr, a.vptr + ri, n_vp * 4, bar);
  if (VCS && n_rv)
    bulk_load(buf + LY::kRvals, static_cast<const float *>(a.vals) + ri, n_rv * 4, bar);
  if (a.xrows) {  // dense rows of the block's slices, into L2 (a hint; stays inside the rows)
    const int s_lo = k.s0, s_hi = k.type == 0 ? k.s1 : k.s0 + 1;
    const char *base = static_cast<const char *>(a.xrows);
    uintptr_t lo = reinterpret_cast<uintptr_t>(base + (int64_t)s_lo * a.xld * a.xes);
    uintptr_t hi =
        reinterpret_cast<uintptr_t>(base + ((int64_t)(s_hi - 1) * a.xld + a.xw) * a.xes);
    lo = (lo + 15) & ~uintptr_t(15);
    hi &= ~uintptr_t(15);
    if (s_hi > s_lo && hi > lo)
      prefetch_l2(reinterpret_cast<const void *>(lo), (uint32_t)(hi - lo));
  }
}

// Same, loading the descriptor of block number b from global memory.
template <typename T, bool VCS>
__device__ __forceinline__ void stage_issue(const StageArrays &a, int b, unsigned char *buf,
                                            uint64_t *bar) {
  const int4 d[3] = {a.blocks[3 * b], a.blocks[3 * b + 1], a.blocks[3 * b + 2]};
  stage_issue<T, VCS>(a, d, buf, bar);
}

template <typename T, bool VCS>
__device__ __forceinline__ Staged<T, VCS> stage_views(const Block &k, unsigned char *buf) {
  using LY = StageLayout<T, VCS>;
  constexpr int VPE = 16 / (int)sizeof(T);
  Staged<T, VCS> v;
  v.idx = reinterpret_cast<const int32_t *>(buf + LY::kIdx) - align_down<4>(k.e0);
  v.vals = VCS ? reinterpret_cast<const T *>(buf + LY::kEvals) - align_down<4>(k.e0)
               : reinterpret_cast<const T *>(buf + LY::kVals) - align_down<VPE>(k.e0);
  v.ptr = reinterpret_cast<const int32_t *>(buf + LY::kPtr) - align_down<4>(k.s0);
  v.vptr =
      VCS ? reinterpret_cast<const int32_t *>(buf + LY::kVptr) - align_down<4>(k.r0) : nullptr;
  v.rvals =
      VCS ? reinterpret_cast<const float *>(buf + LY::kRvals) - align_down<4>(k.r0) : nullptr;
  return v;
}

// The pipeline's shared-memory control words.
template <typename T, bool VCS, int NS = kStages>
struct Pipe {
  using PL = PipeLayout<T, VCS, NS>;
  unsigned char *smem;
  __device__ __forceinline__ unsigned char *buf(int s) const {
    return smem + PL::kBufs + s * StageLayout<T, VCS>::kBytes;
  }
  __device__ __forceinline__ uint64_t *full(int s) const {
    return reinterpret_cast<uint64_t *>(smem + PL::kFull) + s;
  }
  __device__ __forceinline__ uint64_t *empty(int s) const {
    return reinterpret_cast<uint64_t *>(smem + PL::kEmpty) + s;
  }
  __device__ __forceinline__ uint64_t *ready(int s) const {
    return reinterpret_cast<uint64_t *>(smem + PL::kReady) + s;
  }
  __device__ __forceinline__ int *fail() const { return reinterpret_cast<int *>(smem + PL::kFail); }
  __device__ __forceinline__ uint64_t *slab_landed() const {
    return reinterpret_cast<uint64_t *>(smem + PL::kSlab);
  }

  // All threads; contains __syncthreads.  `consumers`: warps that release
  // each buffer.
  __device__ __forceinline__ void init(int consumers = kWarpsPerCta) const {
    if (threadIdx.x == 0) {
      for (int s = 0; s < NS; ++s) {
        mbar_init(full(s), 1);
        mbar_init(empty(s), consumers);
        mbar_init(ready(s), 1);
      }
      mbar_init(slab_landed(), 1);
      *fail() = 0;
      fence_barrier_init();
    }
    __syncthreads();
  }

  __device__ __forceinline__ void give_up(const StageArrays &a) const {
    if ((threadIdx.x & 31) == 0) {
      atomicOr(fail(), 1);
      atomicOr(a.err, 1);
    }
  }

  // VCS, producer warp: block j (number b) has landed; write the run value of
  // each of its entries into the per-entry value array and mark the stage
  // ready.  A block of at most kFillRuns runs is filled run by run.
  // Otherwise run starts go into a bitmap over the block's entries; the run of
  // entry n is then r0 - 1 + (run starts in [e0, n]).  A warp scan of the
  // words' popcounts gives each word the runs started before it; the words
  // are then independent, so the final pass has no chain between words.
  __device__ __forceinline__ void expand(const StageArrays &a, int j, int b) const {
    using LY = StageLayout<T, VCS>;
    const int s = j % NS;
    const int lane = threadIdx.x & 31;
    unsigned char *bp = buf(s);
    const Block k = stage_desc<T, VCS>(bp);
    const int eb = align_down<4>(k.e0);
    const int32_t *vp = reinterpret_cast<const int32_t *>(bp + LY::kVptr) - align_down<4>(k.r0);
    const float *rv = reinterpret_cast<const float *>(bp + LY::kRvals) - align_down<4>(k.r0);
    float *ev = reinterpret_cast<float *>(bp + LY::kEvals) - eb;
    uint32_t *bm = reinterpret_cast<uint32_t *>(bp + LY::kBitmap);
    if (k.r1 - k.r0 <= kFillRuns) {
      // few (long) runs: fill each run's entries with its value directly
      for (int r = k.r0; r < k.r1; ++r) {
        const int lo = max(vp[r], k.e0), hi = min(vp[r + 1], k.e1);
        const float v = rv[r];
        for (int n = lo + lane; n < hi; n += 32) ev[n] = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready(s));
      return;
    }
    const int nwords = (k.e1 - eb + 31) / 32;
    for (int q = lane; q < nwords; q += 32) bm[q] = 0u;
    __syncwarp();
    for (int r = k.r0 + lane; r < k.r1; r += 32) {
      const int st = max(vp[r], k.e0) - eb;
      atomicOr(&bm[st >> 5], 1u << (st & 31));
    }
    __syncwarp();
    // 32 words at a time: lane l holds word q0 + l and the runs started
    // before it (a scan of the popcounts); the words then go round by shuffles
    const unsigned le = lanemask_lt() | (1u << lane);
    int base = k.r0 - 1;  // runs started before word q0
    for (int q0 = 0; q0 < nwords; q0 += 32) {
      const bool has = q0 + lane < nwords;
      const uint32_t mine = has ? bm[q0 + lane] : 0u;
      const int c = __popc(mine);
      int incl = c;  // inclusive scan of the popcounts over the lanes
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += y;
      }
      const int mybase = base + incl - c;
      const int nq = min(32, nwords - q0);
#pragma unroll 8
      for (int q = 0; q < nq; ++q) {
        const uint32_t word = __shfl_sync(kFullMask, mine, q);
        const int wbase = __shfl_sync(kFullMask, mybase, q);
        const int n = eb + 32 * (q0 + q) + lane;
        if (n >= k.e0 && n < k.e1) ev[n] = rv[wbase + __popc(word & le)];
      }
      base += __shfl_sync(kFullMask, incl, 31);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(ready(s));
  }

  // Producer warp (all lanes; lane 0 issues): fills the ring with blocks
  // b_begin, b_begin + step, ... < b_end, each once the consumers released
  // its buffer.  For VCS the warp also expands each block's run values as
  // soon as the block has landed: it polls both conditions, issuing first,
  // so copies stay in flight while it expands.  Every wait is bounded; before
  // returning it waits (bounded) until every issued copy has landed.
  __device__ __forceinline__ void produce(const StageArrays &a, int b_begin, int b_end,
                                          int step) const {
    const int lane = threadIdx.x & 31;
    const int total = b_end > b_begin ? (b_end - b_begin + step - 1) / step : 0;
    int issued = 0, done = 0;  // blocks issued, blocks expanded (VCS)
    bool ok = true;
    DescWindow win;
    auto issue = [&](int i) {
      int4 d[3];
      win.get(a.blocks, b_begin, step, b_end, i, d);
      if (lane == 0) {
        stage_issue<T, VCS>(a, d, buf(i % NS), full(i % NS));
      }
      __syncwarp();
    };
    if constexpr (!VCS) {
      for (; issued < total; ++issued) {
        const int s = issued % NS;
        if ((issued >= NS && !mbar_wait_bounded(empty(s), ((issued / NS) - 1) & 1, kWaitLimitNs)) ||
            *reinterpret_cast<volatile int *>(fail())) {
          ok = false;
          break;
        }
        issue(issued);
      }
    } else {
      int idle = 0;
      uint64_t t0 = 0;
      while (done < total) {
        bool moved = false;
        if (issued < total) {
          const int s = issued % NS;
          bool freed = issued < NS || mbar_test(empty(s), ((issued / NS) - 1) & 1);
          freed = __shfl_sync(kFullMask, freed, 0);
          if (freed) {
            issue(issued++);
            moved = true;
          }
        }
        if (done < issued) {
          bool landed = mbar_test(full(done % NS), (done / NS) & 1);
          landed = __shfl_sync(kFullMask, landed, 0);
          if (landed) {
            expand(a, done, b_begin + done * step);
            ++done;
            moved = true;
          }
        }
        if (moved) {
          idle = 0;
          continue;
        }
        if (idle++ == 0) t0 = global_ns();
        if ((idle & 63) == 0) {
          bool stop = *reinterpret_cast<volatile int *>(fail()) != 0 ||
                      global_ns() - t0 > kWaitLimitNs;
          stop = __shfl_sync(kFullMask, stop, 0);
          if (stop) {
            ok = false;
            break;
          }
        }
      }
    }
    if (!ok) give_up(a);
    if (lane == 0)
      for (int j = issued - NS < 0 ? 0 : issued - NS; j < issued; ++j)
        mbar_wait_bounded(full(j % NS), (j / NS) & 1, kWaitLimitNs);
  }

  // Split producer, issuing warp: issues every block in order, each once the
  // consumers released its buffer; before returning waits (bounded) until
  // every issued copy has landed.  The VCS run values are left to
  // expand_share.
  __device__ __forceinline__ void issue_all(const StageArrays &a, int b_begin, int b_end,
                                            int step) const {
    const int lane = threadIdx.x & 31;
    const int total = b_end > b_begin ? (b_end - b_begin + step - 1) / step : 0;
    DescWindow win;
    int issued = 0;
    bool ok = true;
    for (; issued < total; ++issued) {
      const int s = issued % NS;
      if ((issued >= NS && !mbar_wait_bounded(empty(s), ((issued / NS) - 1) & 1, kWaitLimitNs)) ||
          *reinterpret_cast<volatile int *>(fail())) {
        ok = false;
        break;
      }
      int4 d[3];
      win.get(a.blocks, b_begin, step, b_end, issued, d);
      if (lane == 0) {
        stage_issue<T, VCS>(a, d, buf(s), full(s));
      }
      __syncwarp();
    }
    if (!ok) give_up(a);
    if (lane == 0)
      for (int j = issued - NS < 0 ? 0 : issued - NS; j < issued; ++j)
        mbar_wait_bounded(full(j % NS), (j / NS) & 1, kWaitLimitNs);
  }

  // Split producer, expanding warp e of E (E divides NS, so the blocks of a
  // buffer always come to the same warp, in order, and a parity wait can never
  // see an older phase): expands blocks e, e + E, ... as they land.
  __device__ __forceinline__ void expand_share(const StageArrays &a, int b_begin, int b_end,
                                               int step, int e, int E) const {
    const int total = b_end > b_begin ? (b_end - b_begin + step - 1) / step : 0;
    for (int i = e; i < total; i += E) {
      if (!mbar_wait_bounded(full(i % NS), (i / NS) & 1, kWaitLimitNs) ||
          *reinterpret_cast<volatile int *>(fail())) {
        give_up(a);
        return;
      }
      expand(a, i, b_begin + i * step);
    }
  }

  // Consumer warp: waits for the i-th block of this CTA; false if the wait gave up.
  __device__ __forceinline__ bool acquire(int i, const StageArrays &a) const {
    uint64_t *bar = VCS ? ready(i % NS) : full(i % NS);
    if (mbar_wait_bounded(bar, (i / NS) & 1, kWaitLimitNs)) return true;
    give_up(a);
    return false;
  }

  // Consumer warp: done with the i-th block.
  __device__ __forceinline__ void release(int i) const {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty(i % NS));
  }
};

}  // namespace vs
