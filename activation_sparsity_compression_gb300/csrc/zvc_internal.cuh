// Internal definitions shared by the ZVC kernels and the C-ABI layer (sm_103a).
//
// The stream format is the one documented in include/zvc.h: per 32-word window a 32-bit
// non-zero mask followed by the non-zero words (Rhu et al., "Compressing DMA Engine",
// section V.A), grouped into chunks indexed by a u64 offset table behind a 32-byte header.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zvc.h"

namespace zvc {

constexpr uint32_t kWindow = 32;
constexpr uint32_t kStreamMagic = 0x3143565Au;  // "ZVC1"
constexpr uint32_t kBatchMagic = 0x4243565Au;   // "ZVCB"
constexpr uint32_t kVersionWordBytes = 1u | (4u << 16);  // u16 version 1, u16 word_bytes 4
constexpr uint32_t kStreamHeaderWords = 8;      // 32 bytes
constexpr uint32_t kBatchHeaderWords = 4;       // 16 bytes

// Workspace layout (device memory owned by the caller, 256-byte aligned).
//   [0, 256)        Control: latched error, persists across calls until zvc_get_error.
//   [256, 512)      Counters: finished and failed tile counts, cleared by every call.
//   [512, ...)      u64 tile_status[tiles], then u64 tensor_start[T], cleared by every call.
struct Control {
  uint32_t error;       // first zvc_status latched on the device, 0 if none
  uint32_t pad;
  uint64_t error_info;  // tile or chunk index of that error
};
struct Counters {
  unsigned long long unused;
  unsigned long long done;    // tiles that have published their place
  unsigned long long failed;  // tiles that gave up
};
constexpr uint64_t kControlBytes = 256;
constexpr uint64_t kCountersBytes = 256;
constexpr uint64_t kPerCallOffset = kControlBytes;  // counters + status arrays start here
constexpr uint64_t kStatusOffset = kControlBytes + kCountersBytes;

// Look-back status word: 2-bit flag in bits 63..62, payload word count in bits 61..0.
constexpr uint64_t kFlagShift = 62;
constexpr uint64_t kFlagInvalid = 0;    // nothing published yet
constexpr uint64_t kFlagAggregate = 1;  // value = this tile's own compressed words
constexpr uint64_t kFlagPrefix = 2;     // value = compressed words of this tile and all before it
constexpr uint64_t kFlagError = 3;      // this tile gave up; successors give up too
constexpr uint64_t kValueMask = (1ull << kFlagShift) - 1;

// Compress tiling: one CTA of 256 threads per tile of 4096 words (128 windows); every
// thread holds 16 words as four 16-byte vectors.
constexpr int kCompressThreads = 256;
constexpr int kCompressWarps = kCompressThreads / 32;
constexpr uint32_t kTileElems = 4096;
constexpr uint32_t kTileWindows = kTileElems / kWindow;

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s per device-side wait

__host__ __device__ inline uint64_t ceil_div_u64(uint64_t a, uint64_t b) {
  return a / b + (a % b != 0);
}

inline uint64_t round_up_u64(uint64_t a, uint64_t b) { return ceil_div_u64(a, b) * b; }

inline uint64_t tiles_for(uint64_t n) { return ceil_div_u64(n, kTileElems); }

// Bytes of the per-call region (counters + tile status + tensor starts).
inline uint64_t per_call_bytes(uint64_t total_tiles, uint32_t T) {
  return kCountersBytes + 8 * total_tiles + 8 * (uint64_t)T;
}

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void latch_error(Control* ctl, uint32_t code, uint64_t info) {
  if (atomicCAS(&ctl->error, 0u, code) == 0u) {
    *reinterpret_cast<volatile uint64_t*>(&ctl->error_info) = info;
  }
}

// A bounded wait: returns false once limit_ns has passed since the first call. Between
// polls of global memory it sleeps briefly (16 ns, doubling up to 64 ns): long enough not
// to flood the L2 with polls, short enough that a waiter wakes soon after the flag flips.
struct WaitClock {
  uint64_t start = 0;
  uint32_t backoff = 16;
  __device__ __forceinline__ bool tick(uint64_t limit_ns) {
    const uint64_t now = globaltimer_ns();
    if (start == 0) start = now;
    if (now - start > limit_ns) return false;
    __nanosleep(backoff);
    if (backoff < 64) backoff <<= 1;
    return true;
  }
};

// Decoupled look-back (Merrill and Garland, "Single-pass Parallel Prefix Scan with
// Decoupled Look-back", 2016), warp-collective and wide: one pass reads 32*K predecessors. Load j of lane l reads the
// tile at distance 32j + l + 1, so each load instruction of the warp reads 32 consecutive
// status words (two cache lines): with every tile of a round looking back over the same
// few lines at once, uncoalesced reads would queue up on those L2 lines. The nearest
// inclusive prefix is the smallest distance with a prefix flag; every entry up to it
// counts. A pass can be issued early (lookback_issue) and evaluated later, so that its
// L2 round trip overlaps other work.
template <int K>
__device__ __forceinline__ void lookback_issue(const uint64_t* status, int64_t top, uint32_t lane,
                                               uint64_t (&s)[K], int64_t floor = -1,
                                               uint64_t floor_prefix = 0) {
  // Entries at or below `floor` are not read: the tile at `floor` acts as an inclusive
  // prefix of floor_prefix words (the caller's own earlier tile, or "nothing" at -1).
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int64_t idx = top - 32 * j - (int64_t)lane;
    s[j] = idx > floor ? ld_relaxed_u64(status + idx)
                       : ((kFlagPrefix << kFlagShift) | (idx == floor ? floor_prefix : 0));
  }
}

enum LookbackPassResult { kPassPrefix = 0, kPassAllAggregates = 1, kPassUnpublished = 2, kPassFailed = 3 };

// Evaluates one pass (warp-collective). On kPassPrefix / kPassAllAggregates, *part is the
// sum of the counted entries (the whole window for kPassAllAggregates). Aggregates are at
// most one tile of words each, so the aggregates of one window sum in 32 bits; only the
// nearest prefix needs 64.
template <int K>
__device__ __forceinline__ int lookback_eval(const uint64_t (&s)[K], uint32_t lane, uint64_t* part,
                                             uint32_t* prefix_dist = nullptr) {
  uint32_t jl = K;  // this lane's nearest prefix
#pragma unroll
  for (int j = K - 1; j >= 0; --j)
    if ((s[j] >> kFlagShift) == kFlagPrefix) jl = j;
  const uint32_t jstar = __reduce_min_sync(0xffffffffu, jl);
  const uint32_t lanes_at = __ballot_sync(0xffffffffu, jl == jstar);
  const uint32_t lstar = jstar < K ? (uint32_t)(__ffs(lanes_at) - 1) : 31u;
  bool unpublished = false, failed = false;
  uint32_t aggs = 0;
  uint64_t prefix = 0;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const bool counted = (uint32_t)j < jstar || ((uint32_t)j == jstar && lane <= lstar);
    if (counted) {
      const uint64_t f = s[j] >> kFlagShift;
      unpublished |= (f == kFlagInvalid);
      failed |= (f == kFlagError);
      if (f == kFlagPrefix) prefix = s[j] & kValueMask;
      else aggs += (uint32_t)(s[j] & kValueMask);
    }
  }
  if (__any_sync(0xffffffffu, failed)) return kPassFailed;
  if (__any_sync(0xffffffffu, unpublished)) return kPassUnpublished;
  aggs = __reduce_add_sync(0xffffffffu, aggs);
  if (jstar < K) {
    prefix = __shfl_sync(0xffffffffu, prefix, lstar);
    *part = prefix + aggs;
    if (prefix_dist) *prefix_dist = 32 * jstar + lstar + 1;  // distance below the pass's top + 1
    return kPassPrefix;
  }
  *part = aggs;
  return kPassAllAggregates;
}

// Completes the look-back of `tile` (warp-collective) starting from a pass `s` already
// issued for top = tile - 1 (with the same floor). On success *excl is the number of
// payload words in all tiles before `tile`. Returns false (and latches an error) if a predecessor failed or the wait
// ran past limit_ns.
template <int K>
__device__ __forceinline__ bool lookback_finish(uint64_t* status, uint64_t tile, uint32_t lane,
                                                uint64_t limit_ns, Control* ctl, uint64_t (&s)[K],
                                                uint64_t* excl, int64_t floor = -1,
                                                uint64_t floor_prefix = 0) {
  uint64_t sum = 0;
  int64_t top = (int64_t)tile - 1;
  WaitClock clock;
  while (true) {
    uint64_t part = 0;
    const int r = lookback_eval<K>(s, lane, &part);
    if (r == kPassFailed) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, tile);
      return false;
    }
    if (r == kPassUnpublished) {
      bool alive = true;
      if (lane == 0) alive = clock.tick(limit_ns);
      alive = __shfl_sync(0xffffffffu, alive, 0);
      if (!alive) {
        if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, tile);
        return false;
      }
    } else {
      sum += part;
      if (r == kPassPrefix) break;
      top -= 32 * K;
    }
    lookback_issue<K>(status, top, lane, s, floor, floor_prefix);
  }
  *excl = sum;
  return true;
}

// As lookback_finish, for a look-back bounded below by `floor`, the caller's own earlier
// tile, whose inclusive prefix may not be known yet: the floor is read as a prefix of 0
// words and *at_floor tells whether the walk ended there, in which case the caller adds
// the floor tile's inclusive prefix to *excl.
template <int K>
__device__ __forceinline__ bool lookback_to_floor(uint64_t* status, uint64_t tile, uint32_t lane,
                                                  uint64_t limit_ns, Control* ctl, uint64_t (&s)[K],
                                                  int64_t floor, uint64_t* excl, bool* at_floor) {
  uint64_t sum = 0;
  int64_t top = (int64_t)tile - 1;
  WaitClock clock;
  while (true) {
    uint64_t part = 0;
    uint32_t dist = 0;
    const int r = lookback_eval<K>(s, lane, &part, &dist);
    if (r == kPassFailed) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, tile);
      return false;
    }
    if (r == kPassUnpublished) {
      bool alive = true;
      if (lane == 0) alive = clock.tick(limit_ns);
      alive = __shfl_sync(0xffffffffu, alive, 0);
      if (!alive) {
        if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, tile);
        return false;
      }
    } else {
      sum += part;
      if (r == kPassPrefix) {
        *at_floor = (top + 1 - (int64_t)dist) == floor;
        break;
      }
      top -= 32 * K;
    }
    lookback_issue<K>(status, top, lane, s, floor, 0);
  }
  *excl = sum;
  return true;
}

template <int K>
__device__ __forceinline__ bool lookback_exclusive_wide(uint64_t* status, uint64_t tile,
                                                        uint32_t lane, uint64_t limit_ns,
                                                        Control* ctl, uint64_t* excl) {
  uint64_t s[K];
  lookback_issue<K>(status, (int64_t)tile - 1, lane, s);
  return lookback_finish<K>(status, tile, lane, limit_ns, ctl, s, excl);
}

// Bounded look-back over tile aggregates. Each tile publishes its aggregate (its payload
// words, at least 1, so 0 means "not yet") in aggs[tile]. A tile whose caller already
// knows the inclusive prefix of an earlier tile `floor` needs only the sum of the
// aggregates strictly between floor and itself. One pass reads 32*K of them: load j of
// lane l reads the tile at distance 32j + l + 1 below `top + 1`, so every warp load
// instruction reads 32 consecutive words. A window of at most one tile's words per entry
// sums in 32 bits (32*K * 4224 < 2^32 for K <= 31).
template <int K>
__device__ __forceinline__ void aggsum_issue(const uint32_t* aggs, int64_t top, int64_t floor,
                                             uint32_t lane, uint32_t (&v)[K]) {
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int64_t idx = top - 32 * j - (int64_t)lane;
    v[j] = idx > floor ? ld_relaxed_u32(aggs + idx) : 1u;  // below the floor: a placeholder
  }
}

// Sum of aggs(floor, tile) (warp-collective), starting from a pass `v` already issued with
// top = tile - 1. Returns false (and latches ZVC_ERR_TIMEOUT) if an aggregate is still
// missing after limit_ns.
template <int K>
__device__ __forceinline__ bool aggsum_finish(const uint32_t* aggs, uint64_t tile, int64_t floor,
                                              uint32_t lane, uint64_t limit_ns, Control* ctl,
                                              uint32_t (&v)[K], uint64_t* sum_out) {
  uint64_t sum = 0;
  int64_t top = (int64_t)tile - 1;
  WaitClock clock;
  while (top > floor) {
    bool missing = false;
    uint32_t part = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
      if (top - 32 * j - (int64_t)lane > floor) {
        missing |= (v[j] == 0u);
        part += v[j];
      }
    }
    if (__any_sync(0xffffffffu, missing)) {
      bool alive = true;
      if (lane == 0) alive = clock.tick(limit_ns);
      alive = __shfl_sync(0xffffffffu, alive, 0);
      if (!alive) {
        if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, tile);
        return false;
      }
    } else {
      sum += __reduce_add_sync(0xffffffffu, part);
      top -= 32 * K;
      if (top <= floor) break;
    }
    aggsum_issue<K>(aggs, top, floor, lane, v);
  }
  *sum_out = sum;
  return true;
}

// ------------------------------------------------------------------ mbarrier + TMA bulk
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// Suspend hint for mbarrier.try_wait: a waiting thread sleeps until the phase completes
// or this many nanoseconds pass, so a warp that waits long does not spin on the issue slots.
constexpr uint32_t kMbarSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "n"(kMbarSuspendNs)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete; false after limit_ns. try_wait
// itself suspends the thread in hardware until the phase completes or the suspend hint
// passes, so the loop only re-polls and checks the clock: no sleep that would delay the
// wake-up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - start > limit_ns) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared (TMA), completing `bytes` on the mbarrier. dst, src and
// bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Records e as this thread's last CUDA error and returns ZVC_ERR_CUDA.
zvc_status cuda_failure(cudaError_t e);

// Kernel tracing (zvc_trace_start / zvc_trace_stop): when enabled, every kernel launch
// is bracketed by CUDA events recorded on its own stream.
enum TraceKind { kTraceCompress = 0, kTraceDecompress = 1, kTraceKinds = 2 };
struct TraceMark {
  cudaEvent_t stop = nullptr;  // null when tracing is off
};
TraceMark trace_begin(int kind, cudaStream_t stream);
void trace_end(TraceMark m, cudaStream_t stream);

// ------------------------------------------------------------------ launch plans
struct TensorIn {
  const uint32_t* ptr;
  uint64_t n;
};
struct TensorOut {
  uint32_t* ptr;
  uint64_t n;
};

// Compress T tensors (T == 1 and !batched: a single stream) into `out`.
zvc_status launch_compress(const TensorIn* ts, uint32_t T, bool batched, uint32_t chunk_elems,
                           uint32_t* out, uint64_t out_words, uint64_t* out_size, uint8_t* ws,
                           uint64_t wait_limit_ns, cudaStream_t stream);

// Decompress a single stream (!batched, T == 1) or a batch of T streams.
zvc_status launch_decompress(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts,
                             uint32_t T, bool batched, uint32_t chunk_elems, uint8_t* ws,
                             cudaStream_t stream);

// Runs the look-back on a tile whose predecessor never publishes, with the given limit;
// the wait must give up and latch ZVC_ERR_TIMEOUT. Used by the self-test entry point.
zvc_status launch_lookback_timeout_probe(uint8_t* ws, uint64_t limit_ns, cudaStream_t stream);

}  // namespace zvc
