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
//   [256, 264)      u64 epoch counter of compress launches captured in a CUDA graph.
//   [264, 512)      reserved.
//   [512, ...)      u64 tile status[tiles], then TensorStart[T] (compress only).
// The status entries carry the epoch of the launch that wrote them (a number the host
// draws anew for every compress launch; a launch captured in a graph reads one more than
// the workspace's epoch counter and moves the counter on), so entries left by earlier
// launches never match and nothing needs clearing between calls.
struct Control {
  uint32_t error;       // first zvc_status latched on the device, 0 if none
  uint32_t pad;
  uint64_t error_info;  // tile or chunk index of that error
};
constexpr uint64_t kControlBytes = 256;
constexpr uint64_t kEpochOffset = 256;
constexpr uint64_t kStatusOffset = 512;

// Tile status word: the launch's epoch in bits 63..16 and the tile's payload units (an
// aggregate: at most 4224 four-byte or 4352 two-byte units) in bits 15..0.
constexpr uint32_t kAggBits = 16;
constexpr uint64_t kAggMask = (1ull << kAggBits) - 1;
constexpr uint64_t kEpochLimit = 1ull << (64 - kAggBits);

// A tensor's start in the payload (batched compress), published by the tensor's first
// tile: `value` first, then `tag` = epoch << 2 | flag with release semantics.
struct TensorStart {
  uint64_t value;  // payload words before the tensor
  uint64_t tag;
};
constexpr uint64_t kStartPrefix = 2;  // value is valid
constexpr uint64_t kStartError = 3;   // the first tile gave up

// Compress tiling: tiles of 4096 words (128 windows).
constexpr uint32_t kTileElems = 4096;
constexpr uint32_t kTileWindows = kTileElems / kWindow;

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s per device-side wait

__host__ __device__ inline uint64_t ceil_div_u64(uint64_t a, uint64_t b) {
  return a / b + (a % b != 0);
}

inline uint64_t round_up_u64(uint64_t a, uint64_t b) { return ceil_div_u64(a, b) * b; }

inline uint64_t tiles_for(uint64_t n) { return ceil_div_u64(n, kTileElems); }

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

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
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

// Bounded look-back over tile aggregates (after Merrill and Garland, "Single-pass
// Parallel Prefix Scan with Decoupled Look-back", 2016). Each tile publishes its aggregate
// (its payload words) in status[tile], tagged with the launch's epoch. A tile whose caller
// already knows the inclusive prefix of an earlier tile `floor` needs only the sum of the
// aggregates strictly between floor and itself. One pass reads 32*K of them: load j of
// lane l reads the tile at distance 32j + l + 1 below `top + 1`, so every warp load
// instruction reads 32 consecutive words. A window of at most one tile's words per entry
// sums in 32 bits (32*K * 4224 < 2^32 for K <= 31).
template <int K>
__device__ __forceinline__ void aggsum_issue(const uint64_t* status, uint64_t epoch, int64_t top,
                                             int64_t floor, uint32_t lane, uint64_t (&v)[K]) {
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int64_t idx = top - 32 * j - (int64_t)lane;
    v[j] = idx > floor ? ld_relaxed_u64(status + idx) : (epoch << kAggBits);  // a placeholder
  }
}

// Sum of the aggregates in (floor, tile) (warp-collective), starting from a pass `v`
// already issued with top = tile - 1. With SUFFIX it also sums those of the tiles at or
// above `from` into *suffix_out. Returns false (and latches ZVC_ERR_TIMEOUT) if an
// aggregate is still missing after limit_ns.
template <int K, bool SUFFIX = false>
__device__ __forceinline__ bool aggsum_finish(const uint64_t* status, uint64_t epoch, uint64_t tile,
                                              int64_t floor, uint32_t lane, uint64_t limit_ns,
                                              Control* ctl, uint64_t (&v)[K], uint64_t* sum_out,
                                              int64_t from = 0, uint64_t* suffix_out = nullptr) {
  uint64_t sum = 0, suffix = 0;
  int64_t top = (int64_t)tile - 1;
  WaitClock clock;
  while (top > floor) {
    bool missing = false;
    uint32_t part = 0, spart = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const int64_t idx = top - 32 * j - (int64_t)lane;
      if (idx > floor) {
        missing |= (v[j] >> kAggBits) != epoch;
        part += (uint32_t)(v[j] & kAggMask);
        if (SUFFIX && idx >= from) spart += (uint32_t)(v[j] & kAggMask);
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
      if (SUFFIX) suffix += __reduce_add_sync(0xffffffffu, spart);
      top -= 32 * K;
      if (top <= floor) break;
    }
    aggsum_issue<K>(status, epoch, top, floor, lane, v);
  }
  *sum_out = sum;
  if (SUFFIX) *suffix_out = suffix;
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
  const void* ptr;  // n words of 4 (or, for the 16-bit calls, 2) bytes
  uint64_t n;
};
struct TensorOut {
  void* ptr;  // n words of 4 (or, for the 16-bit calls, 2) bytes
  uint64_t n;
};

// Compress T tensors (T == 1 and !batched: a single stream) into `out`.
zvc_status launch_compress(const TensorIn* ts, uint32_t T, bool batched, uint32_t chunk_elems,
                           uint32_t* out, uint64_t out_words, uint64_t* out_size, uint8_t* ws,
                           uint64_t wait_limit_ns, cudaStream_t stream);

// Compress n 16-bit words into one stream at `out` (4-byte aligned; out_units 2-byte units).
zvc_status launch_compress16(const uint16_t* in, uint64_t n, uint32_t chunk_elems, uint16_t* out,
                             uint64_t out_units, uint64_t* out_size, uint8_t* ws,
                             uint64_t wait_limit_ns, cudaStream_t stream);

// Decompress a single stream (!batched, T == 1) or a batch of T streams.
zvc_status launch_decompress(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts,
                             uint32_t T, bool batched, uint32_t chunk_elems, uint8_t* ws,
                             cudaStream_t stream);

// Decompress one stream of 16-bit words (the stream at `in` is 4-byte aligned).
zvc_status launch_decompress16(const uint32_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n,
                               uint32_t chunk_elems, uint8_t* ws, cudaStream_t stream);

// RLE comparison codec (window of W words, 32 <= W <= ZVC_RLE_MAX_WINDOW).
uint64_t rle_ws_bytes(uint64_t n, uint32_t W);
zvc_status launch_rle_compress(const uint32_t* in, uint64_t n, uint32_t W, uint32_t* out,
                               uint64_t* out_size, uint8_t* ws, cudaStream_t stream);
zvc_status launch_rle_decompress(const uint32_t* in, uint64_t in_bytes, uint32_t* y, uint64_t n,
                                 uint32_t W, uint8_t* ws, cudaStream_t stream);

// Runs the look-back on a tile whose predecessor never publishes (in this launch's
// epoch), with the given limit; the wait must give up and latch ZVC_ERR_TIMEOUT. Used by
// the self-test entry point.
zvc_status launch_lookback_timeout_probe(uint8_t* ws, uint64_t limit_ns, cudaStream_t stream);

}  // namespace zvc
