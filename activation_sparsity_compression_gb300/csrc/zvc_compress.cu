// ZVC compress for sm_103a (Rhu et al., "Compressing DMA Engine", section V.A: per 32-word
// window a 32-bit zero/non-zero mask followed by the non-zero words; section V.B: the
// compressed offsets are prefix sums of the masks' population counts).
//
// A tile is 4096 words. The kernel is persistent and launched cooperatively (every CTA is
// resident at once): CTA b compresses tiles b, b + G, b + 2G, ... (G = grid size) in that
// order, so each round of G tiles is compressed side by side and every tile a CTA waits
// for belongs to a running CTA. A producer lane streams the CTA's next tiles into a ring
// of shared-memory slots with 1-D TMA bulk copies while the tile in hand is processed.
// Per tile:
//   load    each warp reads 512 consecutive words from the slot as 16-byte vectors; lane l
//           of warp w holds words 512w + 128k + 4l .. +3 for k = 0..3
//   mask    lanes 8g..8g+7 hold window g of each 128-word group: a 4-bit nibble per lane,
//           OR-reduced over the 8 lanes by three shuffles (bit i = element i of the window)
//   scan    window sizes 1 + popc(mask) scanned over the 4 groups by two shuffles, over
//           the 4 groups of a warp in registers, over the 8 warps through shared memory
//   offset  a look-back over the published tile aggregates gives the tile's place in the
//           payload: the sum of the aggregates back to the CTA's own previous tile, plus
//           that tile's inclusive prefix; chunk starts inside the tile write their chunk_off
//   store   once the tile's place is known, each warp stores its windows straight from
//           registers: the mask, then the non-zero words at popc(mask & lanes below); the
//           words of one window are contiguous, so every store instruction is coalesced
//   header  the CTA owning the last tile writes the stream header(s) (and the batch
//           table) and the total byte count once that tile knows its place.
#include "zvc_internal.cuh"

namespace zvc {
namespace {

template <int MAXT>
struct CompressArgs {
  uint32_t* out;
  uint64_t out_words;
  uint64_t* out_size;
  uint8_t* ws;
  uint64_t total_tiles;
  uint64_t wait_limit_ns;
  uint64_t hdr_words_end;  // batch prefix + every stream's header and table, in words
  uint32_t chunk_elems;
  uint32_t T;
  uint32_t batched;
  int32_t wpc_log2;  // log2(chunk_elems / 32) when that is a power of two, else -1
  const uint32_t* in[MAXT];
  uint64_t n[MAXT];
  uint64_t tile_begin[MAXT + 1];  // first tile of tensor i; tile_begin[T] = total_tiles
  uint64_t hdr_before[MAXT];      // header/table words (and batch prefix) before stream i
  uint64_t payload_base[MAXT];    // hdr_before + this stream's header and table
};


using PerCallCounters = Counters;
static_assert(sizeof(PerCallCounters) <= kCountersBytes, "counter block");

__device__ __forceinline__ void put_u64_words(uint32_t* p, uint64_t v) {
  p[0] = (uint32_t)v;
  p[1] = (uint32_t)(v >> 32);
}

// Roles of the 14 warps of a CTA. Every role walks the CTA's tiles b, b+G, b+2G, ... in
// order. Tile i of the CTA is copied into input slot i % kInSlots; the mask warps read it
// there and release the slot at once, keeping only the tile's masks and offsets, in
// metadata slot i % kMetaSlots. The store warps later read the tile's words again from
// global memory, where the first read left them in L2. So the mask warps, and the tile
// aggregates they publish, run up to kMetaSlots tiles ahead of the stores, and a look-back
// rarely meets an unpublished predecessor. The roles hand a tile on through mbarriers:
//   full     (input slot) the producer's TMA copy has landed, or the slot holds a direct tile
//   masked   the 4 mask warps have written masks and offsets and published the aggregate
//   settled  a settle warp has found the tile's place in the payload
//   stored   the 8 store warps have written the tile out; the metadata slot is free
constexpr int kInSlots = 4;
constexpr int kMetaSlots = 16;
constexpr int kMaskWarps = 4;                       // warps 0..3
constexpr int kSettleWarp0 = 4;                     // warps 4, 5: even and odd tiles
constexpr int kSettleWarps = 2;
constexpr int kStoreWarp0 = 6;                      // warps 6..13
constexpr int kStoreWarps = 8;
constexpr int kRoleThreads = 32 * (kMaskWarps + kSettleWarps + kStoreWarps);  // 448
constexpr uint32_t kWinPerWarp = kTileWindows / kMaskWarps;      // 32 windows per mask warp
constexpr uint32_t kWinPerStoreWarp = kTileWindows / kStoreWarps;  // 16 windows per store warp
constexpr int kLookbackWidth = 10;  // one look-back pass covers 320 tiles: a round of tiles

struct SlotMeta {
  uint32_t mask[kTileWindows];
  uint32_t woff[kTileWindows];       // window offset inside its mask warp's 32 windows
  uint32_t wtot[kMaskWarps];         // payload words of each mask warp's 32 windows
  uint32_t agg, valid, ti, ok;
  uint64_t lt, dst, excl, pstart;
};

struct __align__(16) CompressShared {
  uint32_t in[kInSlots][kTileElems];  // input ring, filled by 1-D TMA bulk copies
  SlotMeta meta[kMetaSlots];
  uint64_t full[kInSlots];
  uint64_t masked[kMetaSlots], settled[kMetaSlots], stored[kMetaSlots];
  uint64_t handoff[2];               // settle warps: tile i's inclusive prefix is in incl[i % 2]
  uint64_t incl[2];
  uint32_t incl_ok[2];
  unsigned long long tile[kInSlots];
  uint32_t tensor[kInSlots];
  uint32_t direct[kInSlots];         // 1: slot not filled by TMA; the mask warps copy it in
  uint64_t pbuf[ZVC_MAX_BATCH + 1];  // stream starts, for the headers
};

template <int MAXT>
__device__ __forceinline__ uint32_t tensor_of_tile(const CompressArgs<MAXT>& a, uint64_t t) {
  uint32_t lo = 0;
  if (MAXT > 1) {
    uint32_t hi = a.T;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (a.tile_begin[mid] <= t) lo = mid; else hi = mid;
    }
  }
  return lo;
}

// Producer: starts the copy of tile t into ring slot s. Tiles that are not whole
// 16-byte-aligned 16 KB blocks (a tensor's ragged last tile, or a tensor whose base is
// not 16-byte aligned) are marked direct.
template <int MAXT>
__device__ __forceinline__ void fill_slot(const CompressArgs<MAXT>& a, CompressShared& sm, int s,
                                          unsigned long long t) {
  sm.tile[s] = t;
  if (t >= a.total_tiles) {
    sm.direct[s] = 1;
    mbar_arrive(&sm.full[s]);
    return;
  }
  const uint32_t ti = tensor_of_tile(a, t);
  sm.tensor[s] = ti;
  const uint64_t e0 = (t - a.tile_begin[ti]) * kTileElems;
  const uint32_t* src = a.in[ti] + e0;
  const bool whole = a.n[ti] - e0 >= kTileElems && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  sm.direct[s] = whole ? 0u : 1u;
  if (whole) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&sm.full[s], kTileElems * 4);
    bulk_g2s(sm.in[s], src, kTileElems * 4, &sm.full[s]);
  } else {
    mbar_arrive(&sm.full[s]);
  }
}

// Headers of every stream and the batch table (one warp). Runs once the last tile knows
// its place, which gives the total payload; `failed` is set when that tile gave up, in
// which case a failure upstream has been latched already.
template <int MAXT>
__device__ void finalize_warp(const CompressArgs<MAXT>& a, uint64_t total_payload, bool failed,
                              const uint64_t* tstart, Control* ctl, uint64_t* pbuf,
                              uint32_t lane) {
  int bad = failed;
  if (lane == 0) {
    // pbuf[i] = payload words before stream i; an empty tensor starts where the next
    // non-empty one does. A tensor's start is published by its first tile, which runs in
    // some CTA of this grid; wait (bounded) for it.
    uint64_t next = total_payload;
    pbuf[a.T] = total_payload;
    for (int i = (int)a.T - 1; i >= 0 && !bad; --i) {
      uint64_t p = next;
      if (a.tile_begin[i + 1] > a.tile_begin[i]) {
        p = 0;
        if (MAXT > 1) {
          WaitClock clock;
          while (true) {
            const uint64_t st = ld_relaxed_u64(tstart + i);
            if ((st >> kFlagShift) == kFlagPrefix) { p = st & kValueMask; break; }
            if ((st >> kFlagShift) == kFlagError || !clock.tick(a.wait_limit_ns)) {
              latch_error(ctl, ZVC_ERR_TIMEOUT, a.total_tiles);
              bad = 1;
              break;
            }
          }
        }
      }
      pbuf[i] = p;
      next = p;
    }
    if (bad && a.out_size) *a.out_size = 0;
  }
  bad = __shfl_sync(0xffffffffu, bad, 0);
  __syncwarp();
  if (bad) return;
  for (uint32_t i = lane; i < a.T; i += 32) {
    const uint64_t s0 = a.hdr_before[i] + pbuf[i];
    uint32_t* h = a.out + s0;
    h[0] = kStreamMagic;
    h[1] = kVersionWordBytes;
    h[2] = kWindow;
    h[3] = a.chunk_elems;
    put_u64_words(h + 4, a.n[i]);
    put_u64_words(h + 6, 4 * (pbuf[i + 1] - pbuf[i]));
    if (a.batched) put_u64_words(a.out + kBatchHeaderWords + 2 * i, 4 * s0);
  }
  if (lane == 0) {
    const uint64_t total_bytes = 4 * (a.hdr_words_end + total_payload);
    if (a.batched) {
      a.out[0] = kBatchMagic;
      a.out[1] = a.T;
      put_u64_words(a.out + 2, total_bytes);
      put_u64_words(a.out + kBatchHeaderWords + 2 * a.T, total_bytes);
    }
    if (a.out_size) *a.out_size = total_bytes;
  }
}

// Barrier of the four mask warps only (hardware barrier 1; barrier 0 is the CTA's).
__device__ __forceinline__ void mask_warps_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kMaskWarps * 32) : "memory");
}

// The same barrier, returning whether any mask thread passed `c`: keeps every mask warp on
// the same path, so none can leave while the others wait at the barrier.
__device__ __forceinline__ bool mask_warps_any(bool c) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)c), "n"(kMaskWarps * 32)
      : "memory");
  return r != 0;
}

// ---- mask warps: masks, in-warp offsets and the tile's aggregate
template <int MAXT>
__device__ void mask_role(const CompressArgs<MAXT>& a, CompressShared& sm, uint32_t* aggs,
                          Control* ctl, uint32_t warp, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  for (uint32_t i = 0;; ++i) {
    const int s = (int)(i % kInSlots);
    const int ms = (int)(i % kMetaSlots);
    bool late = false;
    if (i >= kMetaSlots)  // metadata slot free once tile i - kMetaSlots is stored
      late = !mbar_wait(&sm.stored[ms], ((i - kMetaSlots) / kMetaSlots) & 1u, a.wait_limit_ns);
    late = late || !mbar_wait(&sm.full[s], (i / kInSlots) & 1u, a.wait_limit_ns);
    if (mask_warps_any(late)) {
      if (warp == 0 && lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, i);
      return;
    }
    const uint64_t t = sm.tile[s];
    if (t >= a.total_tiles) return;
    const uint32_t ti = sm.tensor[s];
    const uint64_t lt = t - a.tile_begin[ti];
    const uint32_t valid = (uint32_t)min((uint64_t)kTileElems, a.n[ti] - lt * kTileElems);
    uint32_t* tile = sm.in[s];
    const uint32_t w0 = warp * kWinPerWarp;  // first window of this warp
    if (sm.direct[s]) {  // copy this warp's quarter of a ragged or unaligned tile in
      const uint32_t* src = a.in[ti] + lt * kTileElems;
      for (uint32_t k = w0 * kWindow + lane; k < (w0 + kWinPerWarp) * kWindow; k += 32)
        tile[k] = k < valid ? __ldcs(src + k) : 0u;
      __syncwarp();
    }
    // window j of this warp is words 32(w0 + j) ..; lane l reads word l, so the ballot is
    // the window's mask; lane j keeps window j's
    uint32_t my_mask = 0;
#pragma unroll 8
    for (uint32_t j = 0; j < kWinPerWarp; ++j) {
      const uint32_t b = __ballot_sync(0xffffffffu, tile[(w0 + j) * kWindow + lane] != 0u);
      my_mask = (lane == j) ? b : my_mask;
    }
    const uint32_t wsz = (w0 + lane) * kWindow < valid ? 1u + __popc(my_mask) : 0u;
    uint32_t incl = wsz;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += y;
    }
    SlotMeta& m = sm.meta[ms];
    m.mask[w0 + lane] = my_mask;
    m.woff[w0 + lane] = incl - wsz;
    if (lane == 31) m.wtot[warp] = incl;
    mask_warps_sync();  // the input slot is read and all four warp totals are in
    if (warp == 0 && lane == 0) {
      fill_slot(a, sm, s, t + kInSlots * G);  // the slot's next tile
      uint32_t agg = 0;
#pragma unroll
      for (int w = 0; w < kMaskWarps; ++w) agg += m.wtot[w];
      m.agg = agg;
      m.valid = valid;
      m.ti = ti;
      m.lt = lt;
      st_relaxed_u32(aggs + t, agg);  // publish the aggregate now
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.masked[ms]);
  }
}

// ---- settle warps: each tile's place in the payload. Tile i of the CTA follows the CTA's
// tile i-1 = t - G, whose inclusive prefix is known by then, so tile t needs only the
// aggregates of the G - 1 tiles in between, which every CTA's mask warps publish well
// ahead: no settle waits for another CTA's settle. Two warps take alternate tiles; each
// sums its window on its own and then adds the previous tile's inclusive prefix, handed
// over through shared memory.
template <int MAXT>
__device__ void settle_role(const CompressArgs<MAXT>& a, CompressShared& sm, uint32_t* aggs,
                            uint64_t* tstart, Control* ctl, uint32_t k, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  uint32_t lb[kLookbackWidth];
  uint32_t i = k;
  unsigned long long t = blockIdx.x + k * G;
  if (t < a.total_tiles)
    aggsum_issue<kLookbackWidth>(aggs, (int64_t)t - 1, i ? (int64_t)(t - G) : -1, lane, lb);
  for (; t < a.total_tiles; i += 2, t += 2 * G) {
    const int s = (int)(i % kMetaSlots);
    if (!mbar_wait(&sm.masked[s], (i / kMetaSlots) & 1u, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    SlotMeta& m = sm.meta[s];
    const uint32_t agg = m.agg, ti = m.ti;
    const uint64_t lt = m.lt;
    const int64_t floor = i ? (int64_t)(t - G) : -1;
    uint64_t excl = 0;
    bool ok = aggsum_finish<kLookbackWidth>(aggs, t, floor, lane, a.wait_limit_ns, ctl, lb, &excl);
    if (t + 2 * G < a.total_tiles)  // start this warp's next pass
      aggsum_issue<kLookbackWidth>(aggs, (int64_t)(t + 2 * G) - 1, (int64_t)(t + G), lane, lb);
    if (i > 0) {  // the CTA's previous tile, from the other settle warp
      const uint32_t h = (i - 1) & 1u;
      if (!mbar_wait(&sm.handoff[h], ((i - 1) / 2) & 1u, a.wait_limit_ns)) {
        if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
        return;
      }
      ok = ok && sm.incl_ok[h];
      excl += sm.incl[h];
    }
    __syncwarp();  // every lane has read the handoff before it is overwritten two tiles on
    if (lane == 0) {
      sm.incl[i & 1u] = excl + agg;
      sm.incl_ok[i & 1u] = ok;
      mbar_arrive(&sm.handoff[i & 1u]);
    }
    const uint64_t dst = a.payload_base[ti] + excl;
    if (ok && dst + agg > a.out_words) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_BUFFER_TOO_SMALL, t);
      ok = false;
    }
    if (lane == 0) {
      uint64_t pstart = 0;
      if (MAXT > 1) {
        if (lt == 0) {
          st_relaxed_u64(tstart + ti, ok ? ((kFlagPrefix << kFlagShift) | excl)
                                         : (kFlagError << kFlagShift));
          pstart = excl;
        } else if (ok) {
          // payload words before this tensor, published by its first tile (a lower tile)
          WaitClock clock;
          while (true) {
            const uint64_t st = ld_relaxed_u64(tstart + ti);
            const uint64_t f = st >> kFlagShift;
            if (f == kFlagPrefix) { pstart = st & kValueMask; break; }
            if (f == kFlagError || !clock.tick(a.wait_limit_ns)) {
              latch_error(ctl, ZVC_ERR_TIMEOUT, t);
              ok = false;
              break;
            }
          }
        }
      }
      m.dst = dst;
      m.excl = excl;
      m.pstart = pstart;
      m.ok = ok;
      mbar_arrive(&sm.settled[s]);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (t + 1 == a.total_tiles)  // the last tile: its place gives the total payload
      finalize_warp(a, ok ? excl + agg : 0, !ok, tstart, ctl, sm.pbuf, lane);
  }
}

// ---- store warps: each writes its 16 windows of the tile straight to the stream. The
// tile's words are read again from global memory (L2 after the producer's copy), as soon
// as the tile is masked, so the reads are in flight while the tile is settled.
template <int MAXT>
__device__ void store_role(const CompressArgs<MAXT>& a, CompressShared& sm, Control* ctl,
                           uint32_t sw, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  const uint32_t lane_below = (1u << lane) - 1u;
  const uint32_t w0 = sw * kWinPerStoreWarp;  // first window of this warp inside the tile
  const uint32_t mw = w0 / kWinPerWarp;       // the mask warp that scanned these windows
  unsigned long long t = blockIdx.x;
  for (uint32_t i = 0; t < a.total_tiles; ++i, t += G) {
    const int s = (int)(i % kMetaSlots);
    const uint32_t par = (i / kMetaSlots) & 1u;
    if (!mbar_wait(&sm.masked[s], par, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    const SlotMeta& m = sm.meta[s];
    const uint32_t valid = m.valid;
    const uint32_t* src = a.in[m.ti] + m.lt * kTileElems + w0 * kWindow;
    uint32_t v[kWinPerStoreWarp];
#pragma unroll
    for (uint32_t j = 0; j < kWinPerStoreWarp; ++j) {
      const uint32_t e = (w0 + j) * kWindow + lane;
      v[j] = e < valid ? __ldcs(src + j * kWindow + lane) : 0u;
    }
    if (!mbar_wait(&sm.settled[s], par, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    if (m.ok) {
      uint32_t wpre = 0;
#pragma unroll
      for (uint32_t w = 0; w < kMaskWarps; ++w) wpre += w < mw ? m.wtot[w] : 0u;
      uint32_t* g = a.out + m.dst + wpre;  // start of the mask warp's payload
      // lanes 0..15 own one window each: its mask, and the chunk table entry if it starts one
      if (lane < kWinPerStoreWarp && (w0 + lane) * kWindow < valid) {
        const uint32_t my_off = m.woff[w0 + lane];
        g[my_off] = m.mask[w0 + lane];
        const uint64_t wg = m.lt * kTileWindows + w0 + lane;  // window index in its tensor
        const uint32_t wpc = a.chunk_elems / kWindow;
        const bool starts = a.wpc_log2 >= 0 ? (wg & ((1ull << a.wpc_log2) - 1)) == 0 : wg % wpc == 0;
        if (starts) {
          const uint64_t c = a.wpc_log2 >= 0 ? (wg >> a.wpc_log2) : wg / wpc;
          put_u64_words(a.out + a.hdr_before[m.ti] + m.pstart + kStreamHeaderWords + 2 * c,
                        4 * (m.excl - m.pstart + wpre + my_off));
        }
      }
      const uint4* mq = reinterpret_cast<const uint4*>(&m.mask[w0]);
      const uint4* oq = reinterpret_cast<const uint4*>(&m.woff[w0]);
#pragma unroll
      for (uint32_t q = 0; q < kWinPerStoreWarp / 4; ++q) {
        const uint4 m4 = mq[q], o4 = oq[q];
        const uint32_t mm[4] = {m4.x, m4.y, m4.z, m4.w};
        const uint32_t oo[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
        for (uint32_t r = 0; r < 4; ++r) {
          const uint32_t j = 4 * q + r;
          if (v[j] != 0u) g[oo[r] + 1u + __popc(mm[r] & lane_below)] = v[j];
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.stored[s]);
  }
}

template <int MAXT>
__global__ void __launch_bounds__(kRoleThreads, 2)
    compress_kernel(const __grid_constant__ CompressArgs<MAXT> a) {
  extern __shared__ __align__(16) uint8_t dsmem[];
  CompressShared& sm = *reinterpret_cast<CompressShared*>(dsmem);
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  // per tile: its aggregate (u32), in the tile-status area of the workspace
  uint32_t* aggs = reinterpret_cast<uint32_t*>(a.ws + kStatusOffset);
  uint64_t* tstart = reinterpret_cast<uint64_t*>(a.ws + kStatusOffset) + a.total_tiles;
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;

  if (a.total_tiles == 0) {  // every tensor empty: headers only
    if (warp == 0) finalize_warp(a, 0, false, tstart, ctl, sm.pbuf, lane);
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kInSlots; ++s) mbar_init(&sm.full[s], 1);
    for (int s = 0; s < kMetaSlots; ++s) {
      mbar_init(&sm.masked[s], kMaskWarps);
      mbar_init(&sm.settled[s], 1);
      mbar_init(&sm.stored[s], kStoreWarps);
    }
    mbar_init(&sm.handoff[0], 1);
    mbar_init(&sm.handoff[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long G = gridDim.x;
  if (warp == 0 && lane == 0)
    for (int s = 0; s < kInSlots; ++s) fill_slot(a, sm, s, blockIdx.x + s * G);
  if (warp < kMaskWarps) mask_role(a, sm, aggs, ctl, warp, lane);
  else if (warp < kStoreWarp0) settle_role(a, sm, aggs, tstart, ctl, warp - kSettleWarp0, lane);
  else store_role(a, sm, ctl, warp - kStoreWarp0, lane);
}

__global__ void lookback_probe_kernel(uint8_t* ws, uint64_t limit_ns) {
  Control* ctl = reinterpret_cast<Control*>(ws);
  const uint32_t* aggs = reinterpret_cast<const uint32_t*>(ws + kStatusOffset);
  // tile 1 sums the aggregate of tile 0, which nothing publishes
  uint32_t v[kLookbackWidth];
  uint64_t sum = 0;
  aggsum_issue<kLookbackWidth>(aggs, 0, -1, threadIdx.x & 31u, v);
  aggsum_finish<kLookbackWidth>(aggs, 1, -1, threadIdx.x & 31u, limit_ns, ctl, v, &sum);
}

template <int MAXT>
zvc_status launch_t(const TensorIn* ts, uint32_t T, bool batched, uint32_t C, uint32_t* out,
                    uint64_t out_words, uint64_t* out_size, uint8_t* ws, uint64_t limit_ns,
                    cudaStream_t stream) {
  CompressArgs<MAXT> args;
  args.out = out;
  args.out_words = out_words;
  args.out_size = out_size;
  args.ws = ws;
  args.wait_limit_ns = limit_ns;
  args.chunk_elems = C;
  args.T = T;
  args.batched = batched ? 1u : 0u;
  const uint32_t wpc = C / kWindow;
  args.wpc_log2 = (wpc & (wpc - 1)) == 0 ? __builtin_ctz(wpc) : -1;
  uint64_t tiles = 0;
  uint64_t hdr = batched ? (kBatchHeaderWords + 2 * ((uint64_t)T + 1)) : 0;
  for (uint32_t i = 0; i < T; ++i) {
    args.in[i] = ts[i].ptr;
    args.n[i] = ts[i].n;
    args.tile_begin[i] = tiles;
    args.hdr_before[i] = hdr;
    tiles += tiles_for(ts[i].n);
    hdr += kStreamHeaderWords + 2 * ceil_div_u64(ts[i].n, C);
    args.payload_base[i] = hdr;
  }
  args.tile_begin[T] = tiles;
  args.total_tiles = tiles;
  args.hdr_words_end = hdr;

  static int resident = 0;  // CTAs of this kernel that fit on the device at once
  const int smem = (int)sizeof(CompressShared);
  cudaError_t e;
  if (resident == 0) {
    e = cudaFuncSetAttribute(compress_kernel<MAXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return cuda_failure(e);
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_failure(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_failure(e);
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compress_kernel<MAXT>,
                                                           kRoleThreads, smem)) != cudaSuccess)
      return cuda_failure(e);
    resident = sms * (per_sm > 0 ? per_sm : 1);
  }
  e = cudaMemsetAsync(ws + kPerCallOffset, 0, per_call_bytes(tiles, T), stream);
  if (e != cudaSuccess) return cuda_failure(e);
  const uint64_t grid = tiles == 0 ? 1 : (tiles < (uint64_t)resident ? tiles : (uint64_t)resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kRoleThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident together
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const TraceMark mark = trace_begin(kTraceCompress, stream);
  e = cudaLaunchKernelEx(&cfg, compress_kernel<MAXT>, args);
  trace_end(mark, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

}  // namespace

zvc_status launch_compress(const TensorIn* ts, uint32_t T, bool batched, uint32_t chunk_elems,
                           uint32_t* out, uint64_t out_words, uint64_t* out_size, uint8_t* ws,
                           uint64_t wait_limit_ns, cudaStream_t stream) {
  if (!batched && T == 1)
    return launch_t<1>(ts, T, false, chunk_elems, out, out_words, out_size, ws, wait_limit_ns,
                       stream);
  if (T <= 64)
    return launch_t<64>(ts, T, batched, chunk_elems, out, out_words, out_size, ws, wait_limit_ns,
                        stream);
  return launch_t<ZVC_MAX_BATCH>(ts, T, batched, chunk_elems, out, out_words, out_size, ws,
                                 wait_limit_ns, stream);
}

zvc_status launch_lookback_timeout_probe(uint8_t* ws, uint64_t limit_ns, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws + kPerCallOffset, 0, per_call_bytes(2, 1), stream);
  if (e != cudaSuccess) return cuda_failure(e);
  lookback_probe_kernel<<<1, 32, 0, stream>>>(ws, limit_ns);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

}  // namespace zvc
