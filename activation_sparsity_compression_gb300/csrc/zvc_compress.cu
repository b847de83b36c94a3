// ZVC compress for sm_103a (Rhu et al., "Compressing DMA Engine", section V.A: per 32-word
// window a 32-bit zero/non-zero mask followed by the non-zero words; section V.B: the
// compressed offsets are prefix sums of the masks' population counts).
//
// A tile is 4096 words (128 windows). The kernel is persistent and launched cooperatively
// (every CTA is resident at once, one per SM): CTA b compresses tiles b, b + G, b + 2G, ...
// (G = grid size) in that order, so every tile a CTA waits for belongs to a running CTA.
// Each CTA keeps a ring of shared-memory slots; a tile's slot goes through four roles:
//   load    a 1-D TMA bulk copy brings the tile's 16 KB into the slot, 128 words in
//   pack    a team of 8 warps takes the tile, 16 windows each: every warp reads its
//           windows' words into registers and takes a ballot per window (the window's mask);
//           the sizes 1 + popc(mask) give each window's place, the team's 8 totals (through
//           shared memory) each warp's base, and popc(mask & lanes below) each word's place
//           inside its window. After a team barrier (every word read) the masks and non-zero
//           words are written back into the same slot, packed from word 0; a warp with very
//           few (or very many) non-zero words skips the empty windows' value stores. The
//           tile's packed size (its aggregate) is published to the other CTAs before the
//           writes.
//   settle  the tile's place in the payload: the CTA's previous tile t - G has its inclusive
//           prefix already, so only the aggregates of the G - 1 tiles in between are summed
//           (no settle waits for another CTA's settle); two warps take alternate tiles and
//           hand the inclusive prefix on through shared memory
//   store   one warp copies the packed tile to its place with coalesced 16-byte stores,
//           writes the chunk table entries of chunks that start in the tile, and starts the
//           copy of the slot's next tile
// The CTA owning the last tile writes the stream header(s), the batch table and the total
// byte count once that tile knows its place.
#include <atomic>
#include <random>

#include "zvc_internal.cuh"

namespace zvc {
namespace {

// WB is the word size in bytes: 4 (any 32-bit type) or 2 (bf16 / fp16). Positions in the
// stream are counted in units of one word: a mask is 4 / WB units.
template <int WB> struct WordOf;
template <> struct WordOf<4> { using T = uint32_t; };
template <> struct WordOf<2> { using T = uint16_t; };

template <int MAXT, int WB>
struct CompressArgs {
  using Word = typename WordOf<WB>::T;
  Word* out;
  uint64_t out_words;  // units of WB bytes
  uint64_t* out_size;
  uint8_t* ws;
  uint64_t total_tiles;
  uint64_t wait_limit_ns;
  uint64_t epoch;          // tags this launch's entries in the workspace (host-drawn)
  uint64_t hdr_words_end;  // batch prefix + every stream's header and table, in units
  uint32_t chunk_elems;
  uint32_t T;
  uint32_t batched;
  uint32_t inner_chunks;  // 1 when chunks can start inside a tile (C not a multiple of 4096)
  const Word* in[MAXT];
  uint64_t n[MAXT];
  uint64_t tile_begin[MAXT + 1];  // first tile of tensor i; tile_begin[T] = total_tiles
  uint64_t hdr_before[MAXT];      // header/table units (and batch prefix) before stream i
  uint64_t payload_base[MAXT];    // hdr_before + this stream's header and table
};


__device__ __forceinline__ void put_u64_words(uint32_t* p, uint64_t v) {
  p[0] = (uint32_t)v;
  p[1] = (uint32_t)(v >> 32);
}

// Warp roles. Tile i of the CTA uses slot i % kSlots and is packed by team i % kTeams,
// settled by settle warp i % 2 and stored by store warp i % kStoreWarps; kSlots is a
// multiple of all three, so a slot always meets the same warps. The slot's mbarriers:
//   full     the TMA copy has landed (or the tile is read from global memory directly)
//   packed   the 8 warps of the pack team have written the packed tile
//   settled  a settle warp has found the tile's place in the payload
// The store warp that empties a slot starts its refill, so no barrier marks it empty.
constexpr int kSlots = 12;
constexpr uint32_t kInOffset = kTileWindows;                 // input lands 128 words in
// Slot words: the input lands 512 bytes in; a dense tile packs into 512 + 4096 WB bytes
// (4224 words for WB = 4, 2176 for WB = 2), which is the slot.
constexpr uint32_t slot_words(int wb) { return kInOffset + kTileElems * (uint32_t)wb / 4u; }
constexpr int kTeamWarps = 8;                                // a pack team: 16 windows per warp
constexpr int kTeams = 2;                                    // warps 0..7 and 8..15
constexpr uint32_t kWinPerWarp = kTileWindows / kTeamWarps;  // 32
constexpr int kSettleWarp0 = kTeams * kTeamWarps;            // warps 16, 17
constexpr int kSettleWarps = 2;
constexpr int kStoreWarp0 = kSettleWarp0 + kSettleWarps;     // warps 18..20
constexpr int kStoreWarps = 3;
constexpr int kRoleThreads = 32 * (kStoreWarp0 + kStoreWarps);  // 672
constexpr int kFirstFills = 2;     // slots filled at the start; the rest follow the first tile
constexpr int kLookbackWidth = 5;  // one look-back pass covers 160 tiles: a round of tiles
static_assert(kSlots % kTeams == 0 && kSlots % kSettleWarps == 0 && kSlots % kStoreWarps == 0,
              "a slot must always meet the same warps");
static_assert(kWinPerWarp * kTeamWarps == kTileWindows && kWinPerWarp <= 32, "a team covers a tile");

struct SlotInfo {
  uint64_t lt;          // tile index inside its tensor
  uint64_t dst;         // word address of the packed tile in the output
  uint64_t excl;        // payload words before the tile (all streams)
  uint64_t pstart;      // payload words before the tile's stream
  uint32_t ti;          // tensor
  uint32_t direct;      // 1: not brought in by TMA; the pack warp reads global memory
  uint32_t valid;       // words of the tile inside its tensor
  uint32_t agg;         // packed words
  uint32_t ok;
  uint32_t pad;
};

template <int WB>
struct __align__(16) CompressShared {
  uint32_t slot[kSlots][slot_words(WB)];
  uint32_t woff[kSlots][kTileWindows];  // window offsets, kept only when chunks start inside tiles
  SlotInfo info[kSlots];
  uint32_t team_tot[kTeams][2][kTeamWarps];  // pack warps' payload words, double-buffered
  uint64_t full[kSlots], packed[kSlots], settled[kSlots];
  uint64_t handoff[2];  // settle warps: tile i's inclusive prefix is in incl[i % 2]
  uint64_t incl[2];
  uint32_t incl_ok[2];
  uint32_t incl_ti[2];   // ... and its tensor, and that tensor's start in the payload
  uint64_t incl_pstart[2];
  uint64_t pbuf[ZVC_MAX_BATCH + 1];  // stream starts, for the headers
  uint64_t epoch;                    // a captured launch's epoch, read at its start
  uint64_t epoch_bar;                // completes once `epoch` is set (captured launches)
};

static_assert(sizeof(CompressShared<4>) <= 227 * 1024, "one CTA per SM must fit");

template <int MAXT, int WB>
__device__ __forceinline__ uint32_t tensor_of_tile(const CompressArgs<MAXT, WB>& a, uint64_t t) {
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

// Starts bringing tile t into slot s (one thread). Tiles that are not whole 16-byte-aligned
// 16 KB blocks (a tensor's ragged last tile, or a tensor whose base is not 16-byte aligned)
// are marked direct: the pack warp reads them from global memory.
template <int MAXT, int WB>
__device__ __forceinline__ void fill_slot(const CompressArgs<MAXT, WB>& a, CompressShared<WB>& sm, int s,
                                          unsigned long long t) {
  if (t >= a.total_tiles) return;
  const uint32_t ti = tensor_of_tile(a, t);
  const uint64_t lt = t - a.tile_begin[ti];
  const uint64_t e0 = lt * kTileElems;
  const typename CompressArgs<MAXT, WB>::Word* src = a.in[ti] + e0;
  const uint64_t left = a.n[ti] - e0;
  const bool whole = left >= kTileElems && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  SlotInfo& f = sm.info[s];
  f.ti = ti;
  f.lt = lt;
  f.valid = (uint32_t)(left < kTileElems ? left : kTileElems);
  f.direct = whole ? 0u : 1u;
  if (whole) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&sm.full[s], kTileElems * WB);
    bulk_g2s(&sm.slot[s][kInOffset], src, kTileElems * WB, &sm.full[s]);
  } else {
    mbar_arrive(&sm.full[s]);
  }
}

// Headers of every stream and the batch table (one warp). Runs once the last tile knows
// its place, which gives the total payload; `failed` is set when that tile gave up, in
// which case a failure upstream has been latched already.
// A tensor's start in the payload, published by its first tile in this launch (bounded
// wait); false if that tile gave up or the wait ran out.
template <int MAXT, int WB>
__device__ bool wait_tensor_start(const CompressArgs<MAXT, WB>& a, uint64_t epoch,
                                  const TensorStart* ts, Control* ctl, uint64_t info,
                                  uint64_t* value) {
  WaitClock clock;
  while (true) {
    const uint64_t tag = ld_acquire_u64(&ts->tag);
    if ((tag >> 2) == epoch) {
      if ((tag & 3u) == kStartPrefix) {
        *value = ld_relaxed_u64(&ts->value);
        return true;
      }
      break;
    }
    if (!clock.tick(a.wait_limit_ns)) break;
  }
  latch_error(ctl, ZVC_ERR_TIMEOUT, info);
  return false;
}

template <int MAXT, int WB>
__device__ void finalize_warp(const CompressArgs<MAXT, WB>& a, uint64_t epoch,
                              uint64_t total_payload, bool failed, const TensorStart* tstart,
                              Control* ctl, uint64_t* pbuf, uint32_t lane) {
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
        if (MAXT > 1 && !wait_tensor_start(a, epoch, tstart + i, ctl, a.total_tiles, &p)) bad = 1;
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
    uint32_t* h = reinterpret_cast<uint32_t*>(a.out + s0);  // 4-byte aligned: see launch_t
    h[0] = kStreamMagic;
    h[1] = 1u | ((uint32_t)WB << 16);  // u16 version 1, u16 word_bytes
    h[2] = kWindow;
    h[3] = a.chunk_elems;
    put_u64_words(h + 4, a.n[i]);
    put_u64_words(h + 6, WB * (pbuf[i + 1] - pbuf[i]));
    if (a.batched)
      put_u64_words(reinterpret_cast<uint32_t*>(a.out) + kBatchHeaderWords + 2 * i, WB * s0);
  }
  if (lane == 0) {
    const uint64_t total_bytes = WB * (a.hdr_words_end + total_payload);
    if (a.batched) {
      uint32_t* b = reinterpret_cast<uint32_t*>(a.out);
      b[0] = kBatchMagic;
      b[1] = a.T;
      put_u64_words(b + 2, total_bytes);
      put_u64_words(b + kBatchHeaderWords + 2 * a.T, total_bytes);
    }
    if (a.out_size) *a.out_size = total_bytes;
  }
}

// ---- epochs. A launch outside a stream capture tags its workspace entries with the epoch
// the host drew for it (CompressArgs::epoch: a process-wide counter started between 2^39
// and 2^40). A launch captured in a CUDA graph is replayed with the arguments of its
// capture, so it reads its epoch on the device instead: one more than the workspace's
// epoch counter, read by every CTA at its start (by a store warp, idle until the first
// tile is settled) and moved on once every CTA has read it (settle_role, tile G - 1). Its
// epochs are 1, 2, ... in a fresh workspace: never the 0 of an unwritten status word,
// never a host-drawn epoch, and a new one on every replay.
template <bool CAPTURED, int MAXT, int WB>
__device__ __forceinline__ uint64_t launch_epoch(const CompressArgs<MAXT, WB>& a, uint64_t dev) {
  return CAPTURED ? dev : a.epoch;
}

// ---- pack teams
// Barrier of one pack team (hardware barriers 1 and 2; barrier 0 is the CTA's), returning
// whether any of its threads passed `c`, so that all four warps take the same path.
__device__ __forceinline__ bool team_any(uint32_t team, bool c) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)c), "r"(1u + team), "n"(kTeamWarps * 32)
      : "memory");
  return r != 0;
}

// Writes one window (this lane's word v, the window's mask m) at unit pos of the slot and
// returns the position after it. A mask is 4 / WB units; with WB = 2 lanes 0 and 1 store
// its two halves, since it need not start on a 4-byte boundary.
template <int WB>
__device__ __forceinline__ uint32_t pack_window(uint32_t* slot, uint32_t pos, uint32_t v,
                                                uint32_t m, uint32_t lane, uint32_t lane_below) {
  using Word = typename WordOf<WB>::T;
  constexpr uint32_t mu = 4u / WB;
  Word* u = reinterpret_cast<Word*>(slot);
  if (v != 0u) u[pos + mu + __popc(m & lane_below)] = (Word)v;
  if (WB == 4) {
    if (lane == 0) u[pos] = (Word)m;
  } else if (lane < 2) {
    u[pos + lane] = (Word)(m >> (16u * lane));
  }
  return pos + mu + __popc(m);
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((unsigned short)v) : "memory");
}

// One packed word (WB bytes) at a shared-memory byte address.
template <int WB>
__device__ __forceinline__ void st_shared_word(uint32_t addr, uint32_t v) {
  if (WB == 4) st_shared_u32(addr, v);
  else st_shared_u16(addr, v);
}

// A window's mask at a shared-memory byte address: lane 0 stores it whole (WB = 4); with
// WB = 2 it may sit on a 2-byte boundary, and lanes 0 and 1 store its halves.
template <int WB>
__device__ __forceinline__ void st_shared_mask(uint32_t addr, uint32_t m, uint32_t lane) {
  if (WB == 4) {
    if (lane == 0) st_shared_u32(addr, m);
  } else if (lane < 2) {
    st_shared_u16(addr + 2u * lane, m >> (16u * lane));
  }
}

// Writes this warp's windows of a whole tile into the slot from unit pos on: per window one
// store of the non-zero words, each at its rank among the window's set bits, and one of the
// mask. Addresses are 32-bit shared-memory byte addresses, and each window's own mask
// bytes (4j for window j) are an immediate of its stores, so the running address only adds
// the non-zero words of the windows before. With SKIP a warp-uniform branch passes
// over an empty window, which is its mask alone: fewer instructions where most windows are
// empty, and (measured) faster where none is; between those the plain loop wins. With WOFF
// lane 0 also records each window's word offset, for chunks that start inside the tile.
template <int WB, bool SKIP, bool WOFF>
__device__ __forceinline__ void pack_whole(uint32_t slot_addr, uint32_t pos,
                                           const uint32_t (&v)[kWinPerWarp],
                                           const uint32_t (&m)[kWinPerWarp], uint32_t lane,
                                           uint32_t lane_below, uint32_t* woff) {
  constexpr uint32_t B = (uint32_t)WB;
  uint32_t acc = slot_addr + B * pos;
#pragma unroll
  for (uint32_t j = 0; j < kWinPerWarp; ++j) {
    if (WOFF && lane == 0) woff[j] = (acc - slot_addr) / B + (4u / B) * j;
    if (SKIP) {
      st_shared_mask<WB>(acc + 4u * j, m[j], lane);
      if (m[j] != 0u) {
        if (v[j] != 0u) st_shared_word<WB>(acc + B * __popc(m[j] & lane_below) + 4u * j + 4u, v[j]);
        acc += B * __popc(m[j]);
      }
    } else {
      if (v[j] != 0u) st_shared_word<WB>(acc + B * __popc(m[j] & lane_below) + 4u * j + 4u, v[j]);
      st_shared_mask<WB>(acc + 4u * j, m[j], lane);
      acc += B * __popc(m[j]);
    }
  }
}

// A warp whose non-zero words number at most kSkipBelow or at least kSkipAbove (of 512)
// packs with the empty-window branch (measured on 2^28-word maps: 0.79 against 0.70 of HBM
// at 0-1% density, 0.96 against 0.91 at 100%); the others without it (0.72 against 0.68
// at 10%).
constexpr uint32_t kSkipBelow = 16;
constexpr uint32_t kSkipAbove = 320;

template <int MAXT, int WB, bool INNER, bool CAPTURED>
__device__ void pack_role(const CompressArgs<MAXT, WB>& a, CompressShared<WB>& sm, uint64_t* status,
                          Control* ctl, uint32_t team, uint32_t q, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  const uint32_t lane_below = (1u << lane) - 1u;
  const bool keep_woff = INNER && a.inner_chunks != 0;
  // window offsets of every window, or (chunks of a multiple of 512 elements, whose starts
  // fall on warps' first windows) of each warp's first window only
  const bool woff_each = keep_woff && a.chunk_elems % (kWinPerWarp * kWindow) != 0;
  const uint32_t w0 = q * kWinPerWarp;  // this warp's first window
  // a captured launch: the team's first warp, which publishes the aggregates, waits for
  // the epoch first (a wait that runs out makes it late for its first tile, so the team
  // gives the tile up together)
  uint64_t dev_epoch = 0;
  bool epoch_ok = true;
  if (CAPTURED && q == 0) {
    epoch_ok = mbar_wait(&sm.epoch_bar, 0u, a.wait_limit_ns);
    dev_epoch = sm.epoch;
  }
  uint32_t round = 0;
  for (uint32_t i = team;; i += kTeams, ++round) {
    const unsigned long long t = blockIdx.x + (unsigned long long)i * G;
    if (t >= a.total_tiles) return;
    const int s = (int)(i % kSlots);
    // a warp whose wait ran out reads nothing; the team learns of it at its barrier below
    const bool late = !mbar_wait(&sm.full[s], (i / kSlots) & 1u, a.wait_limit_ns) || !epoch_ok;
    const SlotInfo& f = sm.info[s];
    uint32_t* slot = sm.slot[s];
    // read: this lane's word of each of the warp's 16 windows
    uint32_t v[kWinPerWarp];
    uint32_t nwin = kTileWindows;
    if (late) {
#pragma unroll
      for (uint32_t j = 0; j < kWinPerWarp; ++j) v[j] = 0u;
    } else if (!f.direct) {
      const typename CompressArgs<MAXT, WB>::Word* in =
          reinterpret_cast<const typename CompressArgs<MAXT, WB>::Word*>(slot + kInOffset);
#pragma unroll
      for (uint32_t j = 0; j < kWinPerWarp; ++j) v[j] = in[(w0 + j) * kWindow + lane];
    } else {  // read from global memory; a ragged tile has fewer windows
      const typename CompressArgs<MAXT, WB>::Word* src = a.in[f.ti] + f.lt * kTileElems;
      const uint32_t valid = f.valid;
      nwin = (valid + kWindow - 1) / kWindow;
#pragma unroll
      for (uint32_t j = 0; j < kWinPerWarp; ++j) {
        const uint32_t e = (w0 + j) * kWindow + lane;
        v[j] = e < valid ? __ldcs(src + e) : 0u;
      }
    }
    // masks and the warp's payload words: a mask per window it holds (the windows past a
    // ragged tile's end hold only zeros, so they add no words) and every non-zero word,
    // counted per lane and summed over the warp
    uint32_t m[kWinPerWarp];
    uint32_t nz = 0;
#pragma unroll
    for (uint32_t j = 0; j < kWinPerWarp; ++j) {
      m[j] = __ballot_sync(0xffffffffu, v[j] != 0u);
      nz += v[j] != 0u ? 1u : 0u;
    }
    const uint32_t held = nwin > w0 ? min(nwin - w0, kWinPerWarp) : 0u;
    const uint32_t tot = held * (4u / WB) + __reduce_add_sync(0xffffffffu, nz);
    uint32_t* tt = sm.team_tot[team][round & 1u];
    if (lane == 0) tt[q] = tot;
    // every word of the tile is read and every warp total is in; a late warp gives up the
    // team's tile here, all its warps together
    if (team_any(team, late)) {
      if (q == 0 && lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    // lane r < kTeamWarps reads warp r's total: the warp's base and the tile's aggregate
    const uint32_t x = lane < kTeamWarps ? tt[lane] : 0u;
    const uint32_t pos0 = __reduce_add_sync(0xffffffffu, lane < q ? x : 0u);
    const uint32_t agg = __reduce_add_sync(0xffffffffu, x);
    uint32_t pos = pos0;
    if (q == 0 && lane == 0) {
      // publish the aggregate now
      st_relaxed_u64(status + t, (launch_epoch<CAPTURED>(a, dev_epoch) << kAggBits) | agg);
      sm.info[s].agg = agg;
    }
    // write back, packed (a store of the non-zero words and one of the mask per window,
    // which costs fewer instructions than folding the mask into the lanes holding a zero)
    const uint32_t nzw = tot - held * (4u / WB);  // the warp's non-zero words
    const uint32_t sa = smem_addr(slot);
    uint32_t* woff = sm.woff[s] + w0;
    // (the order of these branches is measured: with the plain loop first the 5-25% maps
    // gain 2% and the 0-1% ones lose 4-6%, which leaves every density above 0.7 of HBM)
    // chunks of a multiple of 512 elements start only at a warp's first window: its base
    if (keep_woff && lane == 0) woff[0] = pos;
    if (nwin == kTileWindows && !woff_each && nzw > kSkipBelow && nzw < kSkipAbove) {
      pack_whole<WB, false, false>(sa, pos, v, m, lane, lane_below, woff);
    } else if (nwin == kTileWindows && !woff_each) {
      pack_whole<WB, true, false>(sa, pos, v, m, lane, lane_below, woff);
    } else if (INNER && nwin == kTileWindows) {  // chunks start inside tiles: offsets kept
      // one loop only: every unrolled copy of the loop in a kernel slows all of them
      pack_whole<WB, false, true>(sa, pos, v, m, lane, lane_below, woff);
    } else {  // a ragged tile
#pragma unroll
      for (uint32_t j = 0; j < kWinPerWarp; ++j) {
        if (w0 + j < nwin) {
          if (keep_woff && lane == 0) sm.woff[s][w0 + j] = pos;
          pos = pack_window<WB>(slot, pos, v[j], m[j], lane, lane_below);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.packed[s]);
  }
}

// ---- settle warps: each tile's place in the payload. Tile i of the CTA follows the CTA's
// tile i-1 = t - G, whose inclusive prefix is known by then, so tile t needs only the
// aggregates of the G - 1 tiles in between, which every CTA's pack warps publish well
// ahead: no settle waits for another CTA's settle. Two warps take alternate tiles; each
// sums its window on its own and then adds the previous tile's inclusive prefix, handed
// over through shared memory.
template <int MAXT, int WB, bool CAPTURED>
__device__ void settle_role(const CompressArgs<MAXT, WB>& a, CompressShared<WB>& sm, const uint64_t* status,
                            TensorStart* tstart, Control* ctl, uint32_t k, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  uint64_t lb[kLookbackWidth];
  uint32_t i = k;
  unsigned long long t = blockIdx.x + k * G;
  // (the entries a pass holds below its floor are never read, so a captured launch's
  // first pass goes out before its epoch is known)
  if (t < a.total_tiles)
    aggsum_issue<kLookbackWidth>(status, launch_epoch<CAPTURED>(a, 0), (int64_t)t - 1,
                                 i ? (int64_t)(t - G) : -1, lane, lb);
  uint64_t dev_epoch = 0;
  if (CAPTURED) {
    if (!mbar_wait(&sm.epoch_bar, 0u, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    dev_epoch = sm.epoch;
  }
  const uint64_t epoch = launch_epoch<CAPTURED>(a, dev_epoch);
  for (; t < a.total_tiles; i += 2, t += 2 * G) {
    const int s = (int)(i % kSlots);
    if (!mbar_wait(&sm.packed[s], (i / kSlots) & 1u, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    SlotInfo& f = sm.info[s];
    const uint32_t agg = f.agg, ti = f.ti;
    const uint64_t lt = f.lt;
    const int64_t floor = i ? (int64_t)(t - G) : -1;
    uint64_t excl = 0, since_start = 0;
    // Batches: the payload units before the tile's stream (pstart). If the CTA's previous
    // tile t - G lies in the same tensor, it is that tile's; otherwise the tensor's first
    // tile lies inside this tile's look-back window (t - G, t), and pstart is excl less the
    // aggregates from that first tile on, which the look-back reads anyway. So no tile
    // waits for another CTA's settle.
    bool ok = MAXT > 1 ? aggsum_finish<kLookbackWidth, true>(status, epoch, t, floor, lane,
                                                             a.wait_limit_ns, ctl, lb, &excl,
                                                             (int64_t)a.tile_begin[ti],
                                                             &since_start)
                       : aggsum_finish<kLookbackWidth>(status, epoch, t, floor, lane,
                                                       a.wait_limit_ns, ctl, lb, &excl);
    // A captured launch: tile G - 1 is the last of the first round, and its look-back has
    // read the aggregates of tiles 0 .. G - 2, one from every other CTA, each tagged with
    // the epoch that CTA read at its start. So every CTA has read the counter: move it on.
    // After a timeout some CTA may not have read it yet; the counter then skips a value,
    // so that such a CTA's entries never carry the next launch's epoch.
    if (CAPTURED && t + 1 == G && lane == 0)
      st_relaxed_u64(reinterpret_cast<uint64_t*>(a.ws + kEpochOffset), ok ? epoch : epoch + 1);
    if (t + 2 * G < a.total_tiles)  // start this warp's next pass
      aggsum_issue<kLookbackWidth>(status, epoch, (int64_t)(t + 2 * G) - 1, (int64_t)(t + G),
                                   lane, lb);
    uint32_t prev_ti = ~0u;
    uint64_t prev_pstart = 0;
    if (i > 0) {  // the CTA's previous tile, from the other settle warp
      const uint32_t h = (i - 1) & 1u;
      if (!mbar_wait(&sm.handoff[h], ((i - 1) / 2) & 1u, a.wait_limit_ns)) {
        if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
        return;
      }
      ok = ok && sm.incl_ok[h];
      excl += sm.incl[h];
      prev_ti = sm.incl_ti[h];
      prev_pstart = sm.incl_pstart[h];
    }
    uint64_t pstart = 0;
    if (MAXT > 1) pstart = lt == 0 ? excl : (prev_ti == ti ? prev_pstart : excl - since_start);
    __syncwarp();  // every lane has read the handoff before it is overwritten two tiles on
    if (lane == 0) {
      sm.incl[i & 1u] = excl + agg;
      sm.incl_ok[i & 1u] = ok;
      sm.incl_ti[i & 1u] = ti;
      sm.incl_pstart[i & 1u] = pstart;
      mbar_arrive(&sm.handoff[i & 1u]);
    }
    const uint64_t dst = a.payload_base[ti] + excl;
    if (ok && dst + agg > a.out_words) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_BUFFER_TOO_SMALL, t);
      ok = false;
    }
    if (lane == 0) {
      if (MAXT > 1 && lt == 0) {  // the headers need every stream's start (finalize_warp)
        st_relaxed_u64(&tstart[ti].value, excl);
        st_release_u64(&tstart[ti].tag, (epoch << 2) | (ok ? kStartPrefix : kStartError));
      }
      f.dst = dst;
      f.excl = excl;
      f.pstart = pstart;
      f.ok = ok;
      mbar_arrive(&sm.settled[s]);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (t + 1 == a.total_tiles)  // the last tile: its place gives the total payload
      finalize_warp(a, epoch, ok ? excl + agg : 0, !ok, tstart, ctl, sm.pbuf, lane);
  }
}

// ---- the packed tile's copy for WB = 2: units up to the destination's first 16-byte
// boundary one per lane, then 16-byte stores, each put together from the two aligned
// 16-byte groups of the slot it straddles (the slot-side byte phase is twice the head), then
// the last units one per lane. The second group may reach up to 14 bytes past the packed
// tile: still inside the shared-memory block, and those bytes are not used.
template <int PH>  // slot-side byte phase: even, 0..14
__device__ __forceinline__ uint4 take16(const uint4& x, const uint4& y) {
  const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
  constexpr int q = PH / 4;
  if (PH % 4 == 0) return make_uint4(w[q], w[q + 1], w[q + 2], w[q + 3]);
  return make_uint4(__funnelshift_r(w[q], w[q + 1], 16), __funnelshift_r(w[q + 1], w[q + 2], 16),
                    __funnelshift_r(w[q + 2], w[q + 3], 16), __funnelshift_r(w[q + 3], w[q + 4], 16));
}

template <int PH>
__device__ __forceinline__ void copy_body16(uint4* gv, const uint4* sv, uint32_t nv, uint32_t lane) {
#pragma unroll 4
  for (uint32_t q = lane; q < nv; q += 32) gv[q] = PH == 0 ? sv[q] : take16<PH>(sv[q], sv[q + 1]);
}

__device__ __forceinline__ void copy_out16(uint16_t* g, const uint32_t* src, uint32_t units,
                                           uint32_t lane) {
  const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
  const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(g) & 15u);  // even
  const uint32_t head = min(units, ((16u - mis) & 15u) >> 1);
  if (lane < head) g[lane] = s16[lane];
  const uint32_t nv = (units - head) >> 3;
  uint4* gv = reinterpret_cast<uint4*>(g + head);
  const uint4* sv = reinterpret_cast<const uint4*>(src);
  switch (head) {
    case 0: copy_body16<0>(gv, sv, nv, lane); break;
    case 1: copy_body16<2>(gv, sv, nv, lane); break;
    case 2: copy_body16<4>(gv, sv, nv, lane); break;
    case 3: copy_body16<6>(gv, sv, nv, lane); break;
    case 4: copy_body16<8>(gv, sv, nv, lane); break;
    case 5: copy_body16<10>(gv, sv, nv, lane); break;
    case 6: copy_body16<12>(gv, sv, nv, lane); break;
    default: copy_body16<14>(gv, sv, nv, lane); break;
  }
  const uint32_t done = head + 8u * nv;
  if (lane < units - done) g[done + lane] = s16[done + lane];
}

// ---- store warps: copy the packed tile out, write its chunk table entries, refill the slot
template <int MAXT, int WB, bool INNER>
__device__ void store_role(const CompressArgs<MAXT, WB>& a, CompressShared<WB>& sm, Control* ctl,
                           uint32_t k, uint32_t lane) {
  const unsigned long long G = gridDim.x;
  const uint32_t wpc = a.chunk_elems / kWindow;
  for (uint32_t i = k;; i += kStoreWarps) {
    const unsigned long long t = blockIdx.x + (unsigned long long)i * G;
    if (t >= a.total_tiles) return;
    const int s = (int)(i % kSlots);
    if (!mbar_wait(&sm.settled[s], (i / kSlots) & 1u, a.wait_limit_ns)) {
      if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, t);
      return;
    }
    const SlotInfo& f = sm.info[s];
    const uint32_t* src = sm.slot[s];
    if (f.ok && WB == 2) {
      copy_out16(reinterpret_cast<uint16_t*>(a.out + f.dst), src, f.agg, lane);
    } else if (f.ok) {
      const uint32_t agg = f.agg;
      uint32_t* g = reinterpret_cast<uint32_t*>(a.out + f.dst);
      // words up to the first 16-byte boundary of the destination, then 16-byte stores;
      // where the slot side is not 16-byte aligned, every lane reads the two aligned 16-byte
      // groups its four words straddle (conflict-free, unlike four strided 4-byte loads) and
      // picks them out. The second group may reach up to 3 words past the packed tile:
      // still inside the shared-memory block, and those words are not used.
      const uint32_t head = min(agg, (4u - (uint32_t)((reinterpret_cast<uintptr_t>(g) >> 2) & 3u)) & 3u);
      if (lane < head) g[lane] = src[lane];
      const uint32_t nv = (agg - head) >> 2;
      uint4* gv = reinterpret_cast<uint4*>(g + head);
      const uint4* sv = reinterpret_cast<const uint4*>(src);
      if (head == 0) {
#pragma unroll 4
        for (uint32_t q = lane; q < nv; q += 32) gv[q] = sv[q];
      } else if (head == 1) {
#pragma unroll 4
        for (uint32_t q = lane; q < nv; q += 32) {
          const uint4 x = sv[q], y = sv[q + 1];
          gv[q] = make_uint4(x.y, x.z, x.w, y.x);
        }
      } else if (head == 2) {
#pragma unroll 4
        for (uint32_t q = lane; q < nv; q += 32) {
          const uint4 x = sv[q], y = sv[q + 1];
          gv[q] = make_uint4(x.z, x.w, y.x, y.y);
        }
      } else {
#pragma unroll 4
        for (uint32_t q = lane; q < nv; q += 32) {
          const uint4 x = sv[q], y = sv[q + 1];
          gv[q] = make_uint4(x.w, y.x, y.y, y.z);
        }
      }
      const uint32_t done = head + 4 * nv;
      if (lane < agg - done) g[done + lane] = src[done + lane];
    }
    if (f.ok) {
      // chunk table entries of the chunks that start in this tile (the stream, its header
      // and its table start on 4-byte boundaries: see launch_t)
      uint32_t* table = reinterpret_cast<uint32_t*>(a.out + a.hdr_before[f.ti] + f.pstart) +
                        kStreamHeaderWords;
      const uint64_t in_stream = f.excl - f.pstart;  // payload words of the stream before the tile
      const uint64_t w_first = f.lt * kTileWindows;
      if (!INNER || !a.inner_chunks) {  // chunks are whole tiles: at most window 0 starts one
        if (lane == 0 && w_first % wpc == 0)
          put_u64_words(table + 2 * (w_first / wpc), WB * in_stream);
      } else {  // the first chunk starting in the tile, then one every wpc windows
        const uint32_t nwin = (f.valid + kWindow - 1) / kWindow;
        const uint64_t c0 = (w_first + wpc - 1) / wpc;
        const uint32_t first = (uint32_t)(c0 * wpc - w_first);
        for (uint32_t w = first + lane * wpc, c = lane; w < nwin; w += 32 * wpc, c += 32)
          put_u64_words(table + 2 * (c0 + c), WB * (in_stream + sm.woff[s][w]));
      }
    }
    // the slot is read; it takes tile i + kSlots next
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) fill_slot(a, sm, s, t + (unsigned long long)kSlots * G);
  }
}

template <int MAXT, int WB, bool INNER, bool CAPTURED>
__global__ void __launch_bounds__(kRoleThreads, 1)
    compress_kernel(const __grid_constant__ CompressArgs<MAXT, WB> a) {
  extern __shared__ __align__(16) uint8_t dsmem[];
  CompressShared<WB>& sm = *reinterpret_cast<CompressShared<WB>*>(dsmem);
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  // per tile: its aggregate, tagged with this launch's epoch; then the tensor starts
  uint64_t* status = reinterpret_cast<uint64_t*>(a.ws + kStatusOffset);
  TensorStart* tstart = reinterpret_cast<TensorStart*>(status + a.total_tiles);
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;

  if (a.total_tiles == 0) {  // every tensor empty: headers only
    if (warp == 0) finalize_warp(a, 0, 0, false, tstart, ctl, sm.pbuf, lane);
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.packed[s], kTeamWarps);
      mbar_init(&sm.settled[s], 1);
    }
    mbar_init(&sm.handoff[0], 1);
    mbar_init(&sm.handoff[1], 1);
    if (CAPTURED) mbar_init(&sm.epoch_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long G = gridDim.x;
  // The first round: kFirstFills slots at once, the rest when the first tile has landed.
  // Every CTA asks for its whole ring at the start; holding most of it back lets each CTA's
  // first tiles arrive (and the pipeline start) well before the burst is through.
  if (tid == 0)
    for (int s = 0; s < kFirstFills; ++s) fill_slot(a, sm, s, blockIdx.x + (unsigned long long)s * G);
  if (warp < kSettleWarp0)
    pack_role<MAXT, WB, INNER, CAPTURED>(a, sm, status, ctl, warp / kTeamWarps, warp % kTeamWarps,
                                         lane);
  else if (warp < kStoreWarp0)
    settle_role<MAXT, WB, CAPTURED>(a, sm, status, tstart, ctl, warp - kSettleWarp0, lane);
  else {
    if (CAPTURED && warp == kStoreWarp0 + 1 && lane == 0) {  // the launch's epoch (see above)
      sm.epoch = 1u + ld_relaxed_u64(reinterpret_cast<const uint64_t*>(a.ws + kEpochOffset));
      mbar_arrive(&sm.epoch_bar);
    }
    if (warp == kStoreWarp0 && lane == 0 && blockIdx.x < a.total_tiles &&
        mbar_wait(&sm.full[0], 0u, a.wait_limit_ns))
      for (int s = kFirstFills; s < kSlots; ++s)
        fill_slot(a, sm, s, blockIdx.x + (unsigned long long)s * G);
    __syncwarp();
    store_role<MAXT, WB, INNER>(a, sm, ctl, warp - kStoreWarp0, lane);
  }
}

__global__ void lookback_probe_kernel(uint8_t* ws, uint64_t epoch, uint64_t limit_ns) {
  Control* ctl = reinterpret_cast<Control*>(ws);
  const uint64_t* status = reinterpret_cast<const uint64_t*>(ws + kStatusOffset);
  // tile 1 sums the aggregate of tile 0, which nothing publishes in this epoch
  uint64_t v[kLookbackWidth];
  uint64_t sum = 0;
  aggsum_issue<kLookbackWidth>(status, epoch, 0, -1, threadIdx.x & 31u, v);
  aggsum_finish<kLookbackWidth>(status, epoch, 1, -1, threadIdx.x & 31u, limit_ns, ctl, v, &sum);
}

// Epochs of compress launches outside a stream capture: a process-wide counter started at a
// random point between 2^39 and 2^40, so that entries a previous process may have left in
// reused device memory do not match either, so far above the epochs of captured launches
// (a workspace counter from 1) that the two never meet, and far below 2^48, so that it
// never wraps.
std::atomic<uint64_t> g_epoch{0};

uint64_t next_epoch() {
  uint64_t e = g_epoch.load();
  if (e == 0) {
    std::random_device rd;
    const uint64_t seed = ((((uint64_t)rd() << 32) ^ rd()) & ((1ull << 39) - 1)) | (1ull << 39);
    uint64_t expected = 0;
    g_epoch.compare_exchange_strong(expected, seed | 1);
  }
  return g_epoch.fetch_add(1) + 1;
}

// Launches compress_kernel over T tensors of WB-byte words into `out` (out_units words of
// WB bytes). Every stream starts on a 4-byte boundary, so that the kernel can write headers
// and tables as 32-bit words: with WB = 4 every position is one, and WB = 2 is a single
// stream at `out` (4-byte aligned; checked by the caller).
// CTAs of one compress_kernel instantiation that fit on the current device at once, found
// once per device. (cudaFuncSetAttribute also loads the kernel, which a launch under stream
// capture needs done beforehand.)
template <int MAXT, int WB, bool INNER, bool CAPTURED>
zvc_status resident_ctas(int dev, int* out) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> resident_of[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return ZVC_ERR_INVALID_ARG;
  int resident = resident_of[dev].load();
  if (resident == 0) {
    const int smem = (int)sizeof(CompressShared<WB>);
    cudaError_t e = cudaFuncSetAttribute(compress_kernel<MAXT, WB, INNER, CAPTURED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_failure(e);
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_failure(e);
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
             &per_sm, compress_kernel<MAXT, WB, INNER, CAPTURED>, kRoleThreads, smem)) !=
        cudaSuccess)
      return cuda_failure(e);
    resident = sms * (per_sm > 0 ? per_sm : 1);
    resident_of[dev].store(resident);
  }
  *out = resident;
  return ZVC_OK;
}

// Launches compress_kernel over T tensors of WB-byte words into `out` (out_units words of
// WB bytes). Every stream starts on a 4-byte boundary, so that the kernel can write headers
// and tables as 32-bit words: with WB = 4 every position is one, and WB = 2 is a single
// stream at `out` (4-byte aligned; checked by the caller).
template <int MAXT, int WB, bool INNER, bool CAPTURED>
zvc_status launch_k(const TensorIn* ts, uint32_t T, bool batched, uint32_t C, void* out,
                    uint64_t out_units, uint64_t* out_size, uint8_t* ws, uint64_t limit_ns,
                    int dev, cudaStream_t stream) {
  using Word = typename CompressArgs<MAXT, WB>::Word;
  static_assert(WB == 4 || MAXT == 1, "16-bit words: single streams only");
  CompressArgs<MAXT, WB> args;
  args.out = static_cast<Word*>(out);
  args.out_words = out_units;
  args.out_size = out_size;
  args.ws = ws;
  args.wait_limit_ns = limit_ns;
  args.epoch = CAPTURED ? 0 : next_epoch();  // a captured launch reads its own on the device
  args.chunk_elems = C;
  args.T = T;
  args.batched = batched ? 1u : 0u;
  args.inner_chunks = C % kTileElems != 0 ? 1u : 0u;
  uint64_t tiles = 0;
  // header, tables and batch prefix in units of WB bytes
  uint64_t hdr = batched ? (4 * kBatchHeaderWords + 8 * ((uint64_t)T + 1)) / WB : 0;
  for (uint32_t i = 0; i < T; ++i) {
    args.in[i] = static_cast<const Word*>(ts[i].ptr);
    args.n[i] = ts[i].n;
    args.tile_begin[i] = tiles;
    args.hdr_before[i] = hdr;
    tiles += tiles_for(ts[i].n);
    hdr += (4 * kStreamHeaderWords + 8 * ceil_div_u64(ts[i].n, C)) / WB;
    args.payload_base[i] = hdr;
  }
  args.tile_begin[T] = tiles;
  args.total_tiles = tiles;
  args.hdr_words_end = hdr;

  int resident = 0;
  const zvc_status st = resident_ctas<MAXT, WB, INNER, CAPTURED>(dev, &resident);
  if (st != ZVC_OK) return st;
  const uint64_t grid = tiles == 0 ? 1 : (tiles < (uint64_t)resident ? tiles : (uint64_t)resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kRoleThreads);
  cfg.dynamicSmemBytes = sizeof(CompressShared<WB>);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident together
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const TraceMark mark = trace_begin(kTraceCompress, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, compress_kernel<MAXT, WB, INNER, CAPTURED>, args);
  trace_end(mark, stream);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

// Chunks that start inside tiles (C not a multiple of the tile) need the packed offsets of
// windows inside tiles. The kernel for whole-tile chunks carries none of that code, and is
// 1-3% faster for it (the kernel's speed depends on its code size: measured on 2^28-word maps
// and the GoogLeNet batch at C = 4096). The other instantiation keeps its run-time checks,
// which compile to a faster kernel there than the same code with them folded away.
// A launch on a capturing stream takes the instantiation that reads its epoch on the device;
// a launch outside a capture also readies that one, so that a later capture finds it loaded.
template <int MAXT, int WB, bool INNER>
zvc_status launch_i(const TensorIn* ts, uint32_t T, bool batched, uint32_t C, void* out,
                    uint64_t out_units, uint64_t* out_size, uint8_t* ws, uint64_t limit_ns,
                    cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failure(e);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(stream, &cs)) != cudaSuccess) return cuda_failure(e);
  if (cs != cudaStreamCaptureStatusNone)
    return launch_k<MAXT, WB, INNER, true>(ts, T, batched, C, out, out_units, out_size, ws,
                                           limit_ns, dev, stream);
  int r = 0;
  const zvc_status st = resident_ctas<MAXT, WB, INNER, true>(dev, &r);
  if (st != ZVC_OK) return st;
  return launch_k<MAXT, WB, INNER, false>(ts, T, batched, C, out, out_units, out_size, ws,
                                          limit_ns, dev, stream);
}

template <int MAXT, int WB>
zvc_status launch_t(const TensorIn* ts, uint32_t T, bool batched, uint32_t C, void* out,
                    uint64_t out_units, uint64_t* out_size, uint8_t* ws, uint64_t limit_ns,
                    cudaStream_t stream) {
  if (C % kTileElems != 0)
    return launch_i<MAXT, WB, true>(ts, T, batched, C, out, out_units, out_size, ws, limit_ns,
                                    stream);
  return launch_i<MAXT, WB, false>(ts, T, batched, C, out, out_units, out_size, ws, limit_ns,
                                   stream);
}

}  // namespace

zvc_status launch_compress(const TensorIn* ts, uint32_t T, bool batched, uint32_t chunk_elems,
                           uint32_t* out, uint64_t out_words, uint64_t* out_size, uint8_t* ws,
                           uint64_t wait_limit_ns, cudaStream_t stream) {
  if (!batched && T == 1)
    return launch_t<1, 4>(ts, T, false, chunk_elems, out, out_words, out_size, ws, wait_limit_ns,
                          stream);
  if (T <= 64)
    return launch_t<64, 4>(ts, T, batched, chunk_elems, out, out_words, out_size, ws,
                           wait_limit_ns, stream);
  return launch_t<ZVC_MAX_BATCH, 4>(ts, T, batched, chunk_elems, out, out_words, out_size, ws,
                                    wait_limit_ns, stream);
}

zvc_status launch_compress16(const uint16_t* in, uint64_t n, uint32_t chunk_elems, uint16_t* out,
                             uint64_t out_units, uint64_t* out_size, uint8_t* ws,
                             uint64_t wait_limit_ns, cudaStream_t stream) {
  const TensorIn t{in, n};
  return launch_t<1, 2>(&t, 1, false, chunk_elems, out, out_units, out_size, ws, wait_limit_ns,
                        stream);
}

zvc_status launch_lookback_timeout_probe(uint8_t* ws, uint64_t limit_ns, cudaStream_t stream) {
  lookback_probe_kernel<<<1, 32, 0, stream>>>(ws, next_epoch(), limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

}  // namespace zvc
