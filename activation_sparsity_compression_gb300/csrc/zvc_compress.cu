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
//   offset  decoupled look-back over the tile status words gives the tile's place in the
//           payload (each lane reads 10 predecessors per round, so one round covers a
//           whole round of tiles); chunk starts inside the tile write their chunk_off entry
//   store   the packed tile is built in shared memory at the destination's alignment and
//           written with 16-byte streaming stores (scalar stores for the ragged ends)
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
  uint32_t pad;
  const uint32_t* in[MAXT];
  uint64_t n[MAXT];
  uint64_t tile_begin[MAXT + 1];  // first tile of tensor i; tile_begin[T] = total_tiles
  uint64_t hdr_before[MAXT];      // header/table words (and batch prefix) before stream i
  uint64_t payload_base[MAXT];    // hdr_before + this stream's header and table
};

constexpr uint32_t kStageWords = kTileWindows + kTileElems + 4;

using PerCallCounters = Counters;
static_assert(sizeof(PerCallCounters) <= kCountersBytes, "counter block");

__device__ __forceinline__ void put_u64_words(uint32_t* p, uint64_t v) {
  p[0] = (uint32_t)v;
  p[1] = (uint32_t)(v >> 32);
}

// Headers of every stream and the batch table. Runs in the CTA that owns the last tile,
// once that tile knows its place (so the total payload is known); `failed` is set when
// that tile gave up, in which case a failure upstream has been latched already.
template <int MAXT>
__device__ void finalize(const CompressArgs<MAXT>& a, uint64_t total_payload, bool failed,
                         const uint64_t* tstart, Control* ctl, uint64_t* pbuf) {
  const uint32_t tid = threadIdx.x;
  __shared__ int s_fail;
  if (tid == 0) {
    bool bad = failed;
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
              bad = true;
              break;
            }
          }
        }
      }
      pbuf[i] = p;
      next = p;
    }
    s_fail = bad;
    if (bad && a.out_size) *a.out_size = 0;
  }
  __syncthreads();
  if (s_fail) return;
  for (uint32_t i = tid; i < a.T; i += blockDim.x) {
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
  if (tid == 0) {
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

constexpr int kStages = 4;           // input tiles in flight per CTA
constexpr int kLookbackWidth = 10;   // look-back pass covers 32 * 10 predecessor tiles
constexpr int kProducerWarp = kCompressWarps - 1;

struct __align__(16) CompressShared {
  uint32_t in[kStages][kTileElems];     // input ring, filled by 1-D TMA bulk copies
  uint32_t out[2][kStageWords];         // packed tiles k (being written) and k-1 (being stored)
  uint32_t win_off[2][kTileWindows];    // word offset of each window inside its packed tile
  uint64_t full[kStages];               // mbarrier per ring slot
  unsigned long long tile[kStages];
  uint32_t tensor[kStages];
  uint32_t direct[kStages];             // 1: slot not filled, consumers read global memory
  uint32_t warp_words[kCompressWarps];
  // the tile being stored (k-1), as settled by its look-back
  uint64_t st_dst, st_excl, st_pstart, st_c0;
  uint32_t st_words, st_nchunks, st_tensor, st_ok;
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
// not 16-byte aligned) are marked direct and read by the consumers from global memory.
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

// The tile whose packed words wait in sm.out[buf] for their place in the payload.
struct Pending {
  uint64_t t;       // tile index
  uint64_t lt;      // tile index inside its tensor
  uint32_t ti;      // tensor
  uint32_t agg;     // packed words
  uint32_t valid;   // input words
  bool live;
};

// Warp 0: settles the place of tile p (its aggregate is already published) and writes
// what the store step needs into shared memory. s_pre holds a look-back pass issued
// earlier; it is used if it already resolves the prefix, else the look-back re-reads.
template <int MAXT>
__device__ __forceinline__ void settle(const CompressArgs<MAXT>& a, CompressShared& sm,
                                       const Pending& p, uint64_t* status, uint64_t* tstart,
                                       Control* ctl, uint32_t lane) {
  uint64_t excl = 0;
  bool ok = true;
  if (p.t != 0) ok = lookback_exclusive_wide<kLookbackWidth>(status, p.t, lane, a.wait_limit_ns, ctl, &excl);
  const uint64_t dst = a.payload_base[p.ti] + excl;
  if (ok && dst + p.agg > a.out_words) {
    if (lane == 0) latch_error(ctl, ZVC_ERR_BUFFER_TOO_SMALL, p.t);
    ok = false;
  }
  if (lane == 0) {
    if (p.t != 0)
      st_relaxed_u64(status + p.t, ok ? ((kFlagPrefix << kFlagShift) | (excl + p.agg))
                                      : (kFlagError << kFlagShift));
    uint64_t pstart = 0;
    if (MAXT > 1) {
      if (p.lt == 0) {
        st_relaxed_u64(tstart + p.ti,
                       ok ? ((kFlagPrefix << kFlagShift) | excl) : (kFlagError << kFlagShift));
        pstart = excl;
      } else if (ok) {
        // payload words before this tensor, published by its first tile (a lower tile)
        WaitClock clock;
        while (true) {
          const uint64_t st = ld_relaxed_u64(tstart + p.ti);
          const uint64_t f = st >> kFlagShift;
          if (f == kFlagPrefix) { pstart = st & kValueMask; break; }
          if (f == kFlagError || !clock.tick(a.wait_limit_ns)) {
            latch_error(ctl, ZVC_ERR_TIMEOUT, p.t);
            ok = false;
            break;
          }
        }
      }
    }
    // chunks whose first window lies in this tile
    const uint32_t wpc = a.chunk_elems / kWindow;
    const uint64_t w0 = p.lt * kTileWindows;
    const uint64_t c0 = ceil_div_u64(w0, wpc);
    const uint64_t wend = w0 + (p.valid + kWindow - 1) / kWindow;
    sm.st_c0 = c0;
    sm.st_nchunks = c0 * wpc < wend ? (uint32_t)((wend - 1 - c0 * wpc) / wpc + 1) : 0u;
    sm.st_dst = dst;
    sm.st_excl = excl;
    sm.st_pstart = pstart;
    sm.st_words = p.agg;
    sm.st_tensor = p.ti;
    sm.st_ok = ok;
  }
}

// All threads: writes the settled tile from sm.out[buf] to its place, at 16-byte stores
// where the destination allows, and its chunk table entries.
template <int MAXT>
__device__ __forceinline__ void store_tile(const CompressArgs<MAXT>& a, CompressShared& sm,
                                           int buf, uint64_t lt, uint32_t tid) {
  if (!sm.st_ok) return;
  const uint64_t dst = sm.st_dst;
  const uint32_t words = sm.st_words;
  const uint32_t ti = sm.st_tensor;
  const uint32_t* src = sm.out[buf];
  const uint32_t wpc = a.chunk_elems / kWindow;
  const uint64_t w0 = lt * kTileWindows;
  for (uint32_t k = tid; k < sm.st_nchunks; k += kCompressThreads) {
    const uint64_t c = sm.st_c0 + k;
    put_u64_words(a.out + a.hdr_before[ti] + sm.st_pstart + kStreamHeaderWords + 2 * c,
                  4 * (sm.st_excl - sm.st_pstart + sm.win_off[buf][(uint32_t)(c * wpc - w0)]));
  }
  const uint32_t phase = (uint32_t)((reinterpret_cast<uintptr_t>(a.out + dst) >> 2) & 3u);
  uint32_t* g = a.out + dst - phase;  // 16-byte aligned; word w of g is packed word w - phase
  const uint32_t span = phase + words;
  for (uint32_t u = tid; 4u * u < span; u += kCompressThreads) {
    const uint32_t w = 4u * u;
    if (w >= phase && w + 4u <= span) {
      const uint4 q = make_uint4(src[w - phase], src[w + 1 - phase], src[w + 2 - phase],
                                 src[w + 3 - phase]);
      __stcs(reinterpret_cast<uint4*>(g + w), q);
    } else {
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j)
        if (w + j >= phase && w + j < span) g[w + j] = src[w + j - phase];
    }
  }
}

template <int MAXT>
__global__ void __launch_bounds__(kCompressThreads, 2)
    compress_kernel(const __grid_constant__ CompressArgs<MAXT> a) {
  extern __shared__ __align__(16) uint8_t dsmem[];
  CompressShared& sm = *reinterpret_cast<CompressShared*>(dsmem);
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  uint64_t* status = reinterpret_cast<uint64_t*>(a.ws + kStatusOffset);
  uint64_t* tstart = status + a.total_tiles;
  const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;

  if (a.total_tiles == 0) {  // every tensor empty: headers only
    finalize(a, 0, false, tstart, ctl, reinterpret_cast<uint64_t*>(sm.out));
    return;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long G = gridDim.x;
  if (warp == kProducerWarp && lane == 0)
    for (int s = 0; s < kStages; ++s) fill_slot(a, sm, s, blockIdx.x + s * G);

  const uint32_t ebase = warp * 512u + lane * 4u;
  const uint32_t sh = 4u * (lane & 7u);
  Pending prev;
  prev.live = false;

  for (uint32_t it = 0;; ++it) {
    const int slot = (int)(it % kStages);
    const int buf = (int)(it & 1u);
    const bool late = !mbar_wait(&sm.full[slot], (it / kStages) & 1u, a.wait_limit_ns);
    if (__syncthreads_or(late)) {
      if (tid == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, it);
      break;
    }
    const uint64_t t = sm.tile[slot];
    const bool have = t < a.total_tiles;
    if (!have && !prev.live) break;

    Pending cur;
    cur.live = have;
    uint32_t wpre = 0;
    uint32_t v[4][4], mask[4], wsz[4], woff[4];
    if (have) {
      cur.t = t;
      cur.ti = sm.tensor[slot];
      cur.lt = t - a.tile_begin[cur.ti];
      const uint64_t e0 = cur.lt * kTileElems;
      cur.valid = (uint32_t)min((uint64_t)kTileElems, a.n[cur.ti] - e0);

      // ---- load (ring slot, or global memory for a direct tile)
      if (!sm.direct[slot]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 q = *reinterpret_cast<const uint4*>(&sm.in[slot][ebase + 128u * k]);
          v[k][0] = q.x; v[k][1] = q.y; v[k][2] = q.z; v[k][3] = q.w;
        }
      } else {
        const uint32_t* src = a.in[cur.ti] + e0;
        const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t e = ebase + 128u * k;
          if (vec && e + 4 <= cur.valid) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4*>(src + e));
            v[k][0] = q.x; v[k][1] = q.y; v[k][2] = q.z; v[k][3] = q.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[k][j] = (e + j < cur.valid) ? __ldcs(src + e + j) : 0u;
          }
        }
      }

      // ---- masks and window sizes (a window past the end of the tensor has size 0)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t m = ((uint32_t)(v[k][0] != 0u) | ((uint32_t)(v[k][1] != 0u) << 1) |
                      ((uint32_t)(v[k][2] != 0u) << 2) | ((uint32_t)(v[k][3] != 0u) << 3))
                     << sh;
        m |= __shfl_xor_sync(0xffffffffu, m, 1);
        m |= __shfl_xor_sync(0xffffffffu, m, 2);
        m |= __shfl_xor_sync(0xffffffffu, m, 4);
        mask[k] = m;
        const uint32_t wt = warp * 16u + 4u * k + (lane >> 3);
        wsz[k] = (wt * kWindow < cur.valid) ? 1u + __popc(m) : 0u;
      }

      // ---- exclusive scan of window sizes inside the tile
      uint32_t run = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t x = wsz[k];
        uint32_t y = __shfl_up_sync(0xffffffffu, x, 8);
        if (lane >= 8) x += y;
        y = __shfl_up_sync(0xffffffffu, x, 16);
        if (lane >= 16) x += y;
        woff[k] = run + x - wsz[k];
        run += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) sm.warp_words[warp] = run;
    }
    __syncthreads();  // slot consumed, warp totals visible, tile k-2's store finished

    if (have) {
      if (warp == kProducerWarp && lane == 0) fill_slot(a, sm, slot, t + kStages * G);
      uint32_t agg = 0;
#pragma unroll
      for (int w = 0; w < kCompressWarps; ++w) {
        const uint32_t c = sm.warp_words[w];
        wpre += (w < (int)warp) ? c : 0u;
        agg += c;
      }
      cur.agg = agg;
      // publish this tile's aggregate now; its place is settled one iteration later
      if (tid == 0)
        st_relaxed_u64(status + t, t == 0 ? ((kFlagPrefix << kFlagShift) | agg)
                                          : ((kFlagAggregate << kFlagShift) | agg));

      // ---- pack tile k at offset 0 of its buffer
      uint32_t* ob = sm.out[buf];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (wsz[k] == 0u) continue;
        const uint32_t wo = wpre + woff[k];
        if ((lane & 7u) == 0u) {
          ob[wo] = mask[k];
          sm.win_off[buf][warp * 16u + 4u * k + (lane >> 3)] = wo;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (v[k][j] != 0u) {
            const uint32_t below = mask[k] & ((1u << (sh + j)) - 1u);
            ob[wo + 1u + __popc(below)] = v[k][j];
          }
        }
      }
    }

    // ---- settle and store tile k-1
    if (prev.live) {
      if (warp == 0) settle(a, sm, prev, status, tstart, ctl, lane);
      __syncthreads();
      store_tile(a, sm, buf ^ 1, prev.lt, tid);
      if (prev.t + 1 == a.total_tiles) {  // the last tile: its place gives the total
        const bool ok = sm.st_ok;
        const uint64_t total = sm.st_excl + sm.st_words;
        __syncthreads();
        finalize(a, ok ? total : 0, !ok, tstart, ctl,
                 reinterpret_cast<uint64_t*>(sm.out[buf ^ 1]));
      }
    } else {
      __syncthreads();
    }
    prev = cur;
  }
}

__global__ void lookback_probe_kernel(uint8_t* ws, uint64_t limit_ns) {
  Control* ctl = reinterpret_cast<Control*>(ws);
  uint64_t* status = reinterpret_cast<uint64_t*>(ws + kStatusOffset);
  uint64_t excl = 0;
  // tile 1 waits on tile 0, which never publishes
  lookback_exclusive(status, 1, threadIdx.x & 31u, limit_ns, ctl, &excl);
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
  args.pad = 0;
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
                                                           kCompressThreads, smem)) != cudaSuccess)
      return cuda_failure(e);
    resident = sms * (per_sm > 0 ? per_sm : 1);
  }
  e = cudaMemsetAsync(ws + kPerCallOffset, 0, per_call_bytes(tiles, T), stream);
  if (e != cudaSuccess) return cuda_failure(e);
  const uint64_t grid = tiles == 0 ? 1 : (tiles < (uint64_t)resident ? tiles : (uint64_t)resident);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCompressThreads);
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
