// ZVC decompress for sm_103a: the inverse of Rhu et al., "Compressing DMA Engine",
// section V.A (every set mask bit takes the next packed word, every clear bit is a zero;
// section V.B has the engine expand compressed data into 128-byte lines using the masks'
// prefix counts as scatter offsets).
//
// One warp decodes one chunk, located through the stream's chunk offset table:
//   validate  batch table (if any), stream header and this chunk's table entries; every
//             check that fails latches ZVC_ERR_CORRUPT and the warp returns before
//             touching the chunk, so no access leaves the input or output buffers
//   stage     the chunk's compressed words are copied into this warp's shared memory by
//             a 1-D TMA bulk copy (plain loads for the unaligned ends)
//   walk      a window's position depends on every earlier mask, so one lane walks the
//             masks (position += 1 + popc(mask)), recording each window's offset and mask;
//             the walk must end exactly at the next chunk's offset
//   scatter   lane l expands words 4(l mod 8) .. +3 of window 4q + l/8: a set bit at
//             position b reads packed word popc(mask & (2^b - 1)), a clear bit writes 0;
//             each step expands sixteen whole 128-byte windows with 16-byte stores
// Extra work items (one per tensor, after the chunks) check the headers of streams that
// have no chunks; an empty batch gets one item that checks its header and table.
#include "zvc_internal.cuh"

namespace zvc {
namespace {

constexpr uint32_t kBarrierWords = 16;  // one 8-byte mbarrier per warp, up to 8 warps

template <int MAXT>
struct DecompressArgs {
  const uint32_t* in;
  uint64_t in_bytes;
  uint8_t* ws;
  uint64_t total_chunks;
  uint64_t total_items;  // total_chunks + T header checks
  uint32_t chunk_elems;
  uint32_t T;
  uint32_t batched;
  uint32_t warps_per_cta;
  uint32_t buf_words;          // largest valid chunk: C/32 masks + C words
  uint32_t meta_offset_words;  // per window (position of its first value, mask), 8-byte aligned
  uint32_t warp_stride_words;  // shared memory per warp: chunk (+3 for its phase), window table
  uint32_t* out[MAXT];
  uint64_t n[MAXT];
  uint64_t chunk_begin[MAXT + 1];
};

__device__ __forceinline__ uint64_t get_u64_words(const uint32_t* p) {
  return (uint64_t)p[0] | ((uint64_t)p[1] << 32);
}

template <int MAXT>
__global__ void __launch_bounds__(256) decompress_kernel(const __grid_constant__ DecompressArgs<MAXT> a) {
  extern __shared__ __align__(16) uint32_t dsm[];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint64_t item = (uint64_t)blockIdx.x * a.warps_per_cta + warp;
  if (item >= a.total_items) return;
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  const uint32_t C = a.chunk_elems;
  uint64_t* bar = reinterpret_cast<uint64_t*>(dsm) + warp;
  uint32_t* buf = dsm + kBarrierWords + (uint64_t)warp * a.warp_stride_words;
  uint2* wmeta = reinterpret_cast<uint2*>(buf + a.meta_offset_words);  // (first value, mask)

  const bool is_chunk = item < a.total_chunks;
  uint32_t ti = 0;
  uint64_t c = 0;
  if (is_chunk) {
    if (MAXT > 1) {
      uint32_t lo = 0, hi = a.T;
      while (hi - lo > 1) {
        const uint32_t mid = (lo + hi) >> 1;
        if (a.chunk_begin[mid] <= item) lo = mid; else hi = mid;
      }
      ti = lo;
    }
    c = item - a.chunk_begin[ti];
  } else {
    ti = (uint32_t)(item - a.total_chunks);
  }
  const uint64_t n = ti < a.T ? a.n[ti] : 0;
  const uint64_t nc = ceil_div_u64(n, C);

  // ---- locate and validate the stream (all lanes compute the same values). Every
  // address read here is in bounds by sizes known before the round's loads, so each
  // round issues all its loads at once: the batch table, then the stream header and the
  // chunk's table entries.
  bool ok = true;
  uint64_t sb = 0, se = a.in_bytes;
  if (a.batched) {
    const uint64_t pre = 16 + 8 * ((uint64_t)a.T + 1);
    if (a.in_bytes < pre) {
      ok = false;
    } else {
      const uint32_t* bt = a.in + kBatchHeaderWords;
      const uint32_t magic = a.in[0], t = a.in[1];
      const uint64_t total = get_u64_words(a.in + 2);
      const uint64_t first = get_u64_words(bt), last = get_u64_words(bt + 2 * (uint64_t)a.T);
      if (ti < a.T) {
        sb = get_u64_words(bt + 2 * (uint64_t)ti);
        se = get_u64_words(bt + 2 * (uint64_t)ti + 2);
      }
      ok = (magic == kBatchMagic) & (t == a.T) & (total == a.in_bytes) & (first == pre) &
           (last == a.in_bytes);
      if (ti < a.T) ok = ok & (sb <= se) & (se <= a.in_bytes) & (((sb | se) & 3u) == 0);
    }
  }
  if (ti >= a.T) {  // empty batch: only its header and table exist
    if (!ok && lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, item);
    return;
  }
  const uint64_t table_end = 32 + 8 * nc;
  ok = ok && se - sb >= table_end;
  if (!ok) {
    if (lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, item);
    return;
  }
  const uint32_t* sw = a.in + sb / 4;
  const uint64_t payload = (se - sb) - table_end;
  uint32_t h[kStreamHeaderWords];
#pragma unroll
  for (uint32_t j = 0; j < kStreamHeaderWords; ++j) h[j] = sw[j];
  const uint64_t cbeg = c * C;
  const uint32_t count = is_chunk ? (uint32_t)min((uint64_t)C, n - cbeg) : 0u;
  const uint32_t nwin = (count + kWindow - 1) / kWindow;
  uint64_t start = 0, end = payload;
  if (is_chunk) {
    const uint32_t* ct = sw + kStreamHeaderWords + 2 * c;
    start = get_u64_words(ct);
    if (c + 1 < nc) end = get_u64_words(ct + 2);
  }
  ok = (h[0] == kStreamMagic) & (h[1] == kVersionWordBytes) & (h[2] == kWindow) & (h[3] == C) &
       (((uint64_t)h[4] | ((uint64_t)h[5] << 32)) == n) &
       (((uint64_t)h[6] | ((uint64_t)h[7] << 32)) == payload);
  if (is_chunk)
    ok = ok & ((c != 0) | (start == 0)) & (start <= end) & (end <= payload) &
         (((start | end) & 3u) == 0) && (end - start) / 4 >= nwin &&
         (end - start) / 4 <= (uint64_t)nwin + count;
  if (!ok || !is_chunk) {
    if (!ok && lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, item);
    return;
  }

  // ---- stage the chunk: its words sit in shared memory at the same 16-byte phase as in
  // global memory, so one bulk copy moves the aligned body; lanes load the at most three
  // words on either side.
  const uint32_t len = (uint32_t)((end - start) / 4);
  const uint32_t* cw = sw + kStreamHeaderWords + 2 * nc + start / 4;
  const uint32_t phase = (uint32_t)((reinterpret_cast<uintptr_t>(cw) >> 2) & 3u);
  buf += phase;
  const uint32_t head = min(len, (4u - phase) & 3u);
  const uint32_t body = (len - head) & ~3u;
  const uint32_t tail = len - head - body;
  if (body > 0) {
    if (lane == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(bar, body * 4);
      bulk_g2s(buf + head, cw + head, body * 4, bar);
    }
  }
  if (lane < head) buf[lane] = __ldcs(cw + lane);
  if (lane < tail) buf[head + body + lane] = __ldcs(cw + head + body + lane);
  __syncwarp();
  if (body > 0 && !mbar_wait(bar, 0, kDefaultWaitLimitNs)) {
    if (lane == 0) latch_error(ctl, ZVC_ERR_TIMEOUT, item);
    return;
  }
  __syncwarp();

  // ---- walk the masks. The chain position -> mask -> next position is the critical
  // path, so the loop carries nothing else: a window spans at most 33 words, so the k-th
  // read sits below 33k <= buf_words - 33 and stays in this warp's buffer even for a
  // corrupt chunk, and since positions only grow, ending exactly at len proves that every
  // read was inside the chunk.
  uint32_t good = 1;
  if (lane == 0) {
    uint32_t pos = 0, m = 0;
#pragma unroll 4
    for (uint32_t w = 0; w < nwin; ++w) {
      m = buf[pos];
      wmeta[w] = make_uint2(pos + 1u, m);
      pos += 1u + __popc(m);
    }
    const uint32_t ragged = count & (kWindow - 1);
    good = (pos == len) & (ragged == 0 || (m >> ragged) == 0u);
  }
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good) {
    if (lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, item);
    return;
  }
  __syncwarp();

  // ---- scatter: lane l expands words e .. e+3 (e = 4(l mod 8)) of windows l/8 + 4k;
  // four windows per lane are in flight at once
  uint32_t* dst = a.out[ti] + cbeg;
  const bool vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const uint32_t e = 4u * (lane & 7u);
  const uint32_t below = (1u << e) - 1u;
  for (uint32_t w0 = lane >> 3; w0 < nwin; w0 += 16) {
    uint4 r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = w0 + 4u * k;
      const uint2 mo = w < nwin ? wmeta[w] : make_uint2(0u, 0u);
      const uint32_t m = mo.y;
      uint32_t q = mo.x + __popc(m & below);
      uint32_t v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bit = (m >> (e + j)) & 1u;
        v[j] = bit ? buf[q] : 0u;
        q += bit;
      }
      r[k] = make_uint4(v[0], v[1], v[2], v[3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = w0 + 4u * k;
      const uint32_t base = w * kWindow + e;
      if (w >= nwin) break;
      if (vec && base + 4u <= count) {
        *reinterpret_cast<uint4*>(dst + base) = r[k];
      } else {
        const uint32_t vv[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j)
          if (base + j < count) dst[base + j] = vv[j];
      }
    }
  }
}

template <int MAXT>
zvc_status launch_t(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts, uint32_t T,
                    bool batched, uint32_t C, uint8_t* ws, cudaStream_t stream) {
  DecompressArgs<MAXT> args;
  args.in = in;
  args.in_bytes = in_bytes;
  args.ws = ws;
  args.chunk_elems = C;
  args.T = T;
  args.batched = batched ? 1u : 0u;
  uint64_t chunks = 0;
  for (uint32_t i = 0; i < T; ++i) {
    args.out[i] = ts[i].ptr;
    args.n[i] = ts[i].n;
    args.chunk_begin[i] = chunks;
    chunks += ceil_div_u64(ts[i].n, C);
  }
  args.chunk_begin[T] = chunks;
  args.total_chunks = chunks;
  args.total_items = chunks + (batched && T == 0 ? 1 : T);
  const uint32_t wpc = C / kWindow;
  args.buf_words = wpc + C;
  args.meta_offset_words = (uint32_t)round_up_u64(args.buf_words + 4, 2);
  args.warp_stride_words = (uint32_t)round_up_u64(args.meta_offset_words + 2ull * wpc, 4);
  const uint64_t per_warp = 4ull * args.warp_stride_words;
  uint32_t warps = (uint32_t)(73728ull / per_warp);
  warps = warps < 1 ? 1 : (warps > 8 ? 8 : warps);
  args.warps_per_cta = warps;
  const uint64_t smem = 4ull * kBarrierWords + per_warp * warps;
  cudaError_t e = cudaFuncSetAttribute(decompress_kernel<MAXT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_failure(e);
  const uint64_t blocks = ceil_div_u64(args.total_items, warps);
  const TraceMark mark = trace_begin(kTraceDecompress, stream);
  decompress_kernel<MAXT><<<(unsigned)blocks, 32 * warps, smem, stream>>>(args);
  trace_end(mark, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

}  // namespace

zvc_status launch_decompress(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts,
                             uint32_t T, bool batched, uint32_t chunk_elems, uint8_t* ws,
                             cudaStream_t stream) {
  if (!batched && T == 1) return launch_t<1>(in, in_bytes, ts, T, false, chunk_elems, ws, stream);
  if (T <= 64) return launch_t<64>(in, in_bytes, ts, T, batched, chunk_elems, ws, stream);
  return launch_t<ZVC_MAX_BATCH>(in, in_bytes, ts, T, batched, chunk_elems, ws, stream);
}

}  // namespace zvc
