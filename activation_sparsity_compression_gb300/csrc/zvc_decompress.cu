// ZVC decompress for sm_103a: the inverse of Rhu et al., "Compressing DMA Engine",
// section V.A (every set mask bit takes the next packed word, every clear bit is a zero;
// section V.B has the engine expand compressed data into 128-byte lines using the masks'
// prefix counts as scatter offsets).
//
// A chunk, located through the stream's chunk offset table, is decoded by a walker and a
// scatterer: two warps of a CTA of its own (chunks over 2048 words), or one warp that
// walks and then scatters (smaller chunks, 8 per CTA). The walker:
//   validate  batch table (if any), stream header and this chunk's table entries; every
//             check that fails latches ZVC_ERR_CORRUPT before any access to the chunk
//   stage     the chunk's compressed words are copied into shared memory by a 1-D TMA
//             bulk copy (plain loads for the unaligned ends), at their 16-byte phase
//   walk      a window's position depends on every earlier mask, so one lane walks the
//             masks (position += 1 + popc(mask)), recording each window's (first value,
//             mask) in one 8-byte store into a table that starts cleared; the walk must
//             end exactly at the next chunk's offset
// The scatterer expands windows as soon as it reads their entries non-zero, so with two
// warps the
// scatter runs under the walk: lane l expands words 4(l mod 8) .. +3 of window l/8 + 4k of each
// group of 16 windows, a set bit at position b reading packed word popc(mask & (2^b - 1)),
// a clear bit writing 0, with 16-byte stores.
// Extra work items (one per tensor, after the chunks) check the headers of streams that
// have no chunks; an empty batch gets one item that checks its header and table.
#include "zvc_internal.cuh"

namespace zvc {
namespace {

// Shared memory of a CTA: control words, then the chunk buffer (C/32 masks + C words, +3
// for the 16-byte phase), then the window table (first value, mask) per window.
struct DecompressCtl {
  uint64_t full;        // mbarrier of the TMA copy
  uint32_t progress;    // 1 once the chunk is staged
  uint32_t state;       // 0 running, 1 walked and checked, 2 give up (nothing more to do)
};
constexpr uint32_t kCtlWords = 4;       // sizeof(DecompressCtl) / 4
constexpr uint32_t kPublishEvery = 16;  // the scatterer expands 16 windows at a time

template <int MAXT>
struct DecompressArgs {
  const uint32_t* in;
  uint64_t in_bytes;
  uint8_t* ws;
  uint64_t total_chunks;
  uint64_t total_items;  // total_chunks + T header checks
  uint64_t wait_limit_ns;
  uint32_t chunk_elems;
  uint32_t T;
  uint32_t batched;
  uint32_t buf_words;          // largest valid chunk: C/32 masks + C words
  uint32_t meta_offset_words;  // window table, 8-byte aligned
  uint32_t chunks_per_cta;
  uint32_t solo;               // 1: one warp walks and then scatters its chunk
  uint32_t slot_words;         // shared memory of one chunk: control, buffer, table
  uint32_t* out[MAXT];
  uint64_t n[MAXT];
  uint64_t chunk_begin[MAXT + 1];
};

__device__ __forceinline__ uint64_t get_u64_words(const uint32_t* p) {
  return (uint64_t)p[0] | ((uint64_t)p[1] << 32);
}

__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

// Warp 0: validate, stage and walk. Returns with ctl.state set to 1 (table complete and
// checked) or 2 (give up; an error is latched unless the item had no chunk).
template <int MAXT>
__device__ void walker(const DecompressArgs<MAXT>& a, DecompressCtl& ctl, uint32_t* dsm,
                       Control* ec, uint64_t item, uint32_t lane) {
  const uint32_t C = a.chunk_elems;
  uint32_t* buf = dsm + kCtlWords;
  uint2* wmeta = reinterpret_cast<uint2*>(dsm + kCtlWords + a.meta_offset_words);
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
  auto give_up = [&](uint32_t code) {
    if (code != 0 && lane == 0) latch_error(ec, code, item);
    if (lane == 0) st_release_cta(&ctl.state, 2u);
  };

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
    give_up(ok ? 0u : (uint32_t)ZVC_ERR_CORRUPT);
    return;
  }
  const uint64_t table_end = 32 + 8 * nc;
  ok = ok && se - sb >= table_end;
  if (!ok) {
    give_up(ZVC_ERR_CORRUPT);
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
    give_up(ok ? 0u : (uint32_t)ZVC_ERR_CORRUPT);
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
  if (body > 0 && lane == 0) {
    mbar_arrive_expect_tx(&ctl.full, body * 4);
    bulk_g2s(buf + head, cw + head, body * 4, &ctl.full);
  }
  if (lane < head) buf[lane] = __ldcs(cw + lane);
  if (lane < tail) buf[head + body + lane] = __ldcs(cw + head + body + lane);
  __threadfence_block();  // the end words are published with the staged flag
  __syncwarp();
  if (body > 0 && !mbar_wait(&ctl.full, 0, a.wait_limit_ns)) {
    give_up(ZVC_ERR_TIMEOUT);
    return;
  }
  __syncwarp();
  if (lane == 0) st_release_cta(&ctl.progress, 1u);  // staged: the scatterer may read the chunk

  // ---- walk the masks. The chain position -> mask -> next position is the critical
  // path. A window spans at most 33 words, so the k-th read sits below 33k <= buf_words -
  // 33 and stays in this CTA's buffer even for a corrupt chunk, and since positions only
  // grow, ending exactly at len proves that every read was inside the chunk. (For a
  // corrupt chunk the scatterer may already have expanded windows from wrong positions;
  // the output is then unspecified, but every access stays inside the buffers.)
  // Each window's (first value, mask) goes out in one 8-byte store; the first value is never
  // 0, and the table starts cleared, so the scatterer takes an entry once it reads non-zero:
  // no release per group of windows holds up the walk.
  if (lane == 0) {
    uint32_t pos = 0, m = 0;
    unsigned long long* wm = reinterpret_cast<unsigned long long*>(wmeta);
#pragma unroll 4
    for (uint32_t w = 0; w < nwin; ++w) {
      m = buf[pos];
      wm[w] = (unsigned long long)(phase + pos + 1u) | ((unsigned long long)m << 32);
      pos += 1u + __popc(m);
    }
    const uint32_t ragged = count & (kWindow - 1);
    const bool good = (pos == len) & (ragged == 0 || (m >> ragged) == 0u);
    if (!good) latch_error(ec, ZVC_ERR_CORRUPT, item);
    st_release_cta(&ctl.state, good ? 1u : 2u);
  }
}

// Warp 1: expands the recorded windows of its chunk as the walker records them.
template <int MAXT>
__device__ void scatterer(const DecompressArgs<MAXT>& a, DecompressCtl& ctl, uint32_t* dsm,
                          Control* ec, uint64_t item, uint32_t lane) {
  if (item >= a.total_chunks) return;  // header checks only: the walker does them
  const uint32_t C = a.chunk_elems;
  uint32_t ti = 0;
  if (MAXT > 1) {
    uint32_t lo = 0, hi = a.T;
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (a.chunk_begin[mid] <= item) lo = mid; else hi = mid;
    }
    ti = lo;
  }
  const uint64_t c = item - a.chunk_begin[ti];
  const uint64_t cbeg = c * C;
  const uint32_t count = (uint32_t)min((uint64_t)C, a.n[ti] - cbeg);
  const uint32_t nwin = (count + kWindow - 1) / kWindow;
  const uint32_t* buf = dsm + kCtlWords;
  const uint2* wmeta = reinterpret_cast<const uint2*>(dsm + kCtlWords + a.meta_offset_words);
  uint32_t* dst = a.out[ti] + cbeg;
  const bool vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const uint32_t e = 4u * (lane & 7u);
  const uint32_t below = (1u << e) - 1u;
  uint64_t t0 = 0;
  // bounded wait for the walker; false: give up (the walker gave up, or the wait ran out)
  auto waited = [&]() -> bool {
    if (ld_acquire_cta(&ctl.state) == 2u) return false;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > a.wait_limit_ns) {
      if (lane == 0) latch_error(ec, ZVC_ERR_TIMEOUT, item);
      return false;
    }
    __nanosleep(32);
    return true;
  };
  while (ld_acquire_cta(&ctl.progress) == 0u)  // the chunk is staged
    if (!waited()) return;
  const volatile unsigned long long* wm = reinterpret_cast<const volatile unsigned long long*>(wmeta);
  for (uint32_t g0 = 0; g0 < nwin; g0 += kPublishEvery) {
    const uint32_t need = min(nwin, g0 + kPublishEvery);
    // the group's windows: lane group l/8 takes windows g0 + l/8 + 4k, k = 0..3; each lane
    // waits (bounded) until the walker has recorded its windows
    unsigned long long ent[4];
    while (true) {
      bool all = true;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = g0 + (lane >> 3) + 4u * k;
        ent[k] = w < need ? wm[w] : 1ull;
        all &= (uint32_t)ent[k] != 0u;
      }
      if (__all_sync(0xffffffffu, all)) break;
      if (!waited()) return;
    }
    uint4 r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = g0 + (lane >> 3) + 4u * k;
      const uint32_t m = w < need ? (uint32_t)(ent[k] >> 32) : 0u;
      uint32_t q = (uint32_t)ent[k] + __popc(m & below);
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
      const uint32_t w = g0 + (lane >> 3) + 4u * k;
      if (w >= need) break;
      const uint32_t base = w * kWindow + e;
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

// A chunk of up to 2048 words walks in at most 64 steps, so one warp walks it and then
// expands it, and 8 chunks share a CTA; a larger chunk gets a walker and a scatterer warp
// and a CTA of its own.
constexpr uint32_t kSoloChunksPerCta = 8;
constexpr uint32_t kMaxThreads = 256;

template <int MAXT>
__global__ void __launch_bounds__(kMaxThreads)
    decompress_kernel(const __grid_constant__ DecompressArgs<MAXT> a) {
  extern __shared__ __align__(16) uint32_t dsm_all[];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t k = a.solo ? warp : warp >> 1;  // this warp's chunk within the CTA
  uint32_t* dsm = dsm_all + (uint64_t)k * a.slot_words;
  DecompressCtl& ctl = *reinterpret_cast<DecompressCtl*>(dsm);
  const uint64_t item = (uint64_t)blockIdx.x * a.chunks_per_cta + k;
  Control* ec = reinterpret_cast<Control*>(a.ws);
  if (lane == 0 && (a.solo || (warp & 1u) == 0)) {
    mbar_init(&ctl.full, 1);
    fence_mbar_init();
    ctl.progress = 0;
    ctl.state = 0;
  }
  // the window tables start cleared: an entry is taken once it reads non-zero
  for (uint32_t c2 = 0; c2 < a.chunks_per_cta; ++c2) {
    uint32_t* wz = dsm_all + (uint64_t)c2 * a.slot_words + kCtlWords + a.meta_offset_words;
    for (uint32_t i = threadIdx.x; i < 2u * (a.chunk_elems / kWindow); i += blockDim.x) wz[i] = 0u;
  }
  __syncthreads();
  if (item >= a.total_items) return;
  if (a.solo) {
    walker(a, ctl, dsm, ec, item, lane);
    __syncwarp();
    scatterer(a, ctl, dsm, ec, item, lane);
  } else if ((warp & 1u) == 0) {
    walker(a, ctl, dsm, ec, item, lane);
  } else {
    scatterer(a, ctl, dsm, ec, item, lane);
  }
}

template <int MAXT>
zvc_status launch_t(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts, uint32_t T,
                    bool batched, uint32_t C, uint8_t* ws, cudaStream_t stream) {
  DecompressArgs<MAXT> args;
  args.in = in;
  args.in_bytes = in_bytes;
  args.ws = ws;
  args.wait_limit_ns = kDefaultWaitLimitNs;
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
  args.slot_words = (uint32_t)round_up_u64(kCtlWords + args.meta_offset_words + 2ull * wpc, 4);
  args.solo = C <= 2048 ? 1u : 0u;
  args.chunks_per_cta = args.solo ? kSoloChunksPerCta : 1u;
  const uint32_t threads = args.solo ? 32u * kSoloChunksPerCta : 64u;
  const uint64_t smem = 4ull * args.slot_words * args.chunks_per_cta;
  cudaError_t e = cudaFuncSetAttribute(decompress_kernel<MAXT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_failure(e);
  const uint64_t blocks = ceil_div_u64(args.total_items, args.chunks_per_cta);
  const TraceMark mark = trace_begin(kTraceDecompress, stream);
  decompress_kernel<MAXT><<<(unsigned)blocks, threads, smem, stream>>>(args);
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
