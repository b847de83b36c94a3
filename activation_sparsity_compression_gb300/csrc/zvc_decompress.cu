// ZVC decompress for sm_103a: the inverse of Rhu et al., "Compressing DMA Engine",
// section V.A (every set mask bit takes the next packed word, every clear bit is a zero;
// section V.B has the engine expand compressed data into 128-byte lines using the masks'
// prefix counts as scatter offsets).
//
// A chunk, located through the stream's chunk offset table, is decoded by a walker (one
// thread) and a scatterer (one warp). A CTA holds k chunks (k = 1, or 2 or 4 for short
// chunks): lane i of warp 0 walks chunk i and warp i + 1 scatters it.
// The walker:
//   validate  batch table (if any), stream header and this chunk's table entries; every
//             check that fails latches ZVC_ERR_CORRUPT before any access to the chunk
//   stage     the chunk's compressed words are copied into shared memory by a 1-D TMA
//             bulk copy (plain loads for the unaligned ends), at their 16-byte phase; the
//             buffer is sized on the host from the stream's mean chunk, and a longer
//             chunk goes in pieces, each started once the scatterer has drained the last
//   walk      a window's position depends on every earlier mask, so one thread walks the
//             masks (position += 1 + popc(mask)), recording each window's (first value,
//             mask) in one 8-byte store into a table that starts cleared; the walk must
//             end exactly at the next chunk's offset
// The scatterer expands windows as soon as it reads their entries non-zero, so the scatter
// runs under the walk: lane l expands words 4(l mod 8) .. +3 of window l/8 + 4k of each
// group of 16 windows, a set bit at position b reading packed word popc(mask & (2^b - 1)),
// a clear bit writing 0, with 16-byte stores.
// Extra work items (one per tensor, after the chunks) check the headers of streams that
// have no chunks; an empty batch gets one item that checks its header and table.
#include <atomic>

#include "zvc_internal.cuh"
#include "zvc_plan.h"

namespace zvc {
namespace {

// A work item is a group of up to `group` consecutive chunks of one tensor (group = 1 for
// C >= 4096; for smaller chunks up to 8, so that an item covers up to 4096 elements): they
// lie back to back in the stream, so one copy stages them and one walk decodes them, and
// the per-item costs (locating and staging, a CTA's start) are paid once per group.
//
// Shared memory of an item's slot: control words, then the item's buffer (cap words, at
// most its masks + words + 3 for the 16-byte phase), then the window table (first value,
// mask) per window, then (grouped items only) kBndWords words where the walker keeps the
// starts of the item's inner chunks. A CTA holds chunks_per_cta slots. Grouped items have
// a kernel instantiation of their own (GRP), so the C >= 4096 kernel carries none of it.
constexpr uint32_t kMaxGroup = 8;
constexpr uint32_t kBndWords = kMaxGroup;
struct DecompressCtl {
  uint64_t full;      // mbarrier of the TMA copies, one phase per bulk copy
  uint32_t progress;  // pieces of the item staged so far
  uint32_t state;     // 0 running, 1 walked and checked, 2 give up (nothing more to do)
  uint32_t drain;     // 0, or the window the next piece starts at (walker -> scatterer)
  uint32_t expanded;  // the windows before it are read out of the buffer (scatterer -> walker)
  uint32_t pad[2];
};
constexpr uint32_t kCtlWords = plan::kSlotCtlWords;  // sizeof(DecompressCtl) / 4: 16-byte aligned
static_assert(sizeof(DecompressCtl) == 4 * kCtlWords, "control words");
constexpr uint32_t kPublishEvery = 16;  // the scatterer expands 16 windows at a time
constexpr uint32_t kPollSleepNs = 32;   // the scatterer's sleep between polls of the table
constexpr uint32_t kStageSuspendNs = 2000;  // the scatterer's barrier wait for the first piece

// mbarrier.try_wait with a suspend hint of HINT ns.
template <uint32_t HINT>
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "n"(HINT)
      : "memory");
  return done != 0;
}

// WB is the word size in bytes: 4 (any 32-bit type) or 2 (bf16 / fp16, single streams).
// Positions inside a chunk are counted in units of one word; a mask is 4 / WB units, and a
// 16-byte group holds 16 / WB units.
template <int WB> struct WordOf;
template <> struct WordOf<4> { using T = uint32_t; };
template <> struct WordOf<2> { using T = uint16_t; };

template <int MAXT, int WB>
struct DecompressArgs {
  const uint32_t* in;
  uint64_t in_bytes;
  uint8_t* ws;
  uint64_t total_chunks;  // work items that decode chunks (groups of up to `group` chunks)
  uint64_t total_items;   // total_chunks + T header checks
  uint64_t wait_limit_ns;
  uint32_t chunk_elems;
  uint32_t group;         // chunks per work item
  uint32_t T;
  uint32_t batched;
  uint32_t cap_words;          // chunk buffer words (a multiple of 4): longer chunks go in pieces
  uint32_t meta_offset_words;  // window table, 8-byte aligned
  uint32_t chunks_per_cta;
  uint32_t slot_words;         // shared memory of one chunk: control, buffer, table
  typename WordOf<WB>::T* out[MAXT];
  uint64_t n[MAXT];
  uint64_t chunk_begin[MAXT + 1];  // first work item of tensor i
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

// One thread per chunk: validate, stage and walk. Returns with ctl.state set to 1 (table
// complete and checked) or 2 (give up; an error is latched unless the item had no chunk).
template <int MAXT, int WB, bool GRP>
__device__ void walker(const DecompressArgs<MAXT, WB>& a, DecompressCtl& ctl, uint32_t* dsm,
                       Control* ec, uint64_t item) {
  using Word = typename WordOf<WB>::T;
  constexpr uint32_t MU = 4u / WB;   // units of a mask
  constexpr uint32_t UPG = 16u / WB; // units of a 16-byte group
  const uint32_t C = a.chunk_elems;
  const uint32_t group = GRP ? a.group : 1u;
  Word* buf = reinterpret_cast<Word*>(dsm + kCtlWords);
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
    c = (item - a.chunk_begin[ti]) * group;  // the item's first chunk
  } else {
    ti = (uint32_t)(item - a.total_chunks);
  }
  const uint64_t n = ti < a.T ? a.n[ti] : 0;
  const uint64_t nc = ceil_div_u64(n, C);
  // the item's chunks (1 without grouping)
  const uint32_t gc = GRP ? (is_chunk ? (uint32_t)min((uint64_t)group, nc - c) : 0u) : 1u;
  auto give_up = [&](uint32_t code) {
    if (code != 0) latch_error(ec, code, item);
    st_release_cta(&ctl.state, 2u);
  };

  // ---- locate and validate the stream. Every
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
  const uint32_t count =
      is_chunk ? (uint32_t)min((uint64_t)(GRP ? gc * C : C), n - cbeg) : 0u;
  const uint32_t nwin = (count + kWindow - 1) / kWindow;
  uint64_t start = 0, end = payload;
  if (is_chunk) {
    const uint32_t* ct = sw + kStreamHeaderWords + 2 * c;
    start = get_u64_words(ct);
    if constexpr (GRP) {
      if (c + gc < nc) end = get_u64_words(ct + 2 * gc);
    } else {
      if (c + 1 < nc) end = get_u64_words(ct + 2);
    }
  }
  ok = (h[0] == kStreamMagic) & (h[1] == (1u | ((uint32_t)WB << 16))) & (h[2] == kWindow) &
       (h[3] == C) &
       (((uint64_t)h[4] | ((uint64_t)h[5] << 32)) == n) &
       (((uint64_t)h[6] | ((uint64_t)h[7] << 32)) == payload);
  if (is_chunk)
    ok = ok & ((c != 0) | (start == 0)) & (start <= end) & (end <= payload) &
         (((start | end) & (uint64_t)(WB - 1)) == 0) && (end - start) / WB >= (uint64_t)MU * nwin &&
         (end - start) / WB <= (uint64_t)MU * nwin + count;
  if (!ok || !is_chunk) {
    give_up(ok ? 0u : (uint32_t)ZVC_ERR_CORRUPT);
    return;
  }

  // ---- stage the chunk: its units sit in shared memory at the same 16-byte phase as in
  // global memory, so one bulk copy moves the aligned body and plain loads the at most
  // UPG - 1 units on either side. The buffer holds cap units; a longer chunk is staged in
  // pieces (below), the first piece being its first cap - phase units.
  const uint32_t len = (uint32_t)((end - start) / WB);
  const Word* cw = reinterpret_cast<const Word*>(sw) + (4ull * kStreamHeaderWords + 8 * nc + start) / WB;
  const uint32_t cap = a.cap_words * (4u / WB);
  uint32_t ph = (uint32_t)((reinterpret_cast<uintptr_t>(cw) / WB) & (UPG - 1));
  uint32_t e = min(len, cap - ph);  // chunk units [s, e) are staged, s = 0 here
  uint32_t fills = 0;                // bulk copies completed on ctl.full (its phase)
  {
    const uint32_t head = min(e, (UPG - ph) & (UPG - 1));
    const uint32_t body = (e - head) & ~(UPG - 1);
    const uint32_t tail = e - head - body;
    Word x[2 * (UPG - 1)];
#pragma unroll
    for (uint32_t i = 0; i < UPG - 1; ++i) {
      x[i] = i < head ? __ldcs(cw + i) : (Word)0;
      x[UPG - 1 + i] = i < tail ? __ldcs(cw + head + body + i) : (Word)0;
    }
    if (body > 0) {
      mbar_arrive_expect_tx(&ctl.full, body * WB);
      bulk_g2s(buf + ph + head, cw + head, body * WB, &ctl.full);
    }
#pragma unroll
    for (uint32_t i = 0; i < UPG - 1; ++i) {
      if (i < head) buf[ph + i] = x[i];
      if (i < tail) buf[ph + head + body + i] = x[UPG - 1 + i];
    }
    if (body > 0 && !mbar_wait(&ctl.full, 0, a.wait_limit_ns)) {
      give_up(ZVC_ERR_TIMEOUT);
      return;
    }
    fills = body > 0 ? 1u : 0u;
  }
  st_release_cta(&ctl.progress, 1u);  // staged: the scatterer may read the piece
  // The table entries of the item's inner chunks: where each must start, in units from the
  // item's start (an entry outside the item or off a unit boundary can match no window).
  uint32_t* bnd = dsm + kCtlWords + a.meta_offset_words + 2 * (group * C / kWindow);
  if constexpr (GRP) {
    const uint32_t* ct = sw + kStreamHeaderWords + 2 * c;
    uint64_t x[kMaxGroup - 1];
#pragma unroll
    for (uint32_t j = 1; j < kMaxGroup; ++j) x[j - 1] = j < gc ? get_u64_words(ct + 2 * j) : 0;
#pragma unroll
    for (uint32_t j = 1; j < kMaxGroup; ++j)
      if (j < gc)
        bnd[j - 1] = (x[j - 1] >= start && x[j - 1] <= end && (x[j - 1] & (uint64_t)(WB - 1)) == 0)
                         ? (uint32_t)((x[j - 1] - start) / WB)
                         : 0xFFFFFFFFu;
  }

  // ---- walk the masks. The chain position -> mask -> next position is the critical
  // path. A window spans at most 33 words, so from buffer position bp the next
  // (cap - bp) / 33 windows lie inside the buffer and are walked without checks; the rest
  // one by one. Inside the buffer means staged, except in the chunk's last piece, where
  // only a corrupt chunk reads past its end: positions only grow, so ending exactly at len
  // proves that every read was inside the chunk. (For a corrupt chunk the scatterer may
  // already have expanded windows from wrong positions; the output is then unspecified,
  // but every access stays inside the buffers.)
  // Each window's (first value, mask) goes out in one 8-byte store; the first value is never
  // 0, and the table starts cleared, so the scatterer takes an entry once it reads non-zero:
  // no release per group of windows holds up the walk.
  // A window that runs past the buffer before the chunk's end starts the next piece: the
  // walker asks the scatterer to expand every window recorded so far (drain), waits until
  // it has, and stages the chunk from that window on.
  unsigned long long* wm = reinterpret_cast<unsigned long long*>(wmeta);
  uint32_t s = 0, bp = ph, m = 0, w = 0, piece = 1;
  bool good = true;
  // Each inner chunk of the item must start exactly where the walk reaches its first window
  // (the chunk table's rule). Checked after every step, from the window table (or, for the
  // window walked next, bp), while the positions still refer to the current piece.
  const uint32_t wpc = C / kWindow;
  uint32_t jb = 1, nb = wpc;  // the next inner chunk and its first window
  auto check_bounds = [&]() {
    if constexpr (GRP) {
      while (jb < gc && nb <= w) {
        const uint32_t at = nb < w ? (uint32_t)wm[nb] - MU : bp;
        good = good && s + (at - ph) == bnd[jb - 1];
        ++jb;
        nb += wpc;
      }
    }
  };
  // the mask at unit p (for WB = 2 it may sit on a 2-byte boundary: two 16-bit loads)
  auto mask_at = [&](uint32_t p) -> uint32_t {
    if (WB == 4) return (uint32_t)buf[p];
    return (uint32_t)buf[p] | ((uint32_t)buf[p + 1] << 16);
  };
  while (w < nwin) {
    const uint32_t k = min(nwin - w, (cap - bp) / (kWindow + MU));
    if (k > 0) {
      const uint32_t w1 = w + k;
#pragma unroll 4
      for (; w < w1; ++w) {
        m = mask_at(bp);
        wm[w] = (unsigned long long)(bp + MU) | ((unsigned long long)m << 32);
        bp += MU + __popc(m);
      }
      check_bounds();
      continue;
    }
    if (bp + MU <= cap) {
      m = mask_at(bp);
      const uint32_t nb = bp + MU + __popc(m);
      if (nb <= cap) {
        wm[w] = (unsigned long long)(bp + MU) | ((unsigned long long)m << 32);
        bp = nb;
        ++w;
        check_bounds();
        continue;
      }
    }
    // the window runs past the buffer: past the chunk in its last piece (corrupt), else
    // the next piece starts at this window
    if (e >= len) {
      good = false;
      break;
    }
    const uint32_t pos = s + (bp - ph);
    st_release_cta(&ctl.drain, w);
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_cta(&ctl.expanded) != w) {
      if (globaltimer_ns() - t0 > a.wait_limit_ns) {
        latch_error(ec, ZVC_ERR_TIMEOUT, item);
        st_release_cta(&ctl.state, 2u);
        return;
      }
      __nanosleep(64);
    }
    fence_proxy_async_smem();  // the scatterer's reads come before the copy's writes
    // The piece starts at this window's 16-byte group: the at most UPG - 1 units before it
    // are the stream's (a chunk is preceded by the header and table at least), so one bulk
    // copy moves every whole group that fits; a piece that reaches the chunk's end loads
    // the units past its last group with plain loads, under the copy.
    s = pos;
    ph = (uint32_t)((reinterpret_cast<uintptr_t>(cw + s) / WB) & (UPG - 1));
    const Word* src = cw + s - ph;                    // 16-byte aligned
    const uint32_t n = min(len - s + ph, cap);        // units of this piece, from src
    const uint32_t body = n & ~(UPG - 1);             // cap is a multiple of UPG
    const uint32_t rest = n - body;                   // only at the chunk's end: < UPG
    e = s - ph + n;
    Word x[UPG - 1];
#pragma unroll
    for (uint32_t i = 0; i < UPG - 1; ++i) x[i] = i < rest ? __ldcs(src + body + i) : (Word)0;
    if (body > 0) {
      mbar_arrive_expect_tx(&ctl.full, body * WB);
      bulk_g2s(buf, src, body * WB, &ctl.full);
    }
#pragma unroll
    for (uint32_t i = 0; i < UPG - 1; ++i)
      if (i < rest) buf[body + i] = x[i];
    if (body > 0) {
      if (!mbar_wait(&ctl.full, fills & 1u, a.wait_limit_ns)) {
        latch_error(ec, ZVC_ERR_TIMEOUT, item);
        st_release_cta(&ctl.state, 2u);
        return;
      }
      ++fills;
    }
    ++piece;
    st_release_cta(&ctl.progress, piece);
    bp = ph;
  }
  const uint32_t ragged = count & (kWindow - 1);
  good = good & (s + (bp - ph) == len) & (ragged == 0 || (m >> ragged) == 0u);
  if (!good) latch_error(ec, ZVC_ERR_CORRUPT, item);
  st_release_cta(&ctl.state, good ? 1u : 2u);
}

// Warp 1: expands the recorded windows of its chunk as the walker records them.
template <int MAXT, int WB, bool GRP>
__device__ void scatterer(const DecompressArgs<MAXT, WB>& a, DecompressCtl& ctl, uint32_t* dsm,
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
  const uint64_t c = GRP ? (item - a.chunk_begin[ti]) * a.group : item - a.chunk_begin[ti];
  const uint64_t cbeg = c * C;
  const uint32_t count = (uint32_t)min((uint64_t)(GRP ? a.group * C : C), a.n[ti] - cbeg);
  using Word = typename WordOf<WB>::T;
  constexpr uint32_t EPL = 16u / WB;       // units a lane expands: one 16-byte store
  constexpr uint32_t LPW = kWindow / EPL;  // lanes per window: 8 (WB = 4) or 4 (WB = 2)
  constexpr uint32_t WPI = 32u / LPW;      // windows per pass of the warp: 4 or 8
  constexpr int KW = (int)(kPublishEvery / WPI);  // passes per group of 16 windows
  const uint32_t nwin = (count + kWindow - 1) / kWindow;
  const Word* buf = reinterpret_cast<const Word*>(dsm + kCtlWords);
  const uint2* wmeta = reinterpret_cast<const uint2*>(dsm + kCtlWords + a.meta_offset_words);
  Word* dst = a.out[ti] + cbeg;
  const bool vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const uint32_t e = EPL * (lane % LPW);
  const uint32_t below = (1u << e) - 1u;
  uint64_t t0 = 0;
  // bounded wait for the walker; false: give up (the walker gave up, or the wait ran out)
  auto waited = [&](uint32_t sleep_ns) -> bool {
    if (ld_acquire_cta(&ctl.state) == 2u) return false;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) t0 = now;
    if (now - t0 > a.wait_limit_ns) {
      if (lane == 0) latch_error(ec, ZVC_ERR_TIMEOUT, item);
      return false;
    }
    __nanosleep(sleep_ns);
    return true;
  };
  uint32_t piece = 1;  // the piece of the chunk in the buffer
  // The first piece: a hardware wait on the bulk copy's barrier (the warp sleeps until the
  // copy lands), then the walker's staged count, which also covers its plain loads. A
  // chunk too short for a bulk copy, or a walker that gave up, ends the barrier wait at
  // the suspend hint.
  while (ld_acquire_cta(&ctl.progress) < piece) {
    if (mbar_try_wait_hint<kStageSuspendNs>(&ctl.full, 0u)) {
      while (ld_acquire_cta(&ctl.progress) < piece)
        if (!waited(16)) return;
      break;
    }
    if (!waited(0)) return;
  }
  const volatile unsigned long long* wm =
      reinterpret_cast<const volatile unsigned long long*>(wmeta);
  const volatile uint32_t* drain = &ctl.drain;
  uint32_t g0 = 0, handled = 0;
  while (g0 < nwin) {
    const uint32_t need = min(nwin, g0 + kPublishEvery);
    // the group's windows: lane group l/LPW takes windows g0 + l/LPW + WPI k; each lane
    // waits (bounded) until the walker has recorded its windows, or until the walker asks
    // for the windows before d to be expanded (it stages the next piece from window d)
    unsigned long long ent[KW];
    uint32_t lim, d;
    while (true) {
      d = *drain;
      lim = (d > handled && d <= need) ? d : need;
      bool all = true;
#pragma unroll
      for (int k = 0; k < KW; ++k) {
        const uint32_t w = g0 + lane / LPW + WPI * k;
        ent[k] = w < lim ? wm[w] : 1ull;
        all &= (uint32_t)ent[k] != 0u;
      }
      if (__all_sync(0xffffffffu, all)) break;
      if (!waited(kPollSleepNs)) return;
    }
    uint4 r[KW];
#pragma unroll
    for (int k = 0; k < KW; ++k) {
      const uint32_t w = g0 + lane / LPW + WPI * k;
      const uint32_t m = w < lim ? (uint32_t)(ent[k] >> 32) : 0u;
      uint32_t q = (uint32_t)ent[k] + __popc(m & below);
      uint32_t v[EPL];
#pragma unroll
      for (uint32_t j = 0; j < EPL; ++j) {
        const uint32_t bit = (m >> (e + j)) & 1u;
        v[j] = bit ? (uint32_t)buf[q] : 0u;
        q += bit;
      }
      if constexpr (WB == 4)
        r[k] = make_uint4(v[0], v[1], v[2], v[3]);
      else
        r[k] = make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16),
                          v[6] | (v[7] << 16));
    }
#pragma unroll
    for (int k = 0; k < KW; ++k) {
      const uint32_t w = g0 + lane / LPW + WPI * k;
      if (w >= lim) break;
      const uint32_t base = w * kWindow + e;
      if (vec && base + EPL <= count) {
        *reinterpret_cast<uint4*>(dst + base) = r[k];
      } else {
        const uint32_t vv[4] = {r[k].x, r[k].y, r[k].z, r[k].w};
#pragma unroll
        for (uint32_t j = 0; j < EPL; ++j) {
          if constexpr (WB == 4) {
            if (base + j < count) dst[base + j] = vv[j];
          } else {
            if (base + j < count) dst[base + j] = (Word)(vv[j / 2] >> (16u * (j & 1u)));
          }
        }
      }
    }
    g0 = lim;
    if (lim == d && d > handled) {
      // every window before d is read out of the buffer: hand it back, wait for the next piece
      handled = d;
      ++piece;
      __syncwarp();
      if (lane == 0) st_release_cta(&ctl.expanded, d);
      while (ld_acquire_cta(&ctl.progress) < piece)
        if (!waited(64)) return;
    }
  }
}

// Chunks per work item: 1 from 4096 elements on, else up to kMaxGroup chunks of up to 4096
// elements in all (measured: at C = 1024 sparse maps decode at 0.61-0.66 of HBM one chunk
// per item, as C = 4096 chunks do at 0.88-0.97).
__host__ __device__ inline uint32_t group_of(uint32_t C) {
  return C >= kTileElems ? 1u : min(kMaxGroup, kTileElems / C);
}

// Every item gets a scatterer warp of its own and a lane of the CTA's walker warp; the
// host picks the items per CTA and the buffer's size (zvc_plan.h).
constexpr uint32_t kMaxThreads = 32 * (1 + plan::kMaxChunksPerCta);
// Chunks of at most 1024 elements are bound by the chunks in flight per SM, which registers
// limit: their kernel is built for 10 CTAs of kMaxThreads per SM (32 registers; measured
// 8% faster there, and 7-22% slower for 4096-element chunks).
constexpr uint32_t kSmallChunkElems = 1024;
constexpr uint32_t kSmallMinCtas = 10;

template <int MAXT, int WB, bool SMALL, bool GRP>
__global__ void __launch_bounds__(kMaxThreads, SMALL ? kSmallMinCtas : 0)
    decompress_kernel(const __grid_constant__ DecompressArgs<MAXT, WB> a) {
  extern __shared__ __align__(16) uint32_t dsm_all[];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  // this thread's chunk within the CTA: lane k of warp 0 walks chunk k, warp k + 1
  // scatters it
  const uint32_t k = warp == 0 ? min(lane, a.chunks_per_cta - 1) : warp - 1;
  uint32_t* dsm = dsm_all + (uint64_t)k * a.slot_words;
  DecompressCtl& ctl = *reinterpret_cast<DecompressCtl*>(dsm);
  const uint64_t item = (uint64_t)blockIdx.x * a.chunks_per_cta + k;
  Control* ec = reinterpret_cast<Control*>(a.ws);
  if (threadIdx.x < a.chunks_per_cta) {
    DecompressCtl& c0 =
        *reinterpret_cast<DecompressCtl*>(dsm_all + (uint64_t)threadIdx.x * a.slot_words);
    mbar_init(&c0.full, 1);
    fence_mbar_init();
    c0.progress = 0;
    c0.state = 0;
    c0.drain = 0;
    c0.expanded = 0;
  }
  // the window tables start cleared: an entry is taken once it reads non-zero
  for (uint32_t c2 = 0; c2 < a.chunks_per_cta; ++c2) {
    uint32_t* wz = dsm_all + (uint64_t)c2 * a.slot_words + kCtlWords + a.meta_offset_words;
    for (uint32_t i = threadIdx.x; i < 2u * ((GRP ? a.group : 1u) * a.chunk_elems / kWindow);
         i += blockDim.x)
      wz[i] = 0u;
  }
  __syncthreads();
  if (warp == 0) {
    if (lane < a.chunks_per_cta && item < a.total_items) walker<MAXT, WB, GRP>(a, ctl, dsm, ec, item);
  } else {
    if (item >= a.total_items) return;
    scatterer<MAXT, WB, GRP>(a, ctl, dsm, ec, item, lane);
  }
}

// The device's SM count and shared memory, read once per device.
zvc_status device_limits(plan::Limits* d) {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> sms_of[kMaxDevices], smem_of[kMaxDevices], reserved_of[kMaxDevices],
      cta_max_of[kMaxDevices];
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_failure(e);
  if (dev < 0 || dev >= kMaxDevices) return ZVC_ERR_INVALID_ARG;
  d->sms = sms_of[dev].load();
  d->smem_per_sm = smem_of[dev].load();
  d->reserved_per_cta = reserved_of[dev].load();
  d->smem_per_cta_max = cta_max_of[dev].load();
  if (d->sms == 0) {
    if ((e = cudaDeviceGetAttribute(&d->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d->reserved_per_cta, cudaDevAttrReservedSharedMemoryPerBlock,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d->smem_per_cta_max, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_failure(e);
    smem_of[dev].store(d->smem_per_sm);
    reserved_of[dev].store(d->reserved_per_cta);
    cta_max_of[dev].store(d->smem_per_cta_max);
    sms_of[dev].store(d->sms);
  }
  return ZVC_OK;
}

template <int MAXT, int WB, bool SMALL, bool GRP>
zvc_status launch_k(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts, uint32_t T,
                    bool batched, uint32_t C, uint8_t* ws, cudaStream_t stream) {
  static_assert(WB == 4 || MAXT == 1, "16-bit words: single streams only");
  DecompressArgs<MAXT, WB> args;
  args.in = in;
  args.in_bytes = in_bytes;
  args.ws = ws;
  args.wait_limit_ns = kDefaultWaitLimitNs;
  args.chunk_elems = C;
  args.group = GRP ? group_of(C) : 1u;
  args.T = T;
  args.batched = batched ? 1u : 0u;
  const uint32_t IC = args.group * C;  // elements of a whole work item
  uint64_t chunks = 0, table_chunks = 0;
  for (uint32_t i = 0; i < T; ++i) {
    args.out[i] = static_cast<typename WordOf<WB>::T*>(ts[i].ptr);
    args.n[i] = ts[i].n;
    args.chunk_begin[i] = chunks;
    chunks += ceil_div_u64(ceil_div_u64(ts[i].n, C), args.group);
    table_chunks += ceil_div_u64(ts[i].n, C);
  }
  args.chunk_begin[T] = chunks;
  args.total_chunks = chunks;
  args.total_items = chunks + (batched && T == 0 ? 1 : T);
  const uint32_t wpc = IC / kWindow;  // windows of a whole work item
  const uint32_t full_cap = plan::full_cap_words(IC, WB);
  plan::Limits d;
  zvc_status st = device_limits(&d);
  if (st != ZVC_OK) return st;
  // the most shared memory a CTA of this chunk size can ask for (within the device's
  // limit), and all of the SM's unified memory as shared memory
  const uint32_t extra = GRP ? kBndWords : 0u;  // the inner chunks' starts
  const uint64_t most = plan::slot_bytes(full_cap, IC, extra) * plan::kMaxChunksPerCta;
  cudaError_t e = cudaFuncSetAttribute(
      decompress_kernel<MAXT, WB, SMALL, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)min(most, (uint64_t)d.smem_per_cta_max));
  if (e != cudaSuccess) return cuda_failure(e);
  e = cudaFuncSetAttribute(decompress_kernel<MAXT, WB, SMALL, GRP>,
                           cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return cuda_failure(e);
  // the buffer's size and the chunks per CTA, with the occupancy the runtime reports
  cudaError_t occ_err = cudaSuccess;
  auto occ = [&](uint32_t k, uint32_t cap) -> int {
    int n = 0;
    const cudaError_t r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &n, decompress_kernel<MAXT, WB, SMALL, GRP>, (int)(32 * (1 + k)),
        (size_t)(k * plan::slot_bytes(cap, IC, extra)));
    if (r != cudaSuccess) {
      occ_err = r;
      return -1;
    }
    return n;
  };
  plan::Plan pl;
  if (!plan::decompress_plan(chunks, in_bytes, T, batched, IC, d, occ, &pl, WB,
                             table_chunks, extra))
    return cuda_failure(occ_err);
  args.cap_words = pl.cap_words;
  args.chunks_per_cta = pl.chunks_per_cta;
  args.meta_offset_words = args.cap_words;
  args.slot_words = (uint32_t)round_up_u64(kCtlWords + args.cap_words + 2ull * wpc + extra, 4);
  const uint64_t smem = 4ull * args.slot_words * args.chunks_per_cta;
  const uint32_t threads = 32u * (1u + args.chunks_per_cta);
  const uint64_t blocks = ceil_div_u64(args.total_items, args.chunks_per_cta);
  const TraceMark mark = trace_begin(kTraceDecompress, stream);
  decompress_kernel<MAXT, WB, SMALL, GRP><<<(unsigned)blocks, threads, smem, stream>>>(args);
  trace_end(mark, stream);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

template <int MAXT, int WB>
zvc_status launch_t(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts, uint32_t T,
                    bool batched, uint32_t C, uint8_t* ws, cudaStream_t stream) {
  const bool grp = group_of(C) > 1;
  const bool small = group_of(C) * C <= kSmallChunkElems;
  if (grp && small) return launch_k<MAXT, WB, true, true>(in, in_bytes, ts, T, batched, C, ws, stream);
  if (grp) return launch_k<MAXT, WB, false, true>(in, in_bytes, ts, T, batched, C, ws, stream);
  if (small) return launch_k<MAXT, WB, true, false>(in, in_bytes, ts, T, batched, C, ws, stream);
  return launch_k<MAXT, WB, false, false>(in, in_bytes, ts, T, batched, C, ws, stream);
}

}  // namespace

zvc_status launch_decompress(const uint32_t* in, uint64_t in_bytes, const TensorOut* ts,
                             uint32_t T, bool batched, uint32_t chunk_elems, uint8_t* ws,
                             cudaStream_t stream) {
  if (!batched && T == 1)
    return launch_t<1, 4>(in, in_bytes, ts, T, false, chunk_elems, ws, stream);
  if (T <= 64) return launch_t<64, 4>(in, in_bytes, ts, T, batched, chunk_elems, ws, stream);
  return launch_t<ZVC_MAX_BATCH, 4>(in, in_bytes, ts, T, batched, chunk_elems, ws, stream);
}

zvc_status launch_decompress16(const uint32_t* in, uint64_t in_bytes, uint16_t* out, uint64_t n,
                               uint32_t chunk_elems, uint8_t* ws, cudaStream_t stream) {
  const TensorOut t{out, n};
  return launch_t<1, 2>(in, in_bytes, &t, 1, false, chunk_elems, ws, stream);
}

}  // namespace zvc
