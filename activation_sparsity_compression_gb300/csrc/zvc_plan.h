// Decompress launch planning, host-only arithmetic (no CUDA calls): how many words a chunk's
// shared-memory buffer holds and how many chunks a CTA takes, from the compressed stream's
// size and the device's limits. The CTAs per SM that a configuration reaches are asked of
// a callable, so the plan can be checked on a machine without a GPU.
//
// A CTA holds k chunks: lane i of its first warp walks chunk i and warp i + 1 expands it.
// Each chunk has a slot of shared memory: control words, the buffer (cap words), and the
// window table (two words per window). A chunk longer than its buffer is staged in pieces.
#pragma once

#include <stdint.h>

namespace zvc {
namespace plan {

constexpr uint32_t kWindowWords = 32;        // words per window
constexpr uint32_t kSlotCtlWords = 8;        // control words at the head of a slot
// Buffer: 5/4 of the mean chunk + 64 words, at least 1024 words (a piece then holds at least
// 31 windows), at most the largest valid chunk.
constexpr uint64_t kCapSlackNum = 5, kCapSlackDen = 4, kCapExtraWords = 64;
constexpr uint32_t kCapMinWords = 1024;
// ... and at most a dense 4096-element chunk's words (with its phase): longer chunks (C above
// 4096) go in pieces rather than holding so much shared memory that only a few are in flight.
constexpr uint32_t kCapMaxWords = 4240;
constexpr uint32_t kMaxChunksPerCta = 4;     // chunks one walker warp walks at once
constexpr uint64_t kMultiMeanDiv = 6;        // several chunks per CTA: mean <= largest / 6,
constexpr uint32_t kMultiAnyWords = 1060;    // or chunks of at most 1024 elements

struct Limits {
  int sms, smem_per_sm, reserved_per_cta, smem_per_cta_max;
};

struct Plan {
  uint32_t cap_words;       // chunk buffer, a multiple of 4 words
  uint32_t chunks_per_cta;  // 1, 2 or 4
};

inline uint64_t round_up4(uint64_t x) { return (x + 3) & ~3ull; }

// The largest valid chunk of C elements (C/32 masks + C words of wb bytes) in 4-byte words,
// at any 16-byte phase (and, for 2-byte words, starting on either half of a 4-byte word).
inline uint32_t full_cap_words(uint32_t C, uint32_t wb = 4) {
  if (wb == 2) return (uint32_t)round_up4((uint64_t)C / kWindowWords + C / 2 + 4);
  return (uint32_t)round_up4((uint64_t)C / kWindowWords + C + 3);
}

// Shared memory of one chunk's slot whose buffer holds cap words (and `extra` words more).
inline uint64_t slot_bytes(uint32_t cap, uint32_t C, uint32_t extra = 0) {
  return 4ull * round_up4(kSlotCtlWords + (uint64_t)cap + 2ull * (C / kWindowWords) + extra);
}

// The mean chunk in words: the stream's size less its headers (32 bytes per tensor, plus
// the batch header and table when batched) and chunk tables (8 bytes per table entry; a
// work item may group several table chunks, table_chunks of them in all).
inline uint64_t mean_chunk_words(uint64_t in_bytes, uint64_t chunks, uint32_t T, bool batched,
                                 uint64_t table_chunks = 0) {
  if (table_chunks < chunks) table_chunks = chunks;
  const uint64_t fixed = (batched ? 16ull + 8ull * ((uint64_t)T + 1) : 0ull) + 32ull * T +
                         8ull * table_chunks;
  return in_bytes > fixed && chunks > 0 ? (in_bytes - fixed) / 4 / chunks : 0;
}

// The plan for `chunks` chunks of C elements in a stream of in_bytes bytes. occ(k, cap)
// returns how many CTAs of k chunks with buffers of cap words fit on one SM (0 if none).
// Returns false if occ reports an error (a negative count).
//
// - The buffer is sized from the mean chunk (a CTA's shared memory is fixed at launch and
//   sets how many chunks are in flight per SM): chunks up to 5/4 of the mean go in one piece.
// - With short chunks (a mean of at most 1/6 of the largest, or chunks of at most 1024
//   elements) in a launch of two waves or more, k is the chunks per CTA (1, 2 or 4) that
//   keeps the most chunks in flight per SM, more per CTA on a tie: the kernel is then
//   bound by the instructions it issues, and a shared walker warp issues a quarter of them
//   per chunk. Otherwise k = 1: a CTA frees its shared memory only when its slowest chunk
//   is done.
// - Then the buffer is widened to the largest that keeps the CTAs per SM the launch needs:
//   as many as fit, or fewer when fewer hold every chunk in as many waves. A larger buffer
//   stages fewer chunks in pieces.
template <class Occ>
bool decompress_plan(uint64_t chunks, uint64_t in_bytes, uint32_t T, bool batched, uint32_t C,
                     const Limits& d, Occ occ, Plan* out, uint32_t wb = 4,
                     uint64_t table_chunks = 0, uint32_t extra = 0) {
  const uint32_t full_cap = full_cap_words(C, wb);
  out->cap_words = full_cap;
  out->chunks_per_cta = 1;
  if (chunks == 0) return true;
  uint64_t mean = mean_chunk_words(in_bytes, chunks, T, batched, table_chunks);
  if (mean > full_cap) mean = full_cap;
  uint64_t want = round_up4(mean * kCapSlackNum / kCapSlackDen + kCapExtraWords);
  if (want < kCapMinWords) want = kCapMinWords;
  if (want > kCapMaxWords) want = kCapMaxWords;
  uint32_t cap = want < full_cap ? (uint32_t)want : full_cap;

  int o1 = occ(1u, cap);
  if (o1 < 0) return false;
  uint32_t k = 1;
  int best_occ = o1;
  const bool short_chunks = mean * kMultiMeanDiv <= full_cap || full_cap <= kMultiAnyWords;
  const bool waves2 = o1 > 0 && chunks >= 2ull * (uint64_t)o1 * (uint64_t)d.sms;
  uint64_t best = (uint64_t)o1;
  for (uint32_t kk = 2; short_chunks && waves2 && kk <= kMaxChunksPerCta; kk *= 2) {
    if (kk * slot_bytes(cap, C, extra) > (uint64_t)d.smem_per_cta_max) break;
    const int o = occ(kk, cap);
    if (o < 0) return false;
    if (o > 0 && (uint64_t)o * kk >= best) {
      best = (uint64_t)o * kk;
      k = kk;
      best_occ = o;
    }
  }
  out->chunks_per_cta = k;
  out->cap_words = cap;
  if (best_occ <= 0 || d.sms <= 0 || cap >= full_cap) return true;
  const uint64_t ctas = (chunks + k - 1) / k;
  const uint64_t per_wave = (uint64_t)best_occ * (uint64_t)d.sms;
  const uint64_t waves = (ctas + per_wave - 1) / per_wave;
  const uint64_t need = (ctas + waves * d.sms - 1) / (waves * d.sms);  // CTAs per SM
  uint64_t per_cta = (uint64_t)d.smem_per_sm / need;
  const uint64_t cta_max = (uint64_t)d.smem_per_cta_max + (uint64_t)d.reserved_per_cta;
  if (per_cta > cta_max) per_cta = cta_max;
  const uint64_t fixed = (uint64_t)d.reserved_per_cta +
                         4ull * k * (kSlotCtlWords + round_up4(2ull * (C / kWindowWords) + extra));
  if (per_cta <= fixed + 16ull * k) return true;
  uint64_t c = ((per_cta - fixed) / (4ull * k)) & ~3ull;
  if (c > full_cap) c = full_cap;
  if (c <= cap) return true;
  const int o2 = occ(k, (uint32_t)c);
  if (o2 < 0) return false;
  if ((uint64_t)o2 >= need) out->cap_words = (uint32_t)c;
  return true;
}

}  // namespace plan
}  // namespace zvc
