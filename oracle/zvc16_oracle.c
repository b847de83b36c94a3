/*
 * ZVC oracle for 16-bit activation words (bf16 / fp16): TEST INFRASTRUCTURE ONLY.
 *
 * Rhu et al., "Compressing DMA Engine: Leveraging Activation Sparsity for Training Deep
 * Neural Networks" (arXiv:1705.01626), section V.A "Compression Algorithm", describes
 * ZVC on 32 activation values with one 32-bit zero/non-zero mask followed by the
 * non-zero values; its evaluation uses 32-bit activations. This file applies the same
 * rule to 16-bit activation words, a reading beyond the pages: the window stays 32
 * values with a 32-bit mask, and the non-zero values that follow are 2 bytes each.
 * Section VII.A "Compression Efficiency" (larger windows give similar results) is why
 * the chunk size C stays a free parameter, as in the 32-bit stream.
 *
 * Layout (little-endian, no padding anywhere; the same framing as the 32-bit stream
 * with word_bytes = 2):
 *   +0   u32 magic 0x3143565A ("ZVC1")
 *   +4   u16 version = 1
 *   +6   u16 word_bytes = 2
 *   +8   u32 window = 32
 *   +12  u32 chunk_elems C (a positive multiple of 32)
 *   +16  u64 n, the number of 16-bit words
 *   +24  u64 payload_bytes
 *   +32  u64 chunk_off[nc], nc = ceil(n / C): byte offset of chunk c inside the payload
 *   +32+8nc  payload: chunk 0 | chunk 1 | ...
 *   chunk c = for each window of the chunk, in order: u32 mask, then the 16-bit words
 *     whose mask bit is set, in ascending element order, 2 bytes each. Bit i of a mask is
 *     element i of the window (least significant bit first). A word is zero iff its 16
 *     bits are all clear, so -0.0 (0x8000), NaNs and denormals are carried as non-zero
 *     words. In the last window of the stream, bits at or beyond n are clear. Windows
 *     follow each other without padding, so a mask starts on a 2-byte boundary that need
 *     not be a 4-byte one.
 *   Size: 32 + 8 ceil(n / C) + 4 ceil(n / 32) + 2 nnz.
 *
 * Deliberately naive: byte-by-byte little-endian access, one element at a time, no
 * vector code, no threads. Shares nothing with the GPU library. Nothing outside tests,
 * the smoke check and the benchmark's CPU legs may call it.
 */
#include <stddef.h>
#include <stdint.h>

#define ZVCO16_OK 0
#define ZVCO16_ERR_INVALID_ARG (-1)
#define ZVCO16_ERR_BUFFER_TOO_SMALL (-2)
#define ZVCO16_ERR_CORRUPT (-3)

#define ZVCO16_WINDOW 32u
#define ZVCO16_MAGIC 0x3143565Au
#define ZVCO16_HEADER_BYTES 32u
#define ZVCO16_WORD_BYTES 2u

static uint64_t div_up(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

static void wr8(uint8_t *p, uint64_t v, int bytes) {
  for (int k = 0; k < bytes; ++k) p[k] = (uint8_t)((v >> (8 * k)) & 0xffu);
}

static uint64_t rd8(const uint8_t *p, int bytes) {
  uint64_t v = 0;
  for (int k = 0; k < bytes; ++k) v |= (uint64_t)p[k] << (8 * k);
  return v;
}

static int chunk_ok(uint32_t c) { return c != 0 && c % ZVCO16_WINDOW == 0; }

/* Worst case of one stream: every word non-zero. 0 if chunk_elems is invalid. */
uint64_t zvco16_size_bound(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems)) return 0;
  return ZVCO16_HEADER_BYTES + 8 * div_up(n, chunk_elems) + 4 * div_up(n, ZVCO16_WINDOW) +
         ZVCO16_WORD_BYTES * n;
}

/*
 * Encode n 16-bit words into one stream; returns the stream's byte count or a negative
 * error. Per window (section V.A): test each of the 32 values against zero, set its mask
 * bit, write the mask, then the non-zero values in order.
 */
int64_t zvco16_encode(const uint16_t *x, uint64_t n, uint32_t chunk_elems, uint8_t *out,
                      uint64_t cap) {
  if (!chunk_ok(chunk_elems) || out == NULL || (n > 0 && x == NULL))
    return ZVCO16_ERR_INVALID_ARG;
  const uint64_t nc = div_up(n, chunk_elems);
  const uint64_t start = ZVCO16_HEADER_BYTES + 8 * nc;
  if (cap < start) return ZVCO16_ERR_BUFFER_TOO_SMALL;
  uint64_t at = 0; /* payload bytes written */
  for (uint64_t c = 0; c < nc; ++c) {
    wr8(out + ZVCO16_HEADER_BYTES + 8 * c, at, 8);
    const uint64_t lo = c * (uint64_t)chunk_elems;
    const uint64_t hi = (n - lo < chunk_elems) ? n : lo + chunk_elems;
    for (uint64_t w = lo; w < hi; w += ZVCO16_WINDOW) {
      uint32_t mask = 0;
      for (uint32_t i = 0; i < ZVCO16_WINDOW && w + i < hi; ++i)
        if (x[w + i] != 0) mask |= 1u << i;
      if (cap - start - at < 4) return ZVCO16_ERR_BUFFER_TOO_SMALL;
      wr8(out + start + at, mask, 4);
      at += 4;
      for (uint32_t i = 0; i < ZVCO16_WINDOW; ++i) {
        if (!((mask >> i) & 1u)) continue;
        if (cap - start - at < ZVCO16_WORD_BYTES) return ZVCO16_ERR_BUFFER_TOO_SMALL;
        wr8(out + start + at, x[w + i], ZVCO16_WORD_BYTES);
        at += ZVCO16_WORD_BYTES;
      }
    }
  }
  wr8(out + 0, ZVCO16_MAGIC, 4);
  wr8(out + 4, 1, 2);
  wr8(out + 6, ZVCO16_WORD_BYTES, 2);
  wr8(out + 8, ZVCO16_WINDOW, 4);
  wr8(out + 12, chunk_elems, 4);
  wr8(out + 16, n, 8);
  wr8(out + 24, at, 8);
  return (int64_t)(start + at);
}

/*
 * Decode one stream of in_bytes bytes into n 16-bit words: every set mask bit takes the
 * next packed 2-byte word, every clear bit becomes zero. Accepted only if every header
 * field matches (n, chunk_elems), in_bytes equals header + table + payload_bytes, chunk 0
 * starts at payload offset 0, every chunk's windows end exactly where the next chunk (or
 * the payload) begins, and no mask bit names an element at or beyond n. Returns 0 or a
 * negative error; on ZVCO16_ERR_CORRUPT the contents of y are unspecified.
 */
int zvco16_decode(const uint8_t *in, uint64_t in_bytes, uint16_t *y, uint64_t n,
                  uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || in == NULL || (n > 0 && y == NULL))
    return ZVCO16_ERR_INVALID_ARG;
  if (in_bytes < ZVCO16_HEADER_BYTES) return ZVCO16_ERR_CORRUPT;
  if (rd8(in, 4) != ZVCO16_MAGIC || rd8(in + 4, 2) != 1 || rd8(in + 6, 2) != ZVCO16_WORD_BYTES ||
      rd8(in + 8, 4) != ZVCO16_WINDOW || rd8(in + 12, 4) != chunk_elems || rd8(in + 16, 8) != n)
    return ZVCO16_ERR_CORRUPT;
  const uint64_t nc = div_up(n, chunk_elems);
  const uint64_t start = ZVCO16_HEADER_BYTES + 8 * nc;
  if (in_bytes < start) return ZVCO16_ERR_CORRUPT;
  const uint64_t payload = rd8(in + 24, 8);
  if (payload != in_bytes - start) return ZVCO16_ERR_CORRUPT;
  for (uint64_t c = 0; c < nc; ++c) {
    uint64_t at = rd8(in + ZVCO16_HEADER_BYTES + 8 * c, 8);
    const uint64_t stop = (c + 1 < nc) ? rd8(in + ZVCO16_HEADER_BYTES + 8 * (c + 1), 8) : payload;
    if ((c == 0 && at != 0) || at > stop || stop > payload) return ZVCO16_ERR_CORRUPT;
    const uint64_t lo = c * (uint64_t)chunk_elems;
    const uint64_t hi = (n - lo < chunk_elems) ? n : lo + chunk_elems;
    for (uint64_t w = lo; w < hi; w += ZVCO16_WINDOW) {
      if (stop - at < 4) return ZVCO16_ERR_CORRUPT;
      const uint32_t mask = (uint32_t)rd8(in + start + at, 4);
      at += 4;
      const uint64_t count = (hi - w < ZVCO16_WINDOW) ? hi - w : ZVCO16_WINDOW;
      if (count < ZVCO16_WINDOW && (mask >> count) != 0u) return ZVCO16_ERR_CORRUPT;
      for (uint32_t i = 0; i < count; ++i) {
        if ((mask >> i) & 1u) {
          if (stop - at < ZVCO16_WORD_BYTES) return ZVCO16_ERR_CORRUPT;
          y[w + i] = (uint16_t)rd8(in + start + at, ZVCO16_WORD_BYTES);
          at += ZVCO16_WORD_BYTES;
        } else {
          y[w + i] = 0;
        }
      }
    }
    if (at != stop) return ZVCO16_ERR_CORRUPT;
  }
  return ZVCO16_OK;
}
