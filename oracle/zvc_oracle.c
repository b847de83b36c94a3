/*
 * ZVC oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded scalar restatement of zero-value compression (ZVC)
 * as described in Rhu et al., "Compressing DMA Engine: Leveraging Activation Sparsity
 * for Training Deep Neural Networks" (arXiv:1705.01626), section V.A "Compression
 * Algorithm": every 32 consecutive activation words are described by one 32-bit
 * zero/non-zero mask, and the non-zero words follow the mask. A window of 32 zeros
 * therefore costs a single 4-byte mask (32x compression). Offsets of the packed words
 * are the prefix counts of the mask bits (same section; section V.B describes the
 * engine computing compressed offsets with prefix sums).
 *
 * The paper fixes only that core. The framing (stream header, chunk offset table,
 * batch table, bit and value order, zero test, tail handling) is this project's
 * reading, written out here field by field:
 *
 *   single stream, little-endian, no padding anywhere
 *     +0   u32 magic 0x3143565A ("ZVC1")
 *     +4   u16 version = 1
 *     +6   u16 word_bytes = 4
 *     +8   u32 window = 32
 *     +12  u32 chunk_elems C (a positive multiple of 32)
 *     +16  u64 n, the number of 32-bit words
 *     +24  u64 payload_bytes
 *     +32  u64 chunk_off[nc], nc = ceil(n / C), byte offset of chunk c inside the payload
 *     +32+8nc  payload: chunk 0 | chunk 1 | ...
 *   chunk c = for each window of the chunk, in order: u32 mask, then the words whose
 *     mask bit is set, in ascending element order. Bit i of a mask is element i of the
 *     window (least significant bit first). A word is zero iff all 32 bits are clear,
 *     so -0.0, NaNs and denormals are carried as non-zero words. In the last window of
 *     the stream, bits at or beyond n are clear.
 *
 *   batch of T streams
 *     +0   u32 magic 0x4243565A ("ZVCB")
 *     +4   u32 T
 *     +8   u64 total_bytes
 *     +16  u64 tensor_off[T + 1], absolute offsets; stream i spans
 *          [tensor_off[i], tensor_off[i + 1]) and tensor_off[T] = total_bytes
 *
 * This file is deliberately naive: byte-by-byte little-endian access, one element at a
 * time, no blocking, no vector code, no threads. Nothing outside tests, the smoke check
 * and the benchmark's CPU-baseline leg may call it.
 */
#include <stddef.h>
#include <stdint.h>

#define ZVCO_OK 0
#define ZVCO_ERR_INVALID_ARG (-1)
#define ZVCO_ERR_BUFFER_TOO_SMALL (-2)
#define ZVCO_ERR_CORRUPT (-3)

#define ZVCO_WINDOW 32u
#define ZVCO_STREAM_MAGIC 0x3143565Au
#define ZVCO_BATCH_MAGIC 0x4243565Au
#define ZVCO_STREAM_HEADER_BYTES 32u
#define ZVCO_BATCH_HEADER_BYTES 16u

static uint64_t ceil_div(uint64_t a, uint64_t b) { return a / b + (a % b != 0); }

static void put_u16(uint8_t *p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xffu);
  p[1] = (uint8_t)(v >> 8);
}

static void put_u32(uint8_t *p, uint32_t v) {
  for (int k = 0; k < 4; ++k) p[k] = (uint8_t)((v >> (8 * k)) & 0xffu);
}

static void put_u64(uint8_t *p, uint64_t v) {
  for (int k = 0; k < 8; ++k) p[k] = (uint8_t)((v >> (8 * k)) & 0xffu);
}

static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

static uint32_t get_u32(const uint8_t *p) {
  uint32_t v = 0;
  for (int k = 0; k < 4; ++k) v |= (uint32_t)p[k] << (8 * k);
  return v;
}

static uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int k = 0; k < 8; ++k) v |= (uint64_t)p[k] << (8 * k);
  return v;
}

static int chunk_elems_ok(uint32_t chunk_elems) {
  return chunk_elems != 0 && chunk_elems % ZVCO_WINDOW == 0;
}

/* Worst case of one stream: every word non-zero. */
uint64_t zvco_size_bound(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_elems_ok(chunk_elems)) return 0;
  return ZVCO_STREAM_HEADER_BYTES + 8 * ceil_div(n, chunk_elems) +
         4 * ceil_div(n, ZVCO_WINDOW) + 4 * n;
}

/*
 * Encode n words into one stream. Returns the stream's byte count, or a negative
 * ZVCO_ERR_* code. Follows section V.A: per window build the mask, append it, then
 * append the non-zero words (the "gather" whose positions are the mask's prefix counts).
 */
int64_t zvco_encode(const uint32_t *x, uint64_t n, uint32_t chunk_elems, uint8_t *out,
                    uint64_t cap) {
  if (!chunk_elems_ok(chunk_elems) || out == NULL || (n > 0 && x == NULL))
    return ZVCO_ERR_INVALID_ARG;
  const uint64_t nc = ceil_div(n, chunk_elems);
  const uint64_t payload_start = ZVCO_STREAM_HEADER_BYTES + 8 * nc;
  if (cap < payload_start) return ZVCO_ERR_BUFFER_TOO_SMALL;
  uint8_t *payload = out + payload_start;
  const uint64_t payload_cap = cap - payload_start;
  uint64_t cur = 0; /* bytes of payload written so far */

  for (uint64_t c = 0; c < nc; ++c) {
    put_u64(out + ZVCO_STREAM_HEADER_BYTES + 8 * c, cur);
    const uint64_t first = c * (uint64_t)chunk_elems;
    const uint64_t last = (n - first < chunk_elems) ? n : first + chunk_elems;
    for (uint64_t w0 = first; w0 < last; w0 += ZVCO_WINDOW) {
      uint32_t mask = 0;
      for (uint32_t i = 0; i < ZVCO_WINDOW; ++i) {
        if (w0 + i < last && x[w0 + i] != 0u) mask |= 1u << i;
      }
      if (payload_cap - cur < 4) return ZVCO_ERR_BUFFER_TOO_SMALL;
      put_u32(payload + cur, mask);
      cur += 4;
      for (uint32_t i = 0; i < ZVCO_WINDOW; ++i) {
        if ((mask >> i) & 1u) {
          if (payload_cap - cur < 4) return ZVCO_ERR_BUFFER_TOO_SMALL;
          put_u32(payload + cur, x[w0 + i]);
          cur += 4;
        }
      }
    }
  }

  put_u32(out + 0, ZVCO_STREAM_MAGIC);
  put_u16(out + 4, 1);
  put_u16(out + 6, 4);
  put_u32(out + 8, ZVCO_WINDOW);
  put_u32(out + 12, chunk_elems);
  put_u64(out + 16, n);
  put_u64(out + 24, cur);
  return (int64_t)(payload_start + cur);
}

/*
 * Decode one stream of in_bytes bytes into n words (the inverse of section V.A: every
 * set mask bit takes the next packed word, every clear bit becomes a zero word).
 * Returns ZVCO_OK or a negative ZVCO_ERR_* code; on ZVCO_ERR_CORRUPT the contents of
 * y are unspecified. A stream is accepted only if every field matches (n, chunk_elems),
 * in_bytes equals header + table + payload_bytes, chunk 0 starts at payload offset 0,
 * every chunk's windows end exactly where the next chunk (or the payload) begins, and
 * no mask bit names an element at or beyond n.
 */
int zvco_decode(const uint8_t *in, uint64_t in_bytes, uint32_t *y, uint64_t n,
                uint32_t chunk_elems) {
  if (!chunk_elems_ok(chunk_elems) || in == NULL || (n > 0 && y == NULL))
    return ZVCO_ERR_INVALID_ARG;
  if (in_bytes < ZVCO_STREAM_HEADER_BYTES) return ZVCO_ERR_CORRUPT;
  if (get_u32(in + 0) != ZVCO_STREAM_MAGIC) return ZVCO_ERR_CORRUPT;
  if (get_u16(in + 4) != 1 || get_u16(in + 6) != 4) return ZVCO_ERR_CORRUPT;
  if (get_u32(in + 8) != ZVCO_WINDOW || get_u32(in + 12) != chunk_elems) return ZVCO_ERR_CORRUPT;
  if (get_u64(in + 16) != n) return ZVCO_ERR_CORRUPT;

  const uint64_t nc = ceil_div(n, chunk_elems);
  const uint64_t payload_start = ZVCO_STREAM_HEADER_BYTES + 8 * nc;
  if (in_bytes < payload_start) return ZVCO_ERR_CORRUPT;
  const uint64_t payload_bytes = get_u64(in + 24);
  if (payload_bytes != in_bytes - payload_start) return ZVCO_ERR_CORRUPT;
  const uint8_t *payload = in + payload_start;

  for (uint64_t c = 0; c < nc; ++c) {
    const uint64_t start = get_u64(in + ZVCO_STREAM_HEADER_BYTES + 8 * c);
    const uint64_t end =
        (c + 1 < nc) ? get_u64(in + ZVCO_STREAM_HEADER_BYTES + 8 * (c + 1)) : payload_bytes;
    if (c == 0 && start != 0) return ZVCO_ERR_CORRUPT;
    if (start > end || end > payload_bytes) return ZVCO_ERR_CORRUPT;
    const uint64_t first = c * (uint64_t)chunk_elems;
    const uint64_t last = (n - first < chunk_elems) ? n : first + chunk_elems;
    uint64_t cur = start;
    for (uint64_t w0 = first; w0 < last; w0 += ZVCO_WINDOW) {
      if (end - cur < 4) return ZVCO_ERR_CORRUPT;
      const uint32_t mask = get_u32(payload + cur);
      cur += 4;
      const uint64_t valid = (last - w0 < ZVCO_WINDOW) ? last - w0 : ZVCO_WINDOW;
      if (valid < ZVCO_WINDOW && (mask >> valid) != 0u) return ZVCO_ERR_CORRUPT;
      for (uint32_t i = 0; i < valid; ++i) {
        if ((mask >> i) & 1u) {
          if (end - cur < 4) return ZVCO_ERR_CORRUPT;
          y[w0 + i] = get_u32(payload + cur);
          cur += 4;
        } else {
          y[w0 + i] = 0u;
        }
      }
    }
    if (cur != end) return ZVCO_ERR_CORRUPT;
  }
  return ZVCO_OK;
}

/* Bytes in front of the first stream of a batch of T streams. */
uint64_t zvco_batch_prefix_bytes(uint32_t T) {
  return ZVCO_BATCH_HEADER_BYTES + 8 * ((uint64_t)T + 1);
}

/* Encode T tensors into one batch: batch header, offset table, then T complete streams. */
int64_t zvco_encode_batch(uint32_t T, const uint32_t *const *xs, const uint64_t *ns,
                          uint32_t chunk_elems, uint8_t *out, uint64_t cap) {
  if (!chunk_elems_ok(chunk_elems) || out == NULL || (T > 0 && (xs == NULL || ns == NULL)))
    return ZVCO_ERR_INVALID_ARG;
  const uint64_t head = zvco_batch_prefix_bytes(T);
  if (cap < head) return ZVCO_ERR_BUFFER_TOO_SMALL;
  uint64_t pos = head;
  for (uint32_t i = 0; i < T; ++i) {
    put_u64(out + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)i, pos);
    const int64_t r = zvco_encode(xs[i], ns[i], chunk_elems, out + pos, cap - pos);
    if (r < 0) return r;
    pos += (uint64_t)r;
  }
  put_u64(out + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)T, pos);
  put_u32(out + 0, ZVCO_BATCH_MAGIC);
  put_u32(out + 4, T);
  put_u64(out + 8, pos);
  return (int64_t)pos;
}

/* Decode a batch produced by zvco_encode_batch into T output arrays. */
int zvco_decode_batch(const uint8_t *in, uint64_t in_bytes, uint32_t T, const uint64_t *ns,
                      uint32_t chunk_elems, uint32_t *const *ys) {
  if (!chunk_elems_ok(chunk_elems) || in == NULL || (T > 0 && (ns == NULL || ys == NULL)))
    return ZVCO_ERR_INVALID_ARG;
  const uint64_t head = zvco_batch_prefix_bytes(T);
  if (in_bytes < head) return ZVCO_ERR_CORRUPT;
  if (get_u32(in + 0) != ZVCO_BATCH_MAGIC || get_u32(in + 4) != T) return ZVCO_ERR_CORRUPT;
  if (get_u64(in + 8) != in_bytes) return ZVCO_ERR_CORRUPT;
  if (get_u64(in + ZVCO_BATCH_HEADER_BYTES) != head) return ZVCO_ERR_CORRUPT;
  if (get_u64(in + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)T) != in_bytes) return ZVCO_ERR_CORRUPT;
  for (uint32_t i = 0; i < T; ++i) {
    const uint64_t a = get_u64(in + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)i);
    const uint64_t b = get_u64(in + ZVCO_BATCH_HEADER_BYTES + 8 * ((uint64_t)i + 1));
    if (a > b || b > in_bytes) return ZVCO_ERR_CORRUPT;
    const int r = zvco_decode(in + a, b - a, ys[i], ns[i], chunk_elems);
    if (r != ZVCO_OK) return r;
  }
  return ZVCO_OK;
}
