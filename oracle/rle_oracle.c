/* RLE oracle: TEST INFRASTRUCTURE ONLY.
 *
 * Run-length encoding of activation maps, the layout-dependent comparison codec of Rhu et
 * al., "Compressing DMA Engine", section V.A (RLE exploits runs of zeros and of non-zeros,
 * so its ratio depends on how the values are laid out) and section VII.A (compression is
 * measured per 4 KB window, across activation layouts). The pages give no byte layout;
 * this file fixes one, written plainly, one element at a time:
 *
 * A word is zero iff its 32 bits are all clear. The n words are cut into windows of W
 * words (W a positive multiple of 32, at most 32768; the last window may be shorter).
 * Each window is encoded on its own as a sequence of records
 *     u16 zeros, u16 literals, then `literals` words copied bit for bit
 * where a record is the maximal run of zeros at the cursor followed by the maximal run of
 * non-zeros after it. So a new record starts at the window's first word and at every
 * zero that follows a non-zero; only a window's first record can have zeros == 0 and
 * only its last can have literals == 0.
 *
 * Stream (little-endian, no padding):
 *   offset 0   u32 magic 0x31454C52 ("RLE1")
 *   offset 4   u16 version 1
 *   offset 6   u16 word_bytes 4
 *   offset 8   u32 window W
 *   offset 12  u32 reserved, 0
 *   offset 16  u64 n
 *   offset 24  u64 payload_bytes
 *   offset 32  u64 window_off[ceil(n / W)]: byte offset of each window's first record,
 *              from the start of the payload (a multiple of 4: records are whole words)
 *   then the payload: the windows' records in order.
 * Size: 32 + 8 * nw + 4 * (records) + 4 * nnz, where a window has one record plus one per
 * zero that follows a non-zero inside it. At most 32 + 12 * nw + 4 * n.
 */
#include <stdint.h>
#include <string.h>

#define RLE_OK 0
#define RLE_ERR_INVALID_ARG -1
#define RLE_ERR_BUFFER_TOO_SMALL -2
#define RLE_ERR_CORRUPT -3

#define RLE_MAGIC 0x31454C52u

static uint64_t ceil_div(uint64_t a, uint64_t b) { return a / b + (a % b != 0); }

static void put_u16(uint8_t *p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFFu);
  p[1] = (uint8_t)(v >> 8);
}
static void put_u32(uint8_t *p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)((v >> (8 * i)) & 0xFFu);
}
static void put_u64(uint8_t *p, uint64_t v) {
  for (int i = 0; i < 8; ++i) p[i] = (uint8_t)((v >> (8 * i)) & 0xFFu);
}
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 3; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint64_t get_u64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

static int window_ok(uint32_t w) { return w >= 32 && w % 32 == 0 && w <= 32768; }

uint64_t rleo_size_bound(uint64_t n, uint32_t window) {
  if (!window_ok(window)) return 0;
  const uint64_t nw = ceil_div(n, window);
  return 32 + 12 * nw + 4 * n;
}

/* Encodes x[0..n) into out (capacity cap). Returns the stream size or a negative code. */
int64_t rleo_encode(const uint32_t *x, uint64_t n, uint32_t window, uint8_t *out, uint64_t cap) {
  if (!window_ok(window) || (n > 0 && x == 0) || out == 0) return RLE_ERR_INVALID_ARG;
  if (cap < rleo_size_bound(n, window)) return RLE_ERR_BUFFER_TOO_SMALL;
  const uint64_t nw = ceil_div(n, window);
  const uint64_t payload_at = 32 + 8 * nw;
  uint64_t pos = payload_at;  /* absolute write position */
  for (uint64_t w = 0; w < nw; ++w) {
    put_u64(out + 32 + 8 * w, pos - payload_at);
    const uint64_t begin = w * window;
    const uint64_t end = begin + window < n ? begin + window : n;
    uint64_t i = begin;
    while (i < end) {  /* one record per iteration */
      uint64_t zeros = 0, literals = 0;
      while (i < end && x[i] == 0) {
        ++zeros;
        ++i;
      }
      const uint64_t head = pos;
      pos += 4;
      while (i < end && x[i] != 0) {
        put_u32(out + pos, x[i]);
        pos += 4;
        ++literals;
        ++i;
      }
      put_u16(out + head, (uint16_t)zeros);
      put_u16(out + head + 2, (uint16_t)literals);
    }
  }
  put_u32(out + 0, RLE_MAGIC);
  put_u16(out + 4, 1);
  put_u16(out + 6, 4);
  put_u32(out + 8, window);
  put_u32(out + 12, 0);
  put_u64(out + 16, n);
  put_u64(out + 24, pos - payload_at);
  return (int64_t)pos;
}

/* Decodes a stream of exactly in_bytes bytes into y[0..n). Every field is checked; a
 * malformed stream returns RLE_ERR_CORRUPT (y is then unspecified). */
int rleo_decode(const uint8_t *in, uint64_t in_bytes, uint32_t *y, uint64_t n, uint32_t window) {
  if (!window_ok(window) || in == 0 || (n > 0 && y == 0)) return RLE_ERR_INVALID_ARG;
  if (in_bytes < 32) return RLE_ERR_CORRUPT;
  if (get_u32(in) != RLE_MAGIC || get_u16(in + 4) != 1 || get_u16(in + 6) != 4 ||
      get_u32(in + 8) != window || get_u32(in + 12) != 0 || get_u64(in + 16) != n)
    return RLE_ERR_CORRUPT;
  const uint64_t nw = ceil_div(n, window);
  const uint64_t payload_at = 32 + 8 * nw;
  const uint64_t payload = get_u64(in + 24);
  if (in_bytes < payload_at || in_bytes - payload_at != payload) return RLE_ERR_CORRUPT;
  for (uint64_t w = 0; w < nw; ++w) {
    const uint64_t off = get_u64(in + 32 + 8 * w);
    const uint64_t next = w + 1 < nw ? get_u64(in + 32 + 8 * (w + 1)) : payload;
    if ((w == 0 && off != 0) || off > next || next > payload || (off | next) % 4 != 0)
      return RLE_ERR_CORRUPT;
    const uint64_t begin = w * window;
    const uint64_t end = begin + window < n ? begin + window : n;
    uint64_t i = begin, pos = payload_at + off;
    const uint64_t stop = payload_at + next;
    while (i < end) {
      if (pos + 4 > stop) return RLE_ERR_CORRUPT;
      const uint64_t zeros = get_u16(in + pos), literals = get_u16(in + pos + 2);
      pos += 4;
      if (zeros + literals == 0 || zeros + literals > end - i) return RLE_ERR_CORRUPT;
      for (uint64_t k = 0; k < zeros; ++k) y[i++] = 0;
      if (pos + 4 * literals > stop) return RLE_ERR_CORRUPT;
      for (uint64_t k = 0; k < literals; ++k) {
        y[i++] = get_u32(in + pos);
        pos += 4;
      }
    }
    if (pos != stop) return RLE_ERR_CORRUPT;
  }
  return RLE_OK;
}
