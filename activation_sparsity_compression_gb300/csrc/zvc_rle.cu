// Run-length encoding on sm_103a: the layout-dependent comparison codec of Rhu et al.,
// "Compressing DMA Engine", section V.A (RLE exploits runs of zeros and of non-zeros) and
// section VII.A (compression per 4 KB window, across activation layouts). Stream layout
// (documented in include/zvc.h): per window of W words, records of a u16 zero-run length,
// a u16 literal count and the literal words, where a record is the maximal zero run at
// the cursor followed by the maximal non-zero run after it; a 32-byte header and a u64
// window offset table make windows independently decodable.
//
// Compress (two passes over the input; this is a comparison codec, not the hot path):
//   sizes   one warp per window: a ballot per 32 words gives the non-zero mask; records =
//           1 + the zeros that follow a non-zero inside the window; size = 4 (records +
//           non-zeros)
//   scan    exclusive prefix of the window sizes (block scans, a scan of the block
//           totals, then the add), written as the window offset table; the last window
//           writes the header and the total size
//   encode  one warp per window: a non-zero word at window position i goes to word
//           (records started at or before i) + (non-zeros before i) of the window's
//           records; each record start is noted in shared memory, and a second phase
//           writes every record's header from its start and the next one's
// Decompress: one warp per window checks the header and its table entries, stages the
// window's records in shared memory and zero-fills the window's output with coalesced
// stores; then, kRleBatch records at a time, one lane walks the headers (each record's place
// depends on every earlier one) and the lanes copy the walked records' literals.
#include "zvc_internal.cuh"

namespace zvc {
namespace {

constexpr uint32_t kRleMagic = 0x31454C52u;  // "RLE1"
constexpr uint32_t kRleWarps = 8;           // windows per CTA in sizes
constexpr uint32_t kRleMaxWarps = 32;       // windows per CTA in encode / decode, at most
constexpr uint64_t kSmemBudget = 200 * 1024;  // encode / decode: shared memory per CTA
constexpr uint32_t kRleBatch = 128;         // records walked before their literals are copied
constexpr uint32_t kScanThreads = 1024;

__device__ __forceinline__ uint32_t lanemask_le(uint32_t lane) {
  return lane == 31 ? 0xffffffffu : ((2u << lane) - 1u);
}

// ------------------------------------------------------------------ compress
__global__ void __launch_bounds__(32 * kRleWarps)
    rle_sizes_kernel(const uint32_t* in, uint64_t n, uint32_t W, uint64_t nwin, uint32_t* sizes) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t w = (uint64_t)blockIdx.x * kRleWarps + (threadIdx.x >> 5);
  if (w >= nwin) return;
  const uint64_t begin = w * W;
  const uint32_t len = (uint32_t)min((uint64_t)W, n - begin);
  uint32_t recs = 1, nnz = 0, carry = 0;
  for (uint32_t g = 0; g * 32 < len; ++g) {
    const uint32_t e = g * 32 + lane;
    const bool valid = e < len;
    const uint32_t v = valid ? __ldcs(in + begin + e) : 0u;
    const uint32_t m = __ballot_sync(0xffffffffu, valid && v != 0u);
    const uint32_t vm = __ballot_sync(0xffffffffu, valid);
    const uint32_t t = ~m & vm & ((m << 1) | carry);  // zeros that follow a non-zero
    recs += __popc(t);
    nnz += __popc(m);
    carry = m >> 31;
  }
  if (lane == 0) sizes[w] = 4u * (recs + nnz);
}

// Block-local exclusive scan of the sizes into the table (bytes), block totals aside.
__global__ void __launch_bounds__(kScanThreads)
    rle_scan_blocks(const uint32_t* sizes, uint64_t nwin, uint64_t* table, uint64_t* block_sum) {
  __shared__ uint64_t warp_tot[32];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint64_t w = (uint64_t)blockIdx.x * kScanThreads + threadIdx.x;
  const uint64_t v = w < nwin ? sizes[w] : 0;
  uint64_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= (uint32_t)d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint64_t t = warp_tot[lane], ti = t;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, ti, d);
      if (lane >= (uint32_t)d) ti += y;
    }
    warp_tot[lane] = ti - t;  // exclusive
    if (lane == 31) block_sum[blockIdx.x] = ti;
  }
  __syncthreads();
  if (w < nwin) table[w] = warp_tot[warp] + incl - v;
}

// Exclusive scan of the block totals (one CTA, in steps of kScanThreads).
__global__ void __launch_bounds__(kScanThreads) rle_scan_top(uint64_t* block_sum, uint64_t nblk) {
  __shared__ uint64_t warp_tot[32];
  __shared__ uint64_t carry;
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (uint64_t b0 = 0; b0 < nblk; b0 += kScanThreads) {
    const uint64_t b = b0 + threadIdx.x;
    const uint64_t v = b < nblk ? block_sum[b] : 0;
    uint64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= (uint32_t)d) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      uint64_t t = warp_tot[lane], ti = t;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, ti, d);
        if (lane >= (uint32_t)d) ti += y;
      }
      warp_tot[lane] = ti - t;
    }
    __syncthreads();
    const uint64_t base = carry;
    if (b < nblk) block_sum[b] = base + warp_tot[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) carry = base + warp_tot[warp] + incl;
    __syncthreads();
  }
}

// Adds the block prefixes; the last window (or the only thread, for n = 0) writes the
// header and the total size.
__global__ void __launch_bounds__(kScanThreads)
    rle_scan_add(const uint32_t* sizes, uint64_t n, uint32_t W, uint64_t nwin, uint64_t* table,
                 const uint64_t* block_sum, uint32_t* out, uint64_t* out_size) {
  const uint64_t w = (uint64_t)blockIdx.x * kScanThreads + threadIdx.x;
  uint64_t payload = 0;
  bool last = false;
  if (nwin == 0) {
    last = w == 0;
  } else if (w < nwin) {
    const uint64_t off = table[w] + block_sum[blockIdx.x];
    table[w] = off;
    if (w + 1 == nwin) {
      last = true;
      payload = off + sizes[w];
    }
  }
  if (!last) return;
  out[0] = kRleMagic;
  out[1] = kVersionWordBytes;
  out[2] = W;
  out[3] = 0;
  out[4] = (uint32_t)n;
  out[5] = (uint32_t)(n >> 32);
  out[6] = (uint32_t)payload;
  out[7] = (uint32_t)(payload >> 32);
  if (out_size) *out_size = 32 + 8 * nwin + payload;
}

struct RecStart {
  uint32_t pos;  // window position of the record's first word
  uint32_t nz;   // non-zeros of the window before it
};

__global__ void __launch_bounds__(32 * kRleMaxWarps)
    rle_encode_kernel(const uint32_t* in, uint64_t n, uint32_t W, uint64_t nwin, uint32_t* out,
                      uint32_t recs_per_warp) {
  extern __shared__ __align__(16) RecStart rs_all[];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint64_t w = (uint64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  if (w >= nwin) return;
  RecStart* rs = rs_all + (uint64_t)warp * recs_per_warp;
  const uint64_t* table = reinterpret_cast<const uint64_t*>(out + kStreamHeaderWords);
  uint32_t* o = out + kStreamHeaderWords + 2 * nwin + table[w] / 4;  // the window's records
  const uint64_t begin = w * W;
  const uint32_t len = (uint32_t)min((uint64_t)W, n - begin);
  const uint32_t le = lanemask_le(lane), lt = le >> 1;
  uint32_t R = 0, N = 0, carry = 0;
  for (uint32_t g = 0; g * 32 < len; ++g) {
    const uint32_t e = g * 32 + lane;
    const bool valid = e < len;
    const uint32_t v = valid ? __ldcs(in + begin + e) : 0u;
    const uint32_t m = __ballot_sync(0xffffffffu, valid && v != 0u);
    const uint32_t vm = __ballot_sync(0xffffffffu, valid);
    uint32_t t = ~m & vm & ((m << 1) | carry);  // record starts: zeros after a non-zero
    if (g == 0) t |= 1u;                       // and the window's first word
    const uint32_t rl = R + __popc(t & le);    // records started at or before this word
    const uint32_t nl = N + __popc(m & lt);    // non-zeros before it
    if (valid && v != 0u) o[rl + nl] = v;      // literal: after rl headers and nl literals
    if ((t >> lane) & 1u) rs[rl - 1] = RecStart{e, nl};
    R += __popc(t);
    N += __popc(m);
    carry = m >> 31;
  }
  __syncwarp();
  for (uint32_t r = lane; r < R; r += 32) {
    const RecStart a = rs[r];
    const RecStart b = r + 1 < R ? rs[r + 1] : RecStart{len, N};
    const uint32_t lit = b.nz - a.nz, zeros = (b.pos - a.pos) - lit;
    o[r + a.nz] = zeros | (lit << 16);
  }
}

// ------------------------------------------------------------------ decompress
// A walked record: x = window position of its first literal, y = literal count | staged
// word index of its first literal << 16 (both below 2^16: W <= 4096).
__global__ void __launch_bounds__(32 * kRleMaxWarps)
    rle_decode_kernel(const uint32_t* in, uint64_t in_bytes, uint64_t n, uint32_t W,
                      uint64_t nwin, uint32_t* y, uint8_t* ws, uint32_t stage_words) {
  extern __shared__ __align__(16) uint32_t dsm[];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint64_t w = (uint64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  Control* ctl = reinterpret_cast<Control*>(ws);
  if (w >= nwin) {
    if (nwin == 0 && w == 0 && lane == 0) {  // n = 0: the stream is the header alone
      const bool ok = in_bytes == 32 && in[0] == kRleMagic && in[1] == kVersionWordBytes &&
                      in[2] == W && in[3] == 0u && in[4] == 0u && in[5] == 0u && in[6] == 0u &&
                      in[7] == 0u;
      if (!ok) latch_error(ctl, ZVC_ERR_CORRUPT, 0);
    }
    return;
  }
  uint32_t* buf = dsm + (uint64_t)warp * (stage_words + 2 * kRleBatch);
  uint2* runs = reinterpret_cast<uint2*>(buf + stage_words);
  // header and this window's table entries (all lanes, same values; all in bounds once
  // in_bytes covers the header and table, which is checked first)
  const uint64_t table_end = 32 + 8 * nwin;
  bool ok = in_bytes >= table_end;
  uint64_t payload = 0, off = 0, next = 0;
  if (ok) {
    const uint64_t pl = (uint64_t)in[6] | ((uint64_t)in[7] << 32);
    const uint64_t nn = (uint64_t)in[4] | ((uint64_t)in[5] << 32);
    const uint64_t* table = reinterpret_cast<const uint64_t*>(in + kStreamHeaderWords);
    off = table[w];
    next = w + 1 < nwin ? table[w + 1] : pl;
    payload = pl;
    ok = (in[0] == kRleMagic) & (in[1] == kVersionWordBytes) & (in[2] == W) & (in[3] == 0u) &
         (nn == n) & (in_bytes - table_end == pl);
  }
  const uint64_t begin = w * W;
  const uint32_t len = (uint32_t)min((uint64_t)W, n - begin);
  ok = ok && (w != 0 || off == 0) && off <= next && next <= payload && ((off | next) & 3u) == 0 &&
       next - off >= 4 && next - off <= 4 + 4ull * len;
  if (!ok) {
    if (lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, w);
    return;
  }
  // stage the window's records and zero-fill its output
  const uint32_t cnt = (uint32_t)((next - off) / 4);
  const uint32_t* src = in + table_end / 4 + off / 4;
  for (uint32_t k = lane; k < cnt; k += 32) buf[k] = __ldcs(src + k);
  uint32_t* dst = y + begin;
  for (uint32_t k = lane; k < len; k += 32) dst[k] = 0u;
  __syncwarp();
  // walk the headers (lane 0) kRleBatch records at a time, copying each batch's literals;
  // every record covers at least one word, so the walk ends within len records
  uint32_t p = 0, pos = 0, good = 1;
  while (true) {
    uint32_t nb = 0;
    if (lane == 0) {
      while (nb < kRleBatch && pos < len) {
        if (p >= cnt) { good = 0; break; }
        const uint32_t h = buf[p];
        const uint32_t z = h & 0xFFFFu, l = h >> 16;
        if (z + l == 0 || z + l > len - pos || p + 1 + l > cnt) { good = 0; break; }
        runs[nb++] = make_uint2(pos + z, l | ((p + 1) << 16));
        pos += z + l;
        p += 1 + l;
      }
    }
    nb = __shfl_sync(0xffffffffu, nb, 0);
    good = __shfl_sync(0xffffffffu, good, 0);
    pos = __shfl_sync(0xffffffffu, pos, 0);
    __syncwarp();
    if (!good) break;
    for (uint32_t r = lane; r < nb; r += 32) {
      const uint2 a = runs[r];
      const uint32_t lits = a.y & 0xFFFFu, s0 = a.y >> 16;
      for (uint32_t k = 0; k < lits; ++k) dst[a.x + k] = buf[s0 + k];
    }
    __syncwarp();  // the batch's records are read before the next batch overwrites them
    if (pos >= len) break;
  }
  if (lane == 0 && good && p != cnt) good = 0;
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good && lane == 0) latch_error(ctl, ZVC_ERR_CORRUPT, w);
}

bool window_ok(uint32_t W) { return W >= 32 && W % 32 == 0 && W <= ZVC_RLE_MAX_WINDOW; }

}  // namespace

// Workspace: Control + reserved, then u32 sizes[nwin], then u64 block sums.
uint64_t rle_ws_bytes(uint64_t n, uint32_t W) {
  const uint64_t nwin = ceil_div_u64(n, W);
  const uint64_t nblk = ceil_div_u64(nwin, kScanThreads);
  return round_up_u64(kStatusOffset + round_up_u64(4 * nwin, 8) + 8 * nblk + 8,
                      ZVC_WORKSPACE_ALIGN);
}

zvc_status launch_rle_compress(const uint32_t* in, uint64_t n, uint32_t W, uint32_t* out,
                               uint64_t* out_size, uint8_t* ws, cudaStream_t stream) {
  if (!window_ok(W)) return ZVC_ERR_INVALID_ARG;
  const uint64_t nwin = ceil_div_u64(n, W);
  const uint64_t nblk = ceil_div_u64(nwin, kScanThreads);
  uint32_t* sizes = reinterpret_cast<uint32_t*>(ws + kStatusOffset);
  uint64_t* block_sum = reinterpret_cast<uint64_t*>(ws + kStatusOffset + round_up_u64(4 * nwin, 8));
  uint64_t* table = reinterpret_cast<uint64_t*>(out + kStreamHeaderWords);
  if (nwin > 0) {
    rle_sizes_kernel<<<(unsigned)ceil_div_u64(nwin, kRleWarps), 32 * kRleWarps, 0, stream>>>(
        in, n, W, nwin, sizes);
    rle_scan_blocks<<<(unsigned)nblk, kScanThreads, 0, stream>>>(sizes, nwin, table, block_sum);
    rle_scan_top<<<1, kScanThreads, 0, stream>>>(block_sum, nblk);
  }
  rle_scan_add<<<(unsigned)(nblk > 0 ? nblk : 1), kScanThreads, 0, stream>>>(
      sizes, n, W, nwin, table, block_sum, out, out_size);
  if (nwin > 0) {
    const uint32_t recs = W;  // a record covers at least one word
    const uint64_t per_warp = (uint64_t)recs * sizeof(RecStart);
    uint64_t warps = kSmemBudget / per_warp;
    warps = warps < 1 ? 1 : (warps > kRleMaxWarps ? kRleMaxWarps : warps);
    const uint64_t smem = warps * per_warp;
    cudaError_t e = cudaFuncSetAttribute(rle_encode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_failure(e);
    rle_encode_kernel<<<(unsigned)ceil_div_u64(nwin, warps), (unsigned)(32 * warps), smem,
                        stream>>>(in, n, W, nwin, out, recs);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

zvc_status launch_rle_decompress(const uint32_t* in, uint64_t in_bytes, uint32_t* y, uint64_t n,
                                 uint32_t W, uint8_t* ws, cudaStream_t stream) {
  if (!window_ok(W)) return ZVC_ERR_INVALID_ARG;
  const uint64_t nwin = ceil_div_u64(n, W);
  const uint32_t stage_words = (uint32_t)round_up_u64(W + 1, 4);
  const uint64_t per_warp = 4ull * (stage_words + 2ull * kRleBatch);
  uint64_t warps = kSmemBudget / per_warp;
  warps = warps < 1 ? 1 : (warps > kRleMaxWarps ? kRleMaxWarps : warps);
  const uint64_t smem = warps * per_warp;
  cudaError_t e = cudaFuncSetAttribute(rle_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_failure(e);
  const uint64_t blocks = nwin == 0 ? 1 : ceil_div_u64(nwin, warps);
  rle_decode_kernel<<<(unsigned)blocks, (unsigned)(32 * warps), smem, stream>>>(
      in, in_bytes, n, W, nwin, y, ws, stage_words);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_failure(e);
  return ZVC_OK;
}

}  // namespace zvc
