/*
 * zvc.h: C ABI of the GB300 (sm_103a) zero-value-compression (ZVC) library.
 *
 * What it computes. Rhu et al., "Compressing DMA Engine: Leveraging Activation Sparsity
 * for Training Deep Neural Networks" (arXiv:1705.01626), section V.A "Compression
 * Algorithm": every 32 consecutive 32-bit activation words are replaced by a 32-bit
 * zero/non-zero mask followed by the non-zero words, so an all-zero window costs one
 * 4-byte mask (32x). Section V.B: compressed offsets come from prefix sums of the masks'
 * population counts. Section V.D ("Software Interface"): a compressed copy call that
 * reports the compressed size, and offload/prefetch of activation maps with
 * cudaMemcpyAsync. Section IX: activations stay uncompressed in GPU memory; only the
 * copies to and from host memory carry compressed data.
 *
 * Stream format (little-endian, no padding; the framing is this library's reading, the
 * paper only fixes the mask-then-words core):
 *
 *   +0   u32 magic 0x3143565A ("ZVC1")     +4  u16 version 1     +6  u16 word_bytes 4
 *   +8   u32 window 32                     +12 u32 chunk_elems C (positive multiple of 32)
 *   +16  u64 n (words)                     +24 u64 payload_bytes
 *   +32  u64 chunk_off[ceil(n/C)]: byte offset of each chunk inside the payload
 *   then the payload: for every window in order, u32 mask (bit i = element i of the
 *   window, least significant bit first) followed by the words whose bit is set, in
 *   ascending element order. A word is "zero" iff all 32 bits are clear: -0.0, NaN and
 *   denormals are kept bit for bit. Mask bits at or beyond n are clear. Chunks are
 *   independently decodable through chunk_off.
 *   Compressed size S = 32 + 8*ceil(n/C) + 4*ceil(n/32) + 4*nnz.
 *
 * Batch format (zvc_*_batched, zvc_offload): u32 magic 0x4243565A ("ZVCB"), u32 T,
 *   u64 total_bytes, u64 tensor_off[T+1] (absolute; tensor_off[T] = total_bytes), then T
 *   complete streams, stream i at tensor_off[i].
 *
 * Conventions for every call below.
 *   - Elements are any 4-byte type, treated as opaque 32-bit words.
 *   - Pointers named d_* are device pointers, h_* host pointers. All buffers are owned
 *     by the caller; the library allocates nothing. d_* word buffers must be 4-byte
 *     aligned; 16-byte alignment takes the vectorised path.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Device work is
 *     enqueued on it and the call returns without waiting, except where stated.
 *   - The workspace d_ws is device memory of at least the size the matching
 *     *_workspace_size() returns, 256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE
 *     (e.g. cudaMemset), and not shared by calls that may run concurrently.
 *   - Errors found by the host are returned at once. Errors found on the device
 *     (corrupt input, a look-back wait that timed out) are latched in the workspace and
 *     reported by zvc_get_error(). The library never traps or aborts a kernel.
 *   - chunk_elems must be a positive multiple of 32 and at most ZVC_MAX_CHUNK_ELEMS.
 *   - The compress and decompress calls (single, batched, 16-bit, static) may be captured
 *     in a CUDA graph and replayed. A compress launch tags its workspace entries with an
 *     epoch of its own; on a capturing stream it takes that epoch from a counter in the
 *     workspace, on the device, so every replay gets a new one. Make one call of each
 *     kind before capturing (it loads the kernels and sizes their launches). A replayed
 *     decompress keeps the in_bytes of its capture. zvc_offload, zvc_prefetch and
 *     zvc_get_error read or wait on the host and are not for capture.
 */
#ifndef ZVC_H_
#define ZVC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int zvc_status;

#define ZVC_OK 0
#define ZVC_ERR_INVALID_ARG 1      /* bad pointer, size, alignment or parameter */
#define ZVC_ERR_BUFFER_TOO_SMALL 2 /* output or workspace smaller than required */
#define ZVC_ERR_CORRUPT 3          /* compressed input is not a valid stream for (n, C) */
#define ZVC_ERR_TIMEOUT 4          /* a device-side wait gave up (reported via zvc_get_error) */
#define ZVC_ERR_CUDA 5             /* a CUDA runtime call failed; see zvc_last_cuda_error() */

#define ZVC_WINDOW 32u
#define ZVC_DEFAULT_CHUNK_ELEMS 4096u
#define ZVC_MAX_CHUNK_ELEMS 32768u
#define ZVC_MAX_BATCH 512u          /* tensors per batched call */
#define ZVC_WORKSPACE_ALIGN 256u

/* Worst-case (all words non-zero) size in bytes of one stream of n words:
 * 32 + 8*ceil(n/C) + 4*ceil(n/32) + 4*n. Cites section V.A "Compression Algorithm": a
 * window costs its 4-byte mask plus 4 bytes per non-zero word, so a dense window grows
 * by one word. Returns 0 if chunk_elems is invalid. */
uint64_t zvc_size_bound(uint64_t n, uint32_t chunk_elems);

/* Worst-case size of a batch of T streams: 16 + 8*(T+1) + sum of zvc_size_bound.
 * Cites section V.A "Compression Algorithm" per stream; the batch framing (one stream
 * per tensor behind a table of stream offsets) is this library's reading, the paper has
 * no counterpart for it. ns is a host array of T word counts. Returns 0 on invalid
 * arguments. */
uint64_t zvc_batch_size_bound(const uint64_t* ns, uint32_t T, uint32_t chunk_elems);

/* Workspace bytes for zvc_compress / zvc_decompress of n words: the latched error word,
 * then one look-back status word per 4096-word tile. Cites section V.B "Compressing DMA
 * Engine Architecture": the compressed offsets are prefix sums of the masks' population
 * counts; across tiles that prefix sum is carried by these status words. Each compress
 * launch tags the status words it writes with a number of its own, so a workspace needs
 * no clearing between calls; only its error word must start at zero (see the conventions
 * above). */
uint64_t zvc_workspace_size(uint64_t n, uint32_t chunk_elems);

/* Workspace bytes for the batched calls over the T tensors in ns (host array): as
 * zvc_workspace_size (section V.B, prefix sums across tiles) for every tile of every
 * tensor, plus one start word per tensor for the batch framing. */
uint64_t zvc_batch_workspace_size(const uint64_t* ns, uint32_t T, uint32_t chunk_elems);

/* Compress n words at d_in into one stream at d_out (section V.A; the size report of the
 * section V.D compressed-copy call). out_cap must be at least zvc_size_bound(n, C). The
 * stream's byte count is written to the device u64 *d_out_size (if not NULL) when the
 * work completes. Output is byte-identical to the format above. */
zvc_status zvc_compress(const void* d_in, uint64_t n, uint32_t chunk_elems, void* d_out,
                        uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                        void* stream);

/* Compress without a workspace, for callers that cannot allocate device memory: code
 * running under a memory manager that owns all device memory (a framework pool, a fixed
 * memory plan) or code that must not call cudaMalloc, which synchronises the device and
 * fails once memory is fully reserved. The paper has no counterpart; this is a library
 * convenience. Same inputs, output and stream as zvc_compress, minus d_ws/ws_bytes: the
 * scratch is one static device array of about 1 MiB that every GPU loading the library
 * keeps until exit. Limits: n <= ZVC_STATIC_MAX_ELEMS, else ZVC_ERR_INVALID_ARG. Every
 * call looks up the array's device address on the current device (cudaGetSymbolAddress);
 * the first call on a device also loads the library's device code there, so make it
 * before any stream capture. The call allocates nothing. All calls on a device share the
 * array, and nothing in it is cleared between calls (each launch tags its entries with a
 * number of its own; only the error latch below carries over), so
 * calls whose GPU work overlaps (unordered streams) race and must be ordered by the
 * caller. A failure on the device (a wait that gave up) is latched in the array, where
 * it stays until zvc_compress_static_get_error() reads it; the stream's bytes and
 * *d_out_size are then unspecified. */
#define ZVC_STATIC_MAX_ELEMS (1ull << 29) /* 2 GiB of 4-byte words */
zvc_status zvc_compress_static(const void* d_in, uint64_t n, uint32_t chunk_elems, void* d_out,
                               uint64_t out_cap, uint64_t* d_out_size, void* stream);

/* The status latched by zvc_compress_static calls on the current device since the last
 * read (ZVC_OK if none): synchronises `stream`, reads the latch and clears it. The paper
 * has no counterpart, as for zvc_compress_static. */
zvc_status zvc_compress_static_get_error(void* stream);

/* Decompress the stream of in_bytes bytes at d_in into n words at d_out (inverse of
 * section V.A: a set mask bit takes the next packed word, a clear bit writes zero).
 * A stream that is not a valid encoding of n words with chunk_elems C latches
 * ZVC_ERR_CORRUPT; d_out's contents are then unspecified, and no access leaves
 * [d_in, d_in + in_bytes) or [d_out, d_out + 4n). */
zvc_status zvc_decompress(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                          uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream);

/* Compress T tensors in one launch into one batch at d_out: section V.A "Compression
 * Algorithm" applied to every tensor, with one prefix sum (section V.B) over the tiles of
 * all of them; section V.D "Software Interface" offloads every layer's activation maps,
 * and this call serves many small maps with one launch. The per-tensor offset table is
 * this library's framing. d_ins (device pointers) and ns are HOST arrays of T entries;
 * T <= ZVC_MAX_BATCH. out_cap >= zvc_batch_size_bound. The batch's total byte count goes
 * to *d_out_size (device, may be NULL). */
zvc_status zvc_compress_batched(const void* const* d_ins, const uint64_t* ns, uint32_t T,
                                uint32_t chunk_elems, void* d_out, uint64_t out_cap,
                                uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                                void* stream);

/* Decompress a batch of in_bytes bytes into T tensors (the inverse of section V.A for
 * every stream of the batch, found through its per-tensor offset table). d_outs (device
 * pointers) and ns are HOST arrays of T entries. Corruption is latched as for
 * zvc_decompress. */
zvc_status zvc_decompress_batched(const void* d_in, uint64_t in_bytes, void* const* d_outs,
                                  const uint64_t* ns, uint32_t T, uint32_t chunk_elems,
                                  void* d_ws, uint64_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------
 * ZVC on 16-bit words (bf16 / fp16). Section V.A "Compression Algorithm" gives the rule
 * for the 32-bit activations the paper evaluates; these calls apply it unchanged to 2-byte
 * words, a reading beyond the pages: 32 values per window, one 32-bit mask, then the
 * non-zero 2-byte values in ascending element order. The stream is the format above with
 * word_bytes = 2: windows follow each other without padding, so a mask may start on a
 * 2-byte boundary, and chunk offsets are even byte counts. A word is zero iff its 16 bits
 * are clear (-0.0 = 0x8000 is kept). Size: 32 + 8*ceil(n/C) + 4*ceil(n/32) + 2*nnz.
 * Single streams only (no batch, no offload). The workspace is zvc_workspace_size(n, C). */

/* Worst case of one 16-bit stream (every word non-zero), as in section V.A: 32 + 8*ceil(n/C)
 * + 4*ceil(n/32) + 2*n. Returns 0 if chunk_elems is invalid. */
uint64_t zvc_size_bound16(uint64_t n, uint32_t chunk_elems);

/* Compress n 16-bit words at d_in (2-byte aligned) into one stream at d_out (4-byte aligned;
 * out_cap >= zvc_size_bound16(n, C)); the byte count goes to the device u64 *d_out_size
 * (may be NULL). Section V.A on 2-byte words, as above. Errors as for zvc_compress. */
zvc_status zvc_compress16(const void* d_in, uint64_t n, uint32_t chunk_elems, void* d_out,
                          uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                          void* stream);

/* Decompress a 16-bit stream of in_bytes bytes at d_in (4-byte aligned) into n words at
 * d_out (2-byte aligned): the inverse of section V.A on 2-byte words. A stream that is not
 * a valid 16-bit encoding of n words with chunk_elems C latches ZVC_ERR_CORRUPT, with no
 * access outside [d_in, d_in + in_bytes) or [d_out, d_out + 2n). */
zvc_status zvc_decompress16(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                            uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream);

/* Segment length (words) that zvc_offload uses for a tensor of n words: n cut into
 * ceil(n / 2^25) equal parts, rounded up to whole chunks (at most about 32 Mi words,
 * 128 MiB of fp32). Cites section V.D "Software Interface": compression throughput must
 * match the transfer path, so the copy of one segment overlaps the compression of the
 * next; the segment length itself is this library's choice. */
uint64_t zvc_offload_segment_elems(uint64_t n, uint32_t chunk_elems);

/* Host bytes zvc_offload may need: the batch bound over its segments. Cites section V.D
 * "Software Interface": vDNN sizes its host allocations from the compressed size; this is
 * the worst case, before the size is known. */
uint64_t zvc_offload_host_bound(uint64_t n, uint32_t chunk_elems);

/* Workspace bytes for zvc_offload / zvc_prefetch (section V.D "Software Interface":
 * offload and prefetch with cudaMemcpyAsync): device staging for the pipelined
 * segments plus the per-segment kernel workspace. Where these sit inside a workspace
 * depends on its size alone, so one workspace of W bytes serves, in any order and on any
 * stream, every tensor whose zvc_offload_workspace_size is at most W; a smaller W returns
 * ZVC_ERR_BUFFER_TOO_SMALL. */
uint64_t zvc_offload_workspace_size(uint64_t n, uint32_t chunk_elems);

/* Offload (section V.D: vDNN offloads activations during forward propagation with
 * cudaMemcpyAsync, cDMA compresses them on the way). The tensor is cut into segments
 * of zvc_offload_segment_elems() words; each segment is compressed on `stream` into a
 * device staging buffer and copied to the pinned host buffer h_pinned with
 * cudaMemcpyAsync on the library's copy stream (one per device), so the copy of segment
 * k overlaps the compression of segment k+1, and the compression of the next tensor
 * overlaps the copies of this one. h_pinned receives a batch (format above) whose
 * streams are the segments; it is byte-identical to zvc_compress_batched over the
 * segments.
 * BLOCKS the calling thread until the last segment is compressed and its copy enqueued
 * (the host must learn each compressed size before it can enqueue the copy); *h_size
 * (host) holds the batch's byte count on return. Work enqueued on `stream` afterwards
 * waits for the compression only, not for the copies: d_in may be overwritten then,
 * h_pinned is complete once zvc_offload_join() has joined the copies into a stream
 * and that stream has reached that point (or the device is synchronised). A
 * zvc_prefetch of the batch needs no join: its copies follow on the same copy stream.
 * h_cap >= zvc_offload_host_bound(n, C). h_pinned must be page-locked (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister), hence mapped into the device's address space
 * under unified addressing, and 8-byte aligned: the compress kernels store each
 * segment's size straight into the buffer's batch table. Other host memory returns
 * ZVC_ERR_INVALID_ARG. */
zvc_status zvc_offload(const void* d_in, uint64_t n, uint32_t chunk_elems, void* h_pinned,
                       uint64_t h_cap, uint64_t* h_size, void* d_ws, uint64_t ws_bytes,
                       void* stream);

/* Offload join: work enqueued on `stream` after this call waits for every copy that
 * zvc_offload has enqueued on this device so far. Cites section V.D "Software Interface":
 * the copies are asynchronous (cudaMemcpyAsync), so a caller that reads the host copy
 * orders itself after them through this call. */
zvc_status zvc_offload_join(void* stream);

/* Prefetch (section V.D: vDNN prefetches offloaded activations before backward
 * propagation): copies each segment stream of the batch in h_pinned (h_size bytes, as
 * written by zvc_offload for n words and chunk_elems C) to device staging with
 * cudaMemcpyAsync on the library's copy stream and decompresses it into d_out on
 * `stream`, the copy of segment k+1 overlapping the decompression of segment k. The
 * copies follow the library's earlier copies (so an offload of h_pinned completes
 * first) and the kernel that last used each staging buffer; they do not wait for other
 * work on `stream`: a caller that fills h_pinned through `stream` synchronises first.
 * Reads the batch table on the host (a malformed table returns ZVC_ERR_CORRUPT at
 * once); device-side corruption is latched as for zvc_decompress. Does not block the
 * calling thread. */
zvc_status zvc_prefetch(const void* h_pinned, uint64_t h_size, void* d_out, uint64_t n,
                        uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream);

/* Self-test of the device-side wait limit; the paper has no counterpart (its engine is
 * hardware): launches the decoupled look-back of a tile whose predecessor never
 * publishes, with a wait limit of limit_ns (0 < limit_ns <= 1 s).
 * The wait gives up and latches ZVC_ERR_TIMEOUT in d_ws (read it with zvc_get_error);
 * the context stays usable. d_ws needs at least 1024 bytes. */
zvc_status zvc_selftest_wait_timeout(void* d_ws, uint64_t ws_bytes, uint64_t limit_ns,
                                     void* stream);

/* Kernel tracing; the paper has no counterpart (section V.D notes that its own evaluation
 * measured copy latencies on the host). zvc_trace_start() makes every following kernel
 * launch of this library
 * (on any stream, from any call, including the launches inside zvc_offload/zvc_prefetch)
 * record a CUDA event pair on its own stream. zvc_trace_stop() waits for those events,
 * stops tracing and writes, per kernel kind (index 0 = compress, 1 = decompress), the
 * number of launches to launches[2] and their summed device time in milliseconds to
 * device_ms[2] (host arrays). */
zvc_status zvc_trace_start(void);
zvc_status zvc_trace_stop(uint64_t* launches, double* device_ms);

/* Synchronises `stream`, returns the first device-side error latched in d_ws since the
 * last call (ZVC_OK if none) and clears it. Cites section V.D "Software Interface": the
 * proposed compressed copy call returns a result to its caller; errors that only the
 * device can see (a corrupt stream, a wait that gave up) reach the caller through here. */
zvc_status zvc_get_error(void* d_ws, void* stream);

/* ---------------------------------------------------------------------------------
 * Run-length encoding: the layout-dependent comparison codec of section V.A (RLE
 * exploits runs of zeros and of non-zeros, so its ratio depends on how the values are
 * laid out) and section VII.A (per 4 KB window; ZVC's ratio does not depend on the
 * layout, RLE's does). Not on the offload path: it is here to measure that comparison.
 *
 * RLE stream (little-endian, this project's reading: the pages give no byte layout):
 * u32 magic 0x31454C52 ("RLE1"), u16 version 1, u16 word_bytes 4, u32 window W, u32 0,
 * u64 n, u64 payload_bytes; u64 window_off[ceil(n/W)] (byte offset of each window's
 * records from the payload start); then per window of W words (the last may be shorter)
 * records of u16 zeros, u16 literals and `literals` words, where a record is the maximal
 * zero run at the cursor followed by the maximal non-zero run after it.
 * Size: 32 + 8 nw + 4 (records + non-zeros), at most 32 + 12 nw + 4 n. */
#define ZVC_RLE_MAX_WINDOW 4096u    /* words; the paper's 4 KB window is 1024 */

/* Worst-case RLE stream bytes for n words in windows of W (0 on invalid arguments).
 * Cites section V.A "Compression Algorithm" (RLE) under this library's record layout. */
uint64_t zvc_rle_size_bound(uint64_t n, uint32_t window);

/* Workspace bytes for zvc_rle_compress (window sizes and scan totals). Cites section V.A
 * (RLE) and section VII.A "Compression Efficiency" (per 4 KB window). */
uint64_t zvc_rle_workspace_size(uint64_t n, uint32_t window);

/* RLE-compress (section V.A "Compression Algorithm": runs of zeros and of non-zeros;
 * section VII.A: per window) n words at d_in (4-byte aligned) into d_out (8-byte aligned, out_cap >=
 * zvc_rle_size_bound), writing the stream's byte count to *d_out_size (device, 8-byte
 * aligned). Reads the input twice (window sizes, then the records); asynchronous. */
zvc_status zvc_rle_compress(const void* d_in, uint64_t n, uint32_t window, void* d_out,
                            uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                            void* stream);

/* Decompress the RLE stream of in_bytes bytes at d_in (8-byte aligned) into n words at
 * d_out (the inverse of section V.A's RLE). Host-visible size errors return ZVC_ERR_CORRUPT; every other check (header,
 * window offsets, records covering each window exactly) latches ZVC_ERR_CORRUPT in d_ws
 * (at least 256 bytes; read it with zvc_get_error), with no access outside the buffers. */
zvc_status zvc_rle_decompress(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                              uint32_t window, void* d_ws, uint64_t ws_bytes, void* stream);

/* The cudaError_t value behind the most recent ZVC_ERR_CUDA on this thread. The paper
 * has no counterpart: a library convenience. */
int zvc_last_cuda_error(void);

/* A static, human-readable name for a zvc_status. The paper has no counterpart: a
 * library convenience. */
const char* zvc_status_string(zvc_status s);

#ifdef __cplusplus
}
#endif

#endif /* ZVC_H_ */
