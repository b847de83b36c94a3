// C ABI of the ZVC library: argument checks, sizes, launches, the offload/prefetch
// pipeline and error readback. Every byte of compressed data is produced and consumed
// by the kernels in zvc_compress.cu and zvc_decompress.cu; this file only moves
// pointers, sizes and copies.
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include "zvc_internal.cuh"

using namespace zvc;

namespace {

thread_local int t_last_cuda_error = 0;

constexpr uint64_t kMaxElems = 1ull << 40;  // keeps every size computation far from overflow
constexpr int kPipeDepth = 3;               // staging buffers in flight for offload/prefetch

bool chunk_ok(uint32_t c) { return c != 0 && c % kWindow == 0 && c <= ZVC_MAX_CHUNK_ELEMS; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

uint64_t stream_bound(uint64_t n, uint32_t c, uint32_t word_bytes = 4) {
  return 32 + 8 * ceil_div_u64(n, c) + 4 * ceil_div_u64(n, kWindow) + word_bytes * n;
}

// Smallest valid stream for n words: every mask zero.
uint64_t stream_floor(uint64_t n, uint32_t c) {
  return 32 + 8 * ceil_div_u64(n, c) + 4 * ceil_div_u64(n, kWindow);
}

uint64_t batch_prefix(uint32_t T) { return 16 + 8 * ((uint64_t)T + 1); }

uint64_t compress_ws_bytes(uint64_t total_tiles, uint32_t T) {
  return round_up_u64(kStatusOffset + 8 * total_tiles + sizeof(TensorStart) * (uint64_t)T,
                      ZVC_WORKSPACE_ALIGN);
}

void put_u32(uint8_t* p, uint32_t v) { std::memcpy(p, &v, 4); }
void put_u64(uint8_t* p, uint64_t v) { std::memcpy(p, &v, 8); }
uint32_t get_u32(const uint8_t* p) { uint32_t v; std::memcpy(&v, p, 4); return v; }
uint64_t get_u64(const uint8_t* p) { uint64_t v; std::memcpy(&v, p, 8); return v; }

#define ZVC_CUDA_TRY(expr)                          \
  do {                                              \
    const cudaError_t e_ = (expr);                  \
    if (e_ != cudaSuccess) return cuda_failure(e_); \
  } while (0)

// ---------------------------------------------------------------- offload plan
struct SegPlan {
  uint64_t seg;         // words per segment (whole chunks)
  uint64_t count;       // segments
  uint64_t kernel_ws;   // workspace bytes one segment's compress needs
  uint64_t stage;       // bytes one staging buffer needs
};

uint64_t segment_elems(uint64_t n, uint32_t c) {
  // Equal segments of at most about 32 Mi words (128 MiB of fp32), whole chunks. Within a
  // tensor the copy of one segment overlaps the compression of the next; across tensors
  // the copies of one overlap the compression of the next, so only the first segment's
  // compression and the last one's decompression are exposed, and both kernels run on
  // tens of MB per launch.
  constexpr uint64_t kTarget = 1ull << 25;
  const uint64_t count = n == 0 ? 1 : ceil_div_u64(n, kTarget);
  return round_up_u64(ceil_div_u64(n == 0 ? 1 : n, count), c);
}

SegPlan seg_plan(uint64_t n, uint32_t c) {
  SegPlan p;
  p.seg = segment_elems(n, c);
  p.count = ceil_div_u64(n, p.seg);
  const uint64_t seg_n = n < p.seg ? n : p.seg;
  p.kernel_ws = compress_ws_bytes(tiles_for(seg_n), 1);
  p.stage = round_up_u64(stream_bound(seg_n, c), ZVC_WORKSPACE_ALIGN);
  return p;
}

// Where an offload workspace keeps the compress kernel's area and its three staging
// buffers. It depends on the workspace's size alone, so every offload and prefetch through
// one workspace, whatever its tensor's size, puts staging buffer b at the same bytes, and
// the per-buffer events of that workspace order every use of them.
struct WsLayout {
  uint64_t kernel_ws;  // bytes [0, kernel_ws): the compress kernel's area
  uint64_t stage;      // staging buffer b at kernel_ws + b * stage
};

WsLayout ws_layout(uint64_t ws_bytes) {
  WsLayout l;
  const uint64_t k = ceil_div_u64(ws_bytes, 1024);
  l.kernel_ws = round_up_u64(k < 4096 ? 4096 : k, ZVC_WORKSPACE_ALIGN);
  l.stage = ws_bytes > l.kernel_ws
                ? (ws_bytes - l.kernel_ws) / kPipeDepth / ZVC_WORKSPACE_ALIGN * ZVC_WORKSPACE_ALIGN
                : 0;
  return l;
}

bool layout_fits(const WsLayout& l, const SegPlan& p) {
  return l.kernel_ws >= p.kernel_ws && l.stage >= p.stage;
}

// Side stream (the copy stream) for the pipeline, one per device, created on first use,
// and per workspace the events of its staging buffers: the kernel and the copy that last
// used buffer b. A call holds the per-device mutex only to look its workspace's events up
// and to enqueue a group of copy-stream operations (wait, copy, record) in one piece; it
// never holds it while it blocks, so a zvc_prefetch from one thread is not queued behind
// a zvc_offload that waits for a kernel on another.
struct Slots {
  cudaEvent_t kernel_done[kPipeDepth] = {};
  cudaEvent_t copy_done[kPipeDepth] = {};
  // Destroying an event whose work is still pending is allowed: CUDA releases it once
  // the work completes.
  ~Slots() {
    for (int b = 0; b < kPipeDepth; ++b) {
      if (kernel_done[b]) cudaEventDestroy(kernel_done[b]);
      if (copy_done[b]) cudaEventDestroy(copy_done[b]);
    }
  }
};

struct Pipe {
  cudaStream_t side = nullptr;
  cudaEvent_t joined = nullptr;
  std::map<uintptr_t, std::shared_ptr<Slots>> slots;  // by workspace address
  std::mutex mu;
};

std::mutex g_pipes_mu;
std::map<int, Pipe*> g_pipes;

zvc_status get_pipe(Pipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failure(e);
  std::lock_guard<std::mutex> lk(g_pipes_mu);
  auto it = g_pipes.find(dev);
  if (it != g_pipes.end()) {
    *out = it->second;
    return ZVC_OK;
  }
  Pipe* p = new Pipe();
  e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->joined, cudaEventDisableTiming);
  if (e != cudaSuccess) return cuda_failure(e);  // the partial set leaks; CUDA is unusable
  g_pipes[dev] = p;
  *out = p;
  return ZVC_OK;
}

// The staging-buffer events of workspace ws (created on first use). Takes pipe->mu. A
// process that cycles through very many workspaces drops, once the table holds 4096 of
// them, every entry no call is using, after waiting for its events: a later call through
// such a workspace starts from fresh events, with the earlier work already done.
zvc_status slots_for(Pipe* pipe, const void* ws, std::shared_ptr<Slots>* out) {
  std::lock_guard<std::mutex> lk(pipe->mu);
  const uintptr_t key = reinterpret_cast<uintptr_t>(ws);
  auto it = pipe->slots.find(key);
  if (it == pipe->slots.end()) {
    if (pipe->slots.size() >= 4096) {
      for (auto j = pipe->slots.begin(); j != pipe->slots.end();) {
        if (j->second.use_count() != 1) {
          ++j;
          continue;
        }
        for (int b = 0; b < kPipeDepth; ++b) {
          ZVC_CUDA_TRY(cudaEventSynchronize(j->second->kernel_done[b]));
          ZVC_CUDA_TRY(cudaEventSynchronize(j->second->copy_done[b]));
        }
        j = pipe->slots.erase(j);
      }
    }
    auto sl = std::make_shared<Slots>();
    for (int b = 0; b < kPipeDepth; ++b) {
      ZVC_CUDA_TRY(cudaEventCreateWithFlags(&sl->kernel_done[b], cudaEventDisableTiming));
      ZVC_CUDA_TRY(cudaEventCreateWithFlags(&sl->copy_done[b], cudaEventDisableTiming));
    }
    it = pipe->slots.emplace(key, std::move(sl)).first;
  }
  *out = it->second;
  return ZVC_OK;
}

zvc_status read_latched(void* d_ws) {
  uint32_t err = 0;
  cudaError_t e = cudaMemcpy(&err, d_ws, sizeof(err), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_failure(e);
  return err ? (zvc_status)err : ZVC_ERR_CUDA;
}


// ---------------------------------------------------------------- tracing
struct TraceRec {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void recycle_trace() {
  for (const TraceRec& r : g_trace) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_trace.clear();
}

}  // namespace

TraceMark zvc::trace_begin(int kind, cudaStream_t stream) {
  TraceMark m;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace_on) return m;
  TraceRec r{kind, pooled_event(), pooled_event()};
  if (r.start == nullptr || r.stop == nullptr) return m;
  cudaEventRecord(r.start, stream);
  g_trace.push_back(r);
  m.stop = r.stop;
  return m;
}

void zvc::trace_end(TraceMark m, cudaStream_t stream) {
  if (m.stop != nullptr) cudaEventRecord(m.stop, stream);
}

zvc_status zvc::cuda_failure(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return ZVC_ERR_CUDA;
}

extern "C" {

uint64_t zvc_size_bound(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  return stream_bound(n, chunk_elems);
}

uint64_t zvc_batch_size_bound(const uint64_t* ns, uint32_t T, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || T > ZVC_MAX_BATCH || (T > 0 && ns == nullptr)) return 0;
  uint64_t s = batch_prefix(T);
  for (uint32_t i = 0; i < T; ++i) {
    if (ns[i] > kMaxElems) return 0;
    s += stream_bound(ns[i], chunk_elems);
  }
  return s;
}

uint64_t zvc_workspace_size(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  return compress_ws_bytes(tiles_for(n), 1);
}

uint64_t zvc_batch_workspace_size(const uint64_t* ns, uint32_t T, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || T > ZVC_MAX_BATCH || (T > 0 && ns == nullptr)) return 0;
  uint64_t tiles = 0;
  for (uint32_t i = 0; i < T; ++i) {
    if (ns[i] > kMaxElems) return 0;
    tiles += tiles_for(ns[i]);
  }
  return compress_ws_bytes(tiles, T);
}

zvc_status zvc_compress(const void* d_in, uint64_t n, uint32_t chunk_elems, void* d_out,
                        uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                        void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || d_out == nullptr || d_ws == nullptr ||
      (n > 0 && d_in == nullptr) || !aligned(d_in, 4) || !aligned(d_out, 4) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN) || !aligned(d_out_size, 8))
    return ZVC_ERR_INVALID_ARG;
  if (out_cap < stream_bound(n, chunk_elems) || ws_bytes < zvc_workspace_size(n, chunk_elems))
    return ZVC_ERR_BUFFER_TOO_SMALL;
  const TensorIn t{static_cast<const uint32_t*>(d_in), n};
  return launch_compress(&t, 1, false, chunk_elems, static_cast<uint32_t*>(d_out), out_cap / 4,
                         d_out_size, static_cast<uint8_t*>(d_ws), kDefaultWaitLimitNs,
                         static_cast<cudaStream_t>(stream));
}

uint64_t zvc_size_bound16(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  return stream_bound(n, chunk_elems, 2);
}

zvc_status zvc_compress16(const void* d_in, uint64_t n, uint32_t chunk_elems, void* d_out,
                          uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                          void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || d_out == nullptr || d_ws == nullptr ||
      (n > 0 && d_in == nullptr) || !aligned(d_in, 2) || !aligned(d_out, 4) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN) || !aligned(d_out_size, 8))
    return ZVC_ERR_INVALID_ARG;
  if (out_cap < stream_bound(n, chunk_elems, 2) || ws_bytes < zvc_workspace_size(n, chunk_elems))
    return ZVC_ERR_BUFFER_TOO_SMALL;
  return launch_compress16(static_cast<const uint16_t*>(d_in), n, chunk_elems,
                           static_cast<uint16_t*>(d_out), out_cap / 2, d_out_size,
                           static_cast<uint8_t*>(d_ws), kDefaultWaitLimitNs,
                           static_cast<cudaStream_t>(stream));
}

zvc_status zvc_decompress16(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                            uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || d_in == nullptr || d_ws == nullptr ||
      (n > 0 && d_out == nullptr) || !aligned(d_in, 4) || !aligned(d_out, 2) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  if (ws_bytes < kControlBytes) return ZVC_ERR_BUFFER_TOO_SMALL;
  // sizes no valid stream of n 16-bit words can have
  if (in_bytes % 2 != 0 || in_bytes < stream_floor(n, chunk_elems) ||
      in_bytes > stream_bound(n, chunk_elems, 2))
    return ZVC_ERR_CORRUPT;
  return launch_decompress16(static_cast<const uint32_t*>(d_in), in_bytes,
                             static_cast<uint16_t*>(d_out), n, chunk_elems,
                             static_cast<uint8_t*>(d_ws), static_cast<cudaStream_t>(stream));
}

zvc_status zvc_decompress(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                          uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || d_in == nullptr || d_ws == nullptr ||
      (n > 0 && d_out == nullptr) || !aligned(d_in, 4) || !aligned(d_out, 4) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  if (ws_bytes < kControlBytes) return ZVC_ERR_BUFFER_TOO_SMALL;
  // sizes no valid stream of n words can have
  if (in_bytes % 4 != 0 || in_bytes < stream_floor(n, chunk_elems) ||
      in_bytes > stream_bound(n, chunk_elems))
    return ZVC_ERR_CORRUPT;
  const TensorOut t{static_cast<uint32_t*>(d_out), n};
  return launch_decompress(static_cast<const uint32_t*>(d_in), in_bytes, &t, 1, false,
                           chunk_elems, static_cast<uint8_t*>(d_ws),
                           static_cast<cudaStream_t>(stream));
}

zvc_status zvc_compress_batched(const void* const* d_ins, const uint64_t* ns, uint32_t T,
                                uint32_t chunk_elems, void* d_out, uint64_t out_cap,
                                uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                                void* stream) {
  if (!chunk_ok(chunk_elems) || T > ZVC_MAX_BATCH || (T > 0 && (d_ins == nullptr || ns == nullptr)) ||
      d_out == nullptr || d_ws == nullptr || !aligned(d_out, 4) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN) || !aligned(d_out_size, 8))
    return ZVC_ERR_INVALID_ARG;
  std::vector<TensorIn> ts(T);
  for (uint32_t i = 0; i < T; ++i) {
    if (ns[i] > kMaxElems || (ns[i] > 0 && d_ins[i] == nullptr) || !aligned(d_ins[i], 4))
      return ZVC_ERR_INVALID_ARG;
    ts[i] = TensorIn{static_cast<const uint32_t*>(d_ins[i]), ns[i]};
  }
  if (out_cap < zvc_batch_size_bound(ns, T, chunk_elems) ||
      ws_bytes < zvc_batch_workspace_size(ns, T, chunk_elems))
    return ZVC_ERR_BUFFER_TOO_SMALL;
  return launch_compress(ts.data(), T, true, chunk_elems, static_cast<uint32_t*>(d_out),
                         out_cap / 4, d_out_size, static_cast<uint8_t*>(d_ws),
                         kDefaultWaitLimitNs, static_cast<cudaStream_t>(stream));
}

zvc_status zvc_decompress_batched(const void* d_in, uint64_t in_bytes, void* const* d_outs,
                                  const uint64_t* ns, uint32_t T, uint32_t chunk_elems,
                                  void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!chunk_ok(chunk_elems) || T > ZVC_MAX_BATCH || (T > 0 && (d_outs == nullptr || ns == nullptr)) ||
      d_in == nullptr || d_ws == nullptr || !aligned(d_in, 4) || !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  if (ws_bytes < kControlBytes) return ZVC_ERR_BUFFER_TOO_SMALL;
  std::vector<TensorOut> ts(T);
  uint64_t floor = batch_prefix(T);
  for (uint32_t i = 0; i < T; ++i) {
    if (ns[i] > kMaxElems || (ns[i] > 0 && d_outs[i] == nullptr) || !aligned(d_outs[i], 4))
      return ZVC_ERR_INVALID_ARG;
    ts[i] = TensorOut{static_cast<uint32_t*>(d_outs[i]), ns[i]};
    floor += stream_floor(ns[i], chunk_elems);
  }
  if (in_bytes % 4 != 0 || in_bytes < floor || in_bytes > zvc_batch_size_bound(ns, T, chunk_elems))
    return ZVC_ERR_CORRUPT;
  return launch_decompress(static_cast<const uint32_t*>(d_in), in_bytes, ts.data(), T, true,
                           chunk_elems, static_cast<uint8_t*>(d_ws),
                           static_cast<cudaStream_t>(stream));
}

uint64_t zvc_offload_segment_elems(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  return segment_elems(n, chunk_elems);
}

uint64_t zvc_offload_host_bound(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  const SegPlan p = seg_plan(n, chunk_elems);
  uint64_t s = batch_prefix((uint32_t)p.count);
  for (uint64_t k = 0; k < p.count; ++k) {
    const uint64_t nk = (k + 1 < p.count) ? p.seg : n - k * p.seg;
    s += stream_bound(nk, chunk_elems);
  }
  return s;
}

uint64_t zvc_offload_workspace_size(uint64_t n, uint32_t chunk_elems) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems) return 0;
  const SegPlan p = seg_plan(n, chunk_elems);
  // the smallest size whose layout fits: about kPipeDepth * stage + 1/1024 of itself
  uint64_t w = round_up_u64(kPipeDepth * p.stage + p.kernel_ws + 4096, ZVC_WORKSPACE_ALIGN);
  while (!layout_fits(ws_layout(w), p)) w += round_up_u64(w / 512 + 1, ZVC_WORKSPACE_ALIGN);
  return w;
}

zvc_status zvc_offload(const void* d_in, uint64_t n, uint32_t chunk_elems, void* h_pinned,
                       uint64_t h_cap, uint64_t* h_size, void* d_ws, uint64_t ws_bytes,
                       void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || h_pinned == nullptr || h_size == nullptr ||
      d_ws == nullptr || (n > 0 && d_in == nullptr) || !aligned(d_in, 4) ||
      !aligned(h_pinned, 8) || !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  const SegPlan p = seg_plan(n, chunk_elems);
  if (p.count > UINT32_MAX) return ZVC_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(ws_bytes);
  if (h_cap < zvc_offload_host_bound(n, chunk_elems) || !layout_fits(L, p))
    return ZVC_ERR_BUFFER_TOO_SMALL;
  // The kernels store each segment's compressed size straight into the pinned buffer, so
  // the host learns it without a copy queued behind the previous segment's transfer.
  // That needs h_pinned mapped into the device's address space, as page-locked memory
  // is under unified addressing.
  uint8_t* Hdev = nullptr;
  if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&Hdev), h_pinned, 0) != cudaSuccess ||
      Hdev == nullptr) {
    (void)cudaGetLastError();
    return ZVC_ERR_INVALID_ARG;
  }
  Pipe* pipe = nullptr;
  zvc_status st = get_pipe(&pipe);
  if (st != ZVC_OK) return st;
  std::shared_ptr<Slots> sl;
  if ((st = slots_for(pipe, d_ws, &sl)) != ZVC_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  uint8_t* H = static_cast<uint8_t*>(h_pinned);
  const uint32_t* in = static_cast<const uint32_t*>(d_in);
  const uint64_t S = p.count;
  const uint64_t prefix = batch_prefix((uint32_t)S);
  uint64_t pos = prefix;
  std::vector<uint64_t> offs(S + 1, 0);

  // The compress kernel of segment k writes its compressed size into the segment's (not
  // yet written) batch-table slot of the pinned buffer; once the host has seen it, the
  // segment's copy is enqueued. A kernel that fails before its last step leaves the 0 the
  // host put there.
  auto enqueue_copy = [&](uint64_t k) -> zvc_status {
    const int b = (int)(k % kPipeDepth);
    ZVC_CUDA_TRY(cudaEventSynchronize(sl->kernel_done[b]));
    const uint64_t sz = *reinterpret_cast<volatile uint64_t*>(H + 16 + 8 * k);
    if (sz == 0 || sz > L.stage || pos + sz > h_cap) return read_latched(d_ws);
    offs[k] = pos;
    {
      std::lock_guard<std::mutex> lk(pipe->mu);  // the three copy-stream steps in one piece
      ZVC_CUDA_TRY(cudaStreamWaitEvent(pipe->side, sl->kernel_done[b], 0));
      ZVC_CUDA_TRY(cudaMemcpyAsync(H + pos, ws + L.kernel_ws + b * L.stage, sz,
                                   cudaMemcpyDeviceToHost, pipe->side));
      ZVC_CUDA_TRY(cudaEventRecord(sl->copy_done[b], pipe->side));
    }
    pos += sz;
    return ZVC_OK;
  };

  for (uint64_t k = 0; k < S; ++k) {
    const int b = (int)(k % kPipeDepth);
    // staging buffer b is free once the copy and the kernel that last used it (this
    // call's or an earlier one's, on any stream) are done
    ZVC_CUDA_TRY(cudaStreamWaitEvent(s, sl->copy_done[b], 0));
    ZVC_CUDA_TRY(cudaStreamWaitEvent(s, sl->kernel_done[b], 0));
    const uint64_t nk = (k + 1 < S) ? p.seg : n - k * p.seg;
    const TensorIn t{in + k * p.seg, nk};
    *reinterpret_cast<volatile uint64_t*>(H + 16 + 8 * k) = 0;
    st = launch_compress(&t, 1, false, chunk_elems,
                         reinterpret_cast<uint32_t*>(ws + L.kernel_ws + b * L.stage), L.stage / 4,
                         reinterpret_cast<uint64_t*>(Hdev + 16 + 8 * k), ws, kDefaultWaitLimitNs,
                         s);
    if (st != ZVC_OK) return st;
    ZVC_CUDA_TRY(cudaEventRecord(sl->kernel_done[b], s));
    if (k >= 1 && (st = enqueue_copy(k - 1)) != ZVC_OK) return st;
  }
  if (S >= 1 && (st = enqueue_copy(S - 1)) != ZVC_OK) return st;
  offs[S] = pos;

  put_u32(H + 0, kBatchMagic);
  put_u32(H + 4, (uint32_t)S);
  put_u64(H + 8, pos);
  for (uint64_t k = 0; k <= S; ++k) put_u64(H + 16 + 8 * k, offs[k]);
  *h_size = pos;
  return ZVC_OK;
}

zvc_status zvc_offload_join(void* stream) {
  Pipe* pipe = nullptr;
  zvc_status st = get_pipe(&pipe);
  if (st != ZVC_OK) return st;
  std::lock_guard<std::mutex> lk(pipe->mu);
  ZVC_CUDA_TRY(cudaEventRecord(pipe->joined, pipe->side));
  ZVC_CUDA_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), pipe->joined, 0));
  return ZVC_OK;
}

zvc_status zvc_prefetch(const void* h_pinned, uint64_t h_size, void* d_out, uint64_t n,
                        uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!chunk_ok(chunk_elems) || n > kMaxElems || h_pinned == nullptr || d_ws == nullptr ||
      (n > 0 && d_out == nullptr) || !aligned(d_out, 4) || !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  const SegPlan p = seg_plan(n, chunk_elems);
  const WsLayout L = ws_layout(ws_bytes);
  if (!layout_fits(L, p)) return ZVC_ERR_BUFFER_TOO_SMALL;
  const uint8_t* H = static_cast<const uint8_t*>(h_pinned);
  const uint64_t S = p.count;
  const uint64_t prefix = batch_prefix((uint32_t)S);
  if (h_size < prefix || get_u32(H) != kBatchMagic || get_u32(H + 4) != S ||
      get_u64(H + 8) != h_size || get_u64(H + 16) != prefix || get_u64(H + 16 + 8 * S) != h_size)
    return ZVC_ERR_CORRUPT;
  for (uint64_t k = 0; k < S; ++k) {
    const uint64_t a = get_u64(H + 16 + 8 * k), b = get_u64(H + 24 + 8 * k);
    const uint64_t nk = (k + 1 < S) ? p.seg : n - k * p.seg;
    if (a > b || ((a | b) & 3u) != 0 || b - a < stream_floor(nk, chunk_elems) ||
        b - a > stream_bound(nk, chunk_elems))
      return ZVC_ERR_CORRUPT;
  }
  Pipe* pipe = nullptr;
  zvc_status st = get_pipe(&pipe);
  if (st != ZVC_OK) return st;
  std::shared_ptr<Slots> sl;
  if ((st = slots_for(pipe, d_ws, &sl)) != ZVC_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  uint32_t* out = static_cast<uint32_t*>(d_out);
  // The copies run on the library's copy stream, after its earlier copies (an offload's,
  // which wrote h_pinned); staging buffer b is free once the kernel that last read or
  // wrote it is done.
  for (uint64_t k = 0; k < S; ++k) {
    const int b = (int)(k % kPipeDepth);
    const uint64_t a = get_u64(H + 16 + 8 * k), sz = get_u64(H + 24 + 8 * k) - a;
    uint8_t* stage = ws + L.kernel_ws + b * L.stage;
    {
      std::lock_guard<std::mutex> lk(pipe->mu);  // the three copy-stream steps in one piece
      ZVC_CUDA_TRY(cudaStreamWaitEvent(pipe->side, sl->kernel_done[b], 0));
      ZVC_CUDA_TRY(cudaMemcpyAsync(stage, H + a, sz, cudaMemcpyHostToDevice, pipe->side));
      ZVC_CUDA_TRY(cudaEventRecord(sl->copy_done[b], pipe->side));
    }
    ZVC_CUDA_TRY(cudaStreamWaitEvent(s, sl->copy_done[b], 0));
    const uint64_t nk = (k + 1 < S) ? p.seg : n - k * p.seg;
    const TensorOut t{out + k * p.seg, nk};
    st = launch_decompress(reinterpret_cast<const uint32_t*>(stage), sz, &t, 1, false,
                           chunk_elems, ws, s);
    if (st != ZVC_OK) return st;
    ZVC_CUDA_TRY(cudaEventRecord(sl->kernel_done[b], s));
  }
  return ZVC_OK;
}

// ---------------------------------------------------------------- RLE comparison codec
bool rle_window_ok(uint32_t w) { return w >= 32 && w % 32 == 0 && w <= ZVC_RLE_MAX_WINDOW; }

uint64_t zvc_rle_size_bound(uint64_t n, uint32_t window) {
  if (!rle_window_ok(window) || n > kMaxElems) return 0;
  return 32 + 12 * ceil_div_u64(n, window) + 4 * n;
}

uint64_t zvc_rle_workspace_size(uint64_t n, uint32_t window) {
  if (!rle_window_ok(window) || n > kMaxElems) return 0;
  return rle_ws_bytes(n, window);
}

zvc_status zvc_rle_compress(const void* d_in, uint64_t n, uint32_t window, void* d_out,
                            uint64_t out_cap, uint64_t* d_out_size, void* d_ws, uint64_t ws_bytes,
                            void* stream) {
  if (!rle_window_ok(window) || n > kMaxElems || d_out == nullptr || d_ws == nullptr ||
      (n > 0 && d_in == nullptr) || !aligned(d_in, 4) || !aligned(d_out, 8) ||
      !aligned(d_out_size, 8) || !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  if (out_cap < zvc_rle_size_bound(n, window) || ws_bytes < rle_ws_bytes(n, window))
    return ZVC_ERR_BUFFER_TOO_SMALL;
  return launch_rle_compress(static_cast<const uint32_t*>(d_in), n, window,
                             static_cast<uint32_t*>(d_out), d_out_size,
                             static_cast<uint8_t*>(d_ws), static_cast<cudaStream_t>(stream));
}

zvc_status zvc_rle_decompress(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n,
                              uint32_t window, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!rle_window_ok(window) || n > kMaxElems || d_in == nullptr || d_ws == nullptr ||
      (n > 0 && d_out == nullptr) || !aligned(d_in, 8) || !aligned(d_out, 4) ||
      !aligned(d_ws, ZVC_WORKSPACE_ALIGN))
    return ZVC_ERR_INVALID_ARG;
  if (ws_bytes < kControlBytes) return ZVC_ERR_BUFFER_TOO_SMALL;
  const uint64_t nwin = ceil_div_u64(n, window);
  // sizes no valid stream of n words can have: at least one record per window, at most
  // the bound
  if (in_bytes % 4 != 0 || in_bytes < 32 + 12 * nwin || in_bytes > zvc_rle_size_bound(n, window))
    return ZVC_ERR_CORRUPT;
  return launch_rle_decompress(static_cast<const uint32_t*>(d_in), in_bytes,
                               static_cast<uint32_t*>(d_out), n, window,
                               static_cast<uint8_t*>(d_ws), static_cast<cudaStream_t>(stream));
}

zvc_status zvc_get_error(void* d_ws, void* stream) {
  if (d_ws == nullptr || !aligned(d_ws, ZVC_WORKSPACE_ALIGN)) return ZVC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ZVC_CUDA_TRY(cudaStreamSynchronize(s));
  uint32_t err = 0;
  ZVC_CUDA_TRY(cudaMemcpy(&err, d_ws, sizeof(err), cudaMemcpyDeviceToHost));
  if (err != 0) ZVC_CUDA_TRY(cudaMemset(d_ws, 0, sizeof(Control)));
  return (zvc_status)err;
}

zvc_status zvc_selftest_wait_timeout(void* d_ws, uint64_t ws_bytes, uint64_t limit_ns,
                                     void* stream) {
  if (d_ws == nullptr || !aligned(d_ws, ZVC_WORKSPACE_ALIGN) || limit_ns == 0 ||
      limit_ns > kDefaultWaitLimitNs)
    return ZVC_ERR_INVALID_ARG;
  if (ws_bytes < compress_ws_bytes(2, 1)) return ZVC_ERR_BUFFER_TOO_SMALL;
  return launch_lookback_timeout_probe(static_cast<uint8_t*>(d_ws), limit_ns,
                                       static_cast<cudaStream_t>(stream));
}

zvc_status zvc_trace_start(void) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  recycle_trace();
  g_trace_on = true;
  return ZVC_OK;
}

zvc_status zvc_trace_stop(uint64_t* launches, double* device_ms) {
  if (launches == nullptr || device_ms == nullptr) return ZVC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on = false;
  for (int k = 0; k < kTraceKinds; ++k) {
    launches[k] = 0;
    device_ms[k] = 0.0;
  }
  for (const TraceRec& r : g_trace) {
    ZVC_CUDA_TRY(cudaEventSynchronize(r.stop));
    float ms = 0.f;
    ZVC_CUDA_TRY(cudaEventElapsedTime(&ms, r.start, r.stop));
    launches[r.kind] += 1;
    device_ms[r.kind] += ms;
  }
  recycle_trace();
  return ZVC_OK;
}

int zvc_last_cuda_error(void) { return t_last_cuda_error; }

const char* zvc_status_string(zvc_status s) {
  switch (s) {
    case ZVC_OK: return "ZVC_OK";
    case ZVC_ERR_INVALID_ARG: return "ZVC_ERR_INVALID_ARG";
    case ZVC_ERR_BUFFER_TOO_SMALL: return "ZVC_ERR_BUFFER_TOO_SMALL";
    case ZVC_ERR_CORRUPT: return "ZVC_ERR_CORRUPT";
    case ZVC_ERR_TIMEOUT: return "ZVC_ERR_TIMEOUT";
    case ZVC_ERR_CUDA: return "ZVC_ERR_CUDA";
    default: return "ZVC_ERR_UNKNOWN";
  }
}

}  // extern "C"
