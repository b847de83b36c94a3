// zvc_compress_static: the compress call for callers that cannot allocate device memory.
//
// zvc_compress needs a caller-provided workspace for the tiles' look-back status words
// and the error word. Some callers have no way to provide one: code that runs under a
// memory manager which owns every byte of device memory (a framework's pool or a fixed
// memory plan decided ahead of time) and forbids side allocations, or code that must not
// call cudaMalloc because it synchronises the device and can fail once the memory is
// fully reserved. For them this variant keeps its scratch in one file-scope device array
// that is part of the library image: every GPU that loads the library holds
// kStaticScratchBytes of it until the process exits.
//
// The array is shared by every call on a device and keeps the previous call's contents.
// Nothing in it is cleared between calls: every compress launch tags the status words it
// writes with a number drawn anew for that launch, so entries left by earlier calls never
// match the new call's. Only the error latch carries over from one call to the next: it
// keeps a failure until zvc_compress_static_get_error reads and clears it. Two calls whose
// work overlaps on the GPU (different streams, no ordering between them) use the same
// scratch and race: order them on one stream or synchronise between them.
#include "zvc_internal.cuh"

namespace {

// Control block, reserved block, one status word per 4096-word tile for up to
// ZVC_STATIC_MAX_ELEMS words and one tensor start, rounded up to a whole 4 KiB page.
constexpr uint64_t kStaticScratchBytes = 1052672;  // 1 MiB + 4 KiB
static_assert(zvc::kStatusOffset + 8 * (ZVC_STATIC_MAX_ELEMS / zvc::kTileElems) +
                      sizeof(zvc::TensorStart) <=
                  kStaticScratchBytes,
              "static scratch too small for ZVC_STATIC_MAX_ELEMS");

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// The device address of g_static_scratch on the current device. In host code the name
// g_static_scratch is only a host-side stand-in for the symbol, so the address is looked
// up with the device current, on every call: a cached address would dangle once the
// device's context is torn down (cudaDeviceReset) and the module loaded again. The first
// lookup on a device also loads the library's device code there.
zvc_status scratch_for_current_device(uint8_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return zvc::cuda_failure(e);
  *out = static_cast<uint8_t*>(p);
  return ZVC_OK;
}

bool aligned_to(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" zvc_status zvc_compress_static(const void* d_in, uint64_t n, uint32_t chunk_elems,
                                          void* d_out, uint64_t out_cap, uint64_t* d_out_size,
                                          void* stream) {
  if (chunk_elems == 0 || chunk_elems % zvc::kWindow != 0 || chunk_elems > ZVC_MAX_CHUNK_ELEMS ||
      d_out == nullptr || (n > 0 && d_in == nullptr) || !aligned_to(d_in, 4) ||
      !aligned_to(d_out, 4) || !aligned_to(d_out_size, 8))
    return ZVC_ERR_INVALID_ARG;
  if (n > ZVC_STATIC_MAX_ELEMS) return ZVC_ERR_INVALID_ARG;  // beyond the static scratch
  if (out_cap < zvc_size_bound(n, chunk_elems)) return ZVC_ERR_BUFFER_TOO_SMALL;
  uint8_t* scratch = nullptr;
  zvc_status st = scratch_for_current_device(&scratch);
  if (st != ZVC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const zvc::TensorIn t{static_cast<const uint32_t*>(d_in), n};
  return zvc::launch_compress(&t, 1, false, chunk_elems, static_cast<uint32_t*>(d_out),
                              out_cap / 4, d_out_size, scratch, zvc::kDefaultWaitLimitNs, s);
}

extern "C" zvc_status zvc_compress_static_get_error(void* stream) {
  uint8_t* scratch = nullptr;
  zvc_status st = scratch_for_current_device(&scratch);
  if (st != ZVC_OK) return st;
  return zvc_get_error(scratch, stream);
}
