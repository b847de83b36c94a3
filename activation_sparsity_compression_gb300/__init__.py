"""Python binding of the ZVC C ABI declared in include/zvc.h (ctypes).

Zero-value compression of sparse activation maps after Rhu et al., "Compressing DMA
Engine: Leveraging Activation Sparsity for Training Deep Neural Networks", section V.A:
each 32-word window becomes a 32-bit non-zero mask followed by its non-zero words.

The functions named ``zvc_*`` mirror the C calls one to one and take raw integers
(device pointers, sizes, a cudaStream_t handle); they only marshal arguments. The
helpers at the bottom (``compress``, ``decompress``, ...) add PyTorch allocation of the
output and workspace buffers around the same calls. Every byte of compressed data is
produced by the library's sm_103a kernels: if the shared library is missing the first
call raises, there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

ZVC_OK = 0
ZVC_ERR_INVALID_ARG = 1
ZVC_ERR_BUFFER_TOO_SMALL = 2
ZVC_ERR_CORRUPT = 3
ZVC_ERR_TIMEOUT = 4
ZVC_ERR_CUDA = 5
ZVC_WINDOW = 32
ZVC_DEFAULT_CHUNK_ELEMS = 4096
ZVC_MAX_CHUNK_ELEMS = 32768
ZVC_MAX_BATCH = 512
ZVC_WORKSPACE_ALIGN = 256
ZVC_STATIC_MAX_ELEMS = 1 << 29
ZVC_RLE_MAX_WINDOW = 4096

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzvc_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "zvc.h")

_lock = threading.Lock()
_lib = None

_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_vp = ctypes.c_void_p
_st = ctypes.c_int
_SIGS = {
    "zvc_size_bound": (_u64, [_u64, _u32]),
    "zvc_batch_size_bound": (_u64, [ctypes.POINTER(_u64), _u32, _u32]),
    "zvc_workspace_size": (_u64, [_u64, _u32]),
    "zvc_batch_workspace_size": (_u64, [ctypes.POINTER(_u64), _u32, _u32]),
    "zvc_compress": (_st, [_vp, _u64, _u32, _vp, _u64, _vp, _vp, _u64, _vp]),
    "zvc_decompress": (_st, [_vp, _u64, _vp, _u64, _u32, _vp, _u64, _vp]),
    "zvc_compress_static": (_st, [_vp, _u64, _u32, _vp, _u64, _vp, _vp]),
    "zvc_size_bound16": (_u64, [_u64, _u32]),
    "zvc_compress16": (_st, [_vp, _u64, _u32, _vp, _u64, _vp, _vp, _u64, _vp]),
    "zvc_decompress16": (_st, [_vp, _u64, _vp, _u64, _u32, _vp, _u64, _vp]),
    "zvc_compress_batched": (_st, [ctypes.POINTER(_vp), ctypes.POINTER(_u64), _u32, _u32, _vp,
                                   _u64, _vp, _vp, _u64, _vp]),
    "zvc_decompress_batched": (_st, [_vp, _u64, ctypes.POINTER(_vp), ctypes.POINTER(_u64), _u32,
                                     _u32, _vp, _u64, _vp]),
    "zvc_offload_segment_elems": (_u64, [_u64, _u32]),
    "zvc_offload_host_bound": (_u64, [_u64, _u32]),
    "zvc_offload_workspace_size": (_u64, [_u64, _u32]),
    "zvc_compress_static_get_error": (_st, [_vp]),
    "zvc_rle_size_bound": (_u64, [_u64, _u32]),
    "zvc_rle_workspace_size": (_u64, [_u64, _u32]),
    "zvc_rle_compress": (_st, [_vp, _u64, _u32, _vp, _u64, _vp, _vp, _u64, _vp]),
    "zvc_rle_decompress": (_st, [_vp, _u64, _vp, _u64, _u32, _vp, _u64, _vp]),
    "zvc_offload_join": (_st, [_vp]),
    "zvc_offload": (_st, [_vp, _u64, _u32, _vp, _u64, ctypes.POINTER(_u64), _vp, _u64, _vp]),
    "zvc_prefetch": (_st, [_vp, _u64, _vp, _u64, _u32, _vp, _u64, _vp]),
    "zvc_selftest_wait_timeout": (_st, [_vp, _u64, _u64, _vp]),
    "zvc_get_error": (_st, [_vp, _vp]),
    "zvc_trace_start": (_st, []),
    "zvc_trace_stop": (_st, [ctypes.POINTER(_u64), ctypes.POINTER(ctypes.c_double)]),
    "zvc_last_cuda_error": (ctypes.c_int, []),
    "zvc_status_string": (ctypes.c_char_p, [_st]),
}


class ZvcError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})" if where else
                         f"{status_string(status)} ({status})")


def lib():
    """The loaded shared library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "activation_sparsity_compression_gb300.build.build() (needs nvcc)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def header_functions(path: str = HEADER_PATH):
    """Names of the functions declared in include/zvc.h."""
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(zvc_[a-z_0-9]+)\s*\(", text)))


def _u64_array(xs):
    xs = [int(x) for x in xs]
    return (_u64 * max(len(xs), 1))(*xs), len(xs)


def _ptr_array(ps):
    ps = [int(p) for p in ps]
    return (_vp * max(len(ps), 1))(*ps)


# ----------------------------------------------------------------- one-to-one calls
def zvc_size_bound(n, chunk_elems):
    return int(lib().zvc_size_bound(n, chunk_elems))


def zvc_batch_size_bound(ns, chunk_elems):
    arr, T = _u64_array(ns)
    return int(lib().zvc_batch_size_bound(arr, T, chunk_elems))


def zvc_workspace_size(n, chunk_elems):
    return int(lib().zvc_workspace_size(n, chunk_elems))


def zvc_batch_workspace_size(ns, chunk_elems):
    arr, T = _u64_array(ns)
    return int(lib().zvc_batch_workspace_size(arr, T, chunk_elems))


def zvc_compress(d_in, n, chunk_elems, d_out, out_cap, d_out_size, d_ws, ws_bytes, stream):
    return int(lib().zvc_compress(d_in, n, chunk_elems, d_out, out_cap, d_out_size, d_ws,
                                  ws_bytes, stream))


def zvc_compress_static(d_in, n, chunk_elems, d_out, out_cap, d_out_size, stream):
    """zvc_compress for callers that cannot allocate device memory: no workspace, the
    scratch is a static device array inside the library (n <= ZVC_STATIC_MAX_ELEMS)."""
    return int(lib().zvc_compress_static(d_in, n, chunk_elems, d_out, out_cap, d_out_size, stream))


def zvc_compress_static_get_error(stream):
    """Status latched by zvc_compress_static on this device since the last read; clears it."""
    return int(lib().zvc_compress_static_get_error(stream))


def zvc_size_bound16(n, chunk_elems):
    return int(lib().zvc_size_bound16(n, chunk_elems))


def zvc_compress16(d_in, n, chunk_elems, d_out, out_cap, d_out_size, d_ws, ws_bytes, stream):
    return lib().zvc_compress16(d_in, n, chunk_elems, d_out, out_cap, d_out_size, d_ws, ws_bytes,
                                stream)


def zvc_decompress16(d_in, in_bytes, d_out, n, chunk_elems, d_ws, ws_bytes, stream):
    return lib().zvc_decompress16(d_in, in_bytes, d_out, n, chunk_elems, d_ws, ws_bytes, stream)


def zvc_decompress(d_in, in_bytes, d_out, n, chunk_elems, d_ws, ws_bytes, stream):
    return int(lib().zvc_decompress(d_in, in_bytes, d_out, n, chunk_elems, d_ws, ws_bytes, stream))


def zvc_compress_batched(d_ins, ns, chunk_elems, d_out, out_cap, d_out_size, d_ws, ws_bytes,
                         stream):
    arr, T = _u64_array(ns)
    return int(lib().zvc_compress_batched(_ptr_array(d_ins), arr, T, chunk_elems, d_out, out_cap,
                                          d_out_size, d_ws, ws_bytes, stream))


def zvc_decompress_batched(d_in, in_bytes, d_outs, ns, chunk_elems, d_ws, ws_bytes, stream):
    arr, T = _u64_array(ns)
    return int(lib().zvc_decompress_batched(d_in, in_bytes, _ptr_array(d_outs), arr, T,
                                            chunk_elems, d_ws, ws_bytes, stream))


def zvc_offload_segment_elems(n, chunk_elems):
    return int(lib().zvc_offload_segment_elems(n, chunk_elems))


def zvc_offload_host_bound(n, chunk_elems):
    return int(lib().zvc_offload_host_bound(n, chunk_elems))


def zvc_offload_workspace_size(n, chunk_elems):
    return int(lib().zvc_offload_workspace_size(n, chunk_elems))


def zvc_offload(d_in, n, chunk_elems, h_pinned, h_cap, d_ws, ws_bytes, stream):
    """Returns (status, h_size)."""
    size = _u64(0)
    st = int(lib().zvc_offload(d_in, n, chunk_elems, h_pinned, h_cap, ctypes.byref(size), d_ws,
                               ws_bytes, stream))
    return st, int(size.value)


def zvc_rle_size_bound(n, window):
    return int(lib().zvc_rle_size_bound(n, window))


def zvc_rle_workspace_size(n, window):
    return int(lib().zvc_rle_workspace_size(n, window))


def zvc_rle_compress(d_in, n, window, d_out, out_cap, d_out_size, d_ws, ws_bytes, stream):
    return int(lib().zvc_rle_compress(d_in, n, window, d_out, out_cap, d_out_size, d_ws, ws_bytes,
                                      stream))


def zvc_rle_decompress(d_in, in_bytes, d_out, n, window, d_ws, ws_bytes, stream):
    return int(lib().zvc_rle_decompress(d_in, in_bytes, d_out, n, window, d_ws, ws_bytes, stream))


def zvc_offload_join(stream):
    """Work enqueued on `stream` afterwards waits for every copy zvc_offload enqueued."""
    return int(lib().zvc_offload_join(stream))


def zvc_prefetch(h_pinned, h_size, d_out, n, chunk_elems, d_ws, ws_bytes, stream):
    return int(lib().zvc_prefetch(h_pinned, h_size, d_out, n, chunk_elems, d_ws, ws_bytes, stream))


def zvc_selftest_wait_timeout(d_ws, ws_bytes, limit_ns, stream):
    return int(lib().zvc_selftest_wait_timeout(d_ws, ws_bytes, limit_ns, stream))


def zvc_get_error(d_ws, stream):
    return int(lib().zvc_get_error(d_ws, stream))


def zvc_trace_start():
    return int(lib().zvc_trace_start())


def zvc_trace_stop():
    """Returns (status, {"compress": (launches, ms), "decompress": (launches, ms)})."""
    launches = (_u64 * 2)()
    ms = (ctypes.c_double * 2)()
    st = int(lib().zvc_trace_stop(launches, ms))
    return st, {"compress": (int(launches[0]), float(ms[0])),
                "decompress": (int(launches[1]), float(ms[1]))}


def zvc_last_cuda_error():
    return int(lib().zvc_last_cuda_error())


def status_string(status):
    return lib().zvc_status_string(int(status)).decode()


zvc_status_string = status_string


# ----------------------------------------------------------------- torch helpers
def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(st, where):
    if st != ZVC_OK:
        raise ZvcError(st, where)


def new_workspace(nbytes, device="cuda"):
    """A zero-filled, 256-byte aligned device workspace of at least nbytes."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), ZVC_WORKSPACE_ALIGN), dtype=torch.uint8, device=device)


def _words(x):
    torch = _torch()
    if not x.is_cuda or x.element_size() != 4 or not x.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor of a 4-byte dtype")
    return x


def compress(x, chunk_elems=ZVC_DEFAULT_CHUNK_ELEMS, stream=None, out=None, ws=None,
             out_size=None):
    """Compress a contiguous 4-byte CUDA tensor. Returns (stream_bytes, size) where
    stream_bytes is a uint8 device buffer of the worst-case size and size a 1-element
    int64 device tensor holding the stream's byte count (read it after the stream syncs)."""
    torch = _torch()
    x = _words(x)
    n = x.numel()
    cap = zvc_size_bound(n, chunk_elems)
    if cap == 0:
        raise ZvcError(ZVC_ERR_INVALID_ARG, "zvc_size_bound")
    if out is None:
        out = torch.empty(cap, dtype=torch.uint8, device=x.device)
    if ws is None:
        ws = new_workspace(zvc_workspace_size(n, chunk_elems), x.device)
    if out_size is None:
        out_size = torch.zeros(1, dtype=torch.int64, device=x.device)
    _check(zvc_compress(x.data_ptr(), n, chunk_elems, out.data_ptr(), out.numel(),
                        out_size.data_ptr(), ws.data_ptr(), ws.numel(), _stream_handle(stream)),
           "zvc_compress")
    return out, out_size


def decompress(stream_bytes, in_bytes, n, chunk_elems=ZVC_DEFAULT_CHUNK_ELEMS, stream=None,
               out=None, ws=None, dtype=None):
    """Decompress in_bytes bytes of a uint8 CUDA buffer into n words (float32 unless
    dtype or out is given). Device-side corruption is latched in ws (see get_error)."""
    torch = _torch()
    if out is None:
        out = torch.empty(n, dtype=dtype or torch.float32, device=stream_bytes.device)
    if ws is None:
        ws = new_workspace(ZVC_WORKSPACE_ALIGN, stream_bytes.device)
    _check(zvc_decompress(stream_bytes.data_ptr(), int(in_bytes), out.data_ptr(), n, chunk_elems,
                          ws.data_ptr(), ws.numel(), _stream_handle(stream)), "zvc_decompress")
    return out


def get_error(ws, stream=None):
    return zvc_get_error(ws.data_ptr(), _stream_handle(stream))
