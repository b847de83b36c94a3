"""ZVC oracle: TEST INFRASTRUCTURE ONLY.

A plain single-threaded C restatement of zero-value compression (Rhu et al.,
"Compressing DMA Engine: Leveraging Activation Sparsity for Training Deep Neural
Networks", section V.A "Compression Algorithm"), compiled with gcc and loaded with
ctypes. The stream layout it writes is documented at the top of ``zvc_oracle.c``.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zvc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libzvc_oracle.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_BUFFER_TOO_SMALL = -2
ERR_CORRUPT = -3

_POISON = 0xA5A5A5A5
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library (plain -O2, no vector flags)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-Werror",
           *extra_flags, src, "-o", out + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _declare(lib):
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    lib.zvco_size_bound.restype = ctypes.c_uint64
    lib.zvco_size_bound.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
    lib.zvco_encode.restype = ctypes.c_int64
    lib.zvco_encode.argtypes = [u32p, ctypes.c_uint64, ctypes.c_uint32, u8p, ctypes.c_uint64]
    lib.zvco_decode.restype = ctypes.c_int
    lib.zvco_decode.argtypes = [u8p, ctypes.c_uint64, u32p, ctypes.c_uint64, ctypes.c_uint32]
    lib.zvco_batch_prefix_bytes.restype = ctypes.c_uint64
    lib.zvco_batch_prefix_bytes.argtypes = [ctypes.c_uint32]
    lib.zvco_encode_batch.restype = ctypes.c_int64
    lib.zvco_encode_batch.argtypes = [ctypes.c_uint32, ctypes.POINTER(u32p), u64p,
                                      ctypes.c_uint32, u8p, ctypes.c_uint64]
    lib.zvco_decode_batch.restype = ctypes.c_int
    lib.zvco_decode_batch.argtypes = [u8p, ctypes.c_uint64, ctypes.c_uint32, u64p,
                                      ctypes.c_uint32, ctypes.POINTER(u32p)]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library. ``path`` (or the environment
    variable ZVC_ORACLE_LIB) loads a specific build, e.g. a deliberately mutated copy
    in the mutation test."""
    global _lib
    path = path or os.environ.get("ZVC_ORACLE_LIB")
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if stale:
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _u32_words(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype.itemsize != 4:
        raise TypeError(f"ZVC works on 32-bit words, got {a.dtype}")
    return a.reshape(-1).view(np.uint32)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned {code}")
        self.code = code


def size_bound(n: int, chunk_elems: int, lib=None) -> int:
    lib = lib or load()
    return int(lib.zvco_size_bound(n, chunk_elems))


def encode(x, chunk_elems: int = 4096, lib=None) -> np.ndarray:
    """Encode a 4-byte-per-element array (any shape) into one ZVC stream (uint8)."""
    lib = lib or load()
    w = _u32_words(x)
    n = w.size
    cap = int(lib.zvco_size_bound(n, chunk_elems))
    if cap == 0:
        raise OracleError(ERR_INVALID_ARG)
    out = np.empty(cap, dtype=np.uint8)
    r = lib.zvco_encode(_ptr(w, ctypes.c_uint32), n, chunk_elems, _ptr(out, ctypes.c_uint8), cap)
    if r < 0:
        raise OracleError(int(r))
    return out[:r].copy()


def decode(stream, n: int, chunk_elems: int = 4096, lib=None):
    """Decode one stream. Returns (status, words) with words a uint32 array of n."""
    lib = lib or load()
    s = np.ascontiguousarray(stream, dtype=np.uint8).reshape(-1)
    y = np.full(max(n, 1), _POISON, dtype=np.uint32)  # every word must be written
    r = lib.zvco_decode(_ptr(s, ctypes.c_uint8), s.size, _ptr(y, ctypes.c_uint32), n, chunk_elems)
    return int(r), y[:n]


def encode_batch(xs, chunk_elems: int = 4096, lib=None) -> np.ndarray:
    """Encode a list of 4-byte arrays into one batch (uint8)."""
    lib = lib or load()
    ws = [_u32_words(x) for x in xs]
    T = len(ws)
    ns = np.array([w.size for w in ws], dtype=np.uint64)
    cap = int(lib.zvco_batch_prefix_bytes(T)) + sum(
        int(lib.zvco_size_bound(int(n), chunk_elems)) for n in ns)
    out = np.empty(cap, dtype=np.uint8)
    ptrs = (ctypes.POINTER(ctypes.c_uint32) * max(T, 1))(*[_ptr(w, ctypes.c_uint32) for w in ws])
    r = lib.zvco_encode_batch(T, ptrs, _ptr(ns, ctypes.c_uint64), chunk_elems,
                              _ptr(out, ctypes.c_uint8), cap)
    if r < 0:
        raise OracleError(int(r))
    return out[:r].copy()


def decode_batch(stream, ns, chunk_elems: int = 4096, lib=None):
    """Decode a batch. Returns (status, [uint32 arrays])."""
    lib = lib or load()
    s = np.ascontiguousarray(stream, dtype=np.uint8).reshape(-1)
    ns_a = np.array(list(ns), dtype=np.uint64)
    T = ns_a.size
    ys = [np.full(max(int(n), 1), _POISON, dtype=np.uint32) for n in ns_a]
    ptrs = (ctypes.POINTER(ctypes.c_uint32) * max(T, 1))(*[_ptr(y, ctypes.c_uint32) for y in ys])
    r = lib.zvco_decode_batch(_ptr(s, ctypes.c_uint8), s.size, T, _ptr(ns_a, ctypes.c_uint64),
                              chunk_elems, ptrs)
    return int(r), [y[:int(n)] for y, n in zip(ys, ns_a)]


# ------------------------------------------------------------------ RLE (comparison codec)
# Run-length encoding as the pages' layout-dependent comparison codec (section V.A and
# VII.A); the layout is documented at the top of ``rle_oracle.c``. A separate library, so
# that the ZVC oracle above stays exactly as pinned.
_RLE_SRC = os.path.join(_HERE, "rle_oracle.c")
_RLE_LIB_PATH = os.path.join(_BUILD_DIR, "librle_oracle.so")
_rle_lib = None


def build_all() -> None:
    """Compile every oracle library (ZVC on 32-bit words, ZVC on 16-bit words, RLE)."""
    build()
    build(_RLE_SRC, _RLE_LIB_PATH)
    build(_Z16_SRC, _Z16_LIB_PATH)


def rle_load(path: str | None = None):
    """Load (building first if needed) the RLE oracle library."""
    global _rle_lib

    def declare(lib):
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u32p = ctypes.POINTER(ctypes.c_uint32)
        lib.rleo_size_bound.restype = ctypes.c_uint64
        lib.rleo_size_bound.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        lib.rleo_encode.restype = ctypes.c_int64
        lib.rleo_encode.argtypes = [u32p, ctypes.c_uint64, ctypes.c_uint32, u8p, ctypes.c_uint64]
        lib.rleo_decode.restype = ctypes.c_int
        lib.rleo_decode.argtypes = [u8p, ctypes.c_uint64, u32p, ctypes.c_uint64, ctypes.c_uint32]
        return lib

    if path is not None:
        return declare(ctypes.CDLL(path))
    with _lock:
        if _rle_lib is None:
            stale = (not os.path.exists(_RLE_LIB_PATH)
                     or os.path.getmtime(_RLE_LIB_PATH) < os.path.getmtime(_RLE_SRC))
            if stale:
                build(_RLE_SRC, _RLE_LIB_PATH)
            _rle_lib = declare(ctypes.CDLL(_RLE_LIB_PATH))
    return _rle_lib


def rle_size_bound(n: int, window: int, lib=None) -> int:
    lib = lib or rle_load()
    return int(lib.rleo_size_bound(n, window))


def rle_encode(x, window: int = 1024, lib=None) -> np.ndarray:
    """RLE-encode a 4-byte-per-element array (any shape) into one stream (uint8)."""
    lib = lib or rle_load()
    w = _u32_words(x)
    n = w.size
    cap = int(lib.rleo_size_bound(n, window))
    if cap == 0:
        raise OracleError(ERR_INVALID_ARG)
    out = np.empty(cap, dtype=np.uint8)
    r = lib.rleo_encode(_ptr(w, ctypes.c_uint32), n, window, _ptr(out, ctypes.c_uint8), cap)
    if r < 0:
        raise OracleError(int(r))
    return out[:r].copy()


def rle_decode(stream, n: int, window: int = 1024, lib=None):
    """Decode one RLE stream. Returns (status, words) with words a uint32 array of n."""
    lib = lib or rle_load()
    s = np.ascontiguousarray(stream, dtype=np.uint8).reshape(-1)
    y = np.full(max(n, 1), _POISON, dtype=np.uint32)
    r = lib.rleo_decode(_ptr(s, ctypes.c_uint8), s.size, _ptr(y, ctypes.c_uint32), n, window)
    return int(r), y[:n]


# ------------------------------------------------------------------ ZVC on 16-bit words
# The same rule on bf16 / fp16 activation words (a 32-bit mask per 32 values, then the
# non-zero 2-byte values); the layout is documented at the top of ``zvc16_oracle.c``. A
# separate library, so that the 32-bit oracle above stays exactly as pinned.
_Z16_SRC = os.path.join(_HERE, "zvc16_oracle.c")
_Z16_LIB_PATH = os.path.join(_BUILD_DIR, "libzvc16_oracle.so")
_z16_lib = None


def z16_load(path: str | None = None):
    """Load (building first if needed) the 16-bit ZVC oracle library. ``path`` (or the
    environment variable ZVC16_ORACLE_LIB) loads a specific build, e.g. a mutant."""
    global _z16_lib

    def declare(lib):
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.zvco16_size_bound.restype = ctypes.c_uint64
        lib.zvco16_size_bound.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        lib.zvco16_encode.restype = ctypes.c_int64
        lib.zvco16_encode.argtypes = [u16p, ctypes.c_uint64, ctypes.c_uint32, u8p, ctypes.c_uint64]
        lib.zvco16_decode.restype = ctypes.c_int
        lib.zvco16_decode.argtypes = [u8p, ctypes.c_uint64, u16p, ctypes.c_uint64, ctypes.c_uint32]
        return lib

    path = path or os.environ.get("ZVC16_ORACLE_LIB")
    if path is not None:
        return declare(ctypes.CDLL(path))
    with _lock:
        if _z16_lib is None:
            stale = (not os.path.exists(_Z16_LIB_PATH)
                     or os.path.getmtime(_Z16_LIB_PATH) < os.path.getmtime(_Z16_SRC))
            if stale:
                build(_Z16_SRC, _Z16_LIB_PATH)
            _z16_lib = declare(ctypes.CDLL(_Z16_LIB_PATH))
    return _z16_lib


def _u16_words(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype.itemsize != 2:
        raise TypeError(f"16-bit ZVC works on 16-bit words, got {a.dtype}")
    return a.reshape(-1).view(np.uint16)


def size_bound16(n: int, chunk_elems: int, lib=None) -> int:
    lib = lib or z16_load()
    return int(lib.zvco16_size_bound(n, chunk_elems))


def encode16(x, chunk_elems: int = 4096, lib=None) -> np.ndarray:
    """Encode a 2-byte-per-element array (any shape) into one 16-bit ZVC stream (uint8)."""
    lib = lib or z16_load()
    w = _u16_words(x)
    n = w.size
    cap = int(lib.zvco16_size_bound(n, chunk_elems))
    if cap == 0:
        raise OracleError(ERR_INVALID_ARG)
    out = np.empty(cap, dtype=np.uint8)
    r = lib.zvco16_encode(_ptr(w, ctypes.c_uint16), n, chunk_elems, _ptr(out, ctypes.c_uint8), cap)
    if r < 0:
        raise OracleError(int(r))
    return out[:r].copy()


def decode16(stream, n: int, chunk_elems: int = 4096, lib=None):
    """Decode one 16-bit stream. Returns (status, words) with words a uint16 array of n."""
    lib = lib or z16_load()
    s = np.ascontiguousarray(stream, dtype=np.uint8).reshape(-1)
    y = np.full(max(n, 1), 0xA5A5, dtype=np.uint16)  # every word must be written
    r = lib.zvco16_decode(_ptr(s, ctypes.c_uint8), s.size, _ptr(y, ctypes.c_uint16), n,
                          chunk_elems)
    return int(r), y[:n]
