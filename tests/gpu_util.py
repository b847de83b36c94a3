"""Helpers for the GPU tests: run the library through its C ABI on device buffers and
bring results back to the host for comparison with the oracle."""
import struct

import numpy as np
import torch

import activation_sparsity_compression_gb300 as zvc
from activation_sparsity_compression_gb300 import build as zbuild

import oracle

_built = False


def ensure_lib():
    global _built
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if not _built:
        zbuild.build()
        zvc.lib()
        _built = True


def sh():
    return torch.cuda.current_stream().cuda_stream


def words_of(x: torch.Tensor) -> np.ndarray:
    return x.detach().contiguous().view(-1).view(torch.int32).cpu().numpy().view(np.uint32)


def gpu_compress(x: torch.Tensor, chunk_elems: int, out_pad_bytes: int = 0, ws=None):
    """Compress through zvc_compress. out_pad_bytes shifts the destination by that many
    bytes inside a larger buffer (to exercise unaligned destinations). Returns
    (status, stream bytes as numpy uint8, latched error)."""
    ensure_lib()
    n = x.numel()
    cap = zvc.zvc_size_bound(n, chunk_elems)
    buf = torch.full((cap + out_pad_bytes + 64,), 0xEE, dtype=torch.uint8, device=x.device)
    size = torch.zeros(1, dtype=torch.int64, device=x.device)
    if ws is None:
        ws = zvc.new_workspace(zvc.zvc_workspace_size(n, chunk_elems), x.device)
    st = zvc.zvc_compress(x.data_ptr(), n, chunk_elems, buf.data_ptr() + out_pad_bytes, cap,
                          size.data_ptr(), ws.data_ptr(), ws.numel(), sh())
    if st != zvc.ZVC_OK:
        return st, None, None
    err = zvc.zvc_get_error(ws.data_ptr(), sh())
    s = int(size.item())
    host = buf.cpu().numpy()
    # nothing outside [pad, pad + s) may be written
    assert (host[:out_pad_bytes] == 0xEE).all()
    assert (host[out_pad_bytes + s:] == 0xEE).all()
    return st, host[out_pad_bytes:out_pad_bytes + s].copy(), err


def gpu_decompress(stream_bytes: np.ndarray, n: int, chunk_elems: int, device="cuda",
                   out_offset_words: int = 0):
    """Decompress host stream bytes through zvc_decompress. Returns (status, latched
    error, words as numpy uint32)."""
    ensure_lib()
    d_in = torch.from_numpy(np.array(stream_bytes, dtype=np.uint8, copy=True)).to(device)
    out = torch.full((n + out_offset_words + 16,), -1, dtype=torch.int32, device=device)
    ws = zvc.new_workspace(zvc.ZVC_WORKSPACE_ALIGN, device)
    st = zvc.zvc_decompress(d_in.data_ptr(), d_in.numel(), out.data_ptr() + 4 * out_offset_words,
                            n, chunk_elems, ws.data_ptr(), ws.numel(), sh())
    err = zvc.zvc_get_error(ws.data_ptr(), sh()) if st == zvc.ZVC_OK else None
    host = out.cpu().numpy().view(np.uint32)
    if err == zvc.ZVC_OK:
        # nothing outside the output range may be written
        assert (host[:out_offset_words] == 0xFFFFFFFF).all()
        assert (host[out_offset_words + n:] == 0xFFFFFFFF).all()
    return st, err, host[out_offset_words:out_offset_words + n].copy()


def chunk_table(stream: np.ndarray, n: int, chunk_elems: int) -> np.ndarray:
    nc = -(-n // chunk_elems)
    return np.frombuffer(stream[32:32 + 8 * nc].tobytes(), dtype="<u8").astype(np.int64)


def check_stream_by_samples(stream: np.ndarray, words: np.ndarray, chunk_elems: int,
                            samples: int, seed: int = 0):
    """Checks a full-size stream without encoding all of it on the CPU: the header, the
    closed-form size, the chunk table against per-chunk sizes counted with numpy, and the
    bytes of `samples` chunks (plus the first and last) against the oracle encoding each
    sampled chunk on its own."""
    n = words.size
    C = chunk_elems
    nc = -(-n // C)
    nnz = int(np.count_nonzero(words))
    assert stream.size == 32 + 8 * nc + 4 * (-(-n // 32)) + 4 * nnz
    hdr = stream[:32].tobytes()
    assert hdr[:16] == struct.pack("<IHHII", 0x3143565A, 1, 4, 32, C)
    assert int.from_bytes(hdr[16:24], "little") == n
    payload_start = 32 + 8 * nc
    assert int.from_bytes(hdr[24:32], "little") == stream.size - payload_start
    offs = chunk_table(stream, n, C)
    full = (n // C) * C
    per = np.count_nonzero(words[:full].reshape(-1, C), axis=1).astype(np.int64) * 4 + 4 * (C // 32)
    if full < n:
        tail = words[full:]
        per = np.append(per, 4 * (-(-tail.size // 32)) + 4 * int(np.count_nonzero(tail)))
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(per)[:-1]]))
    rng = np.random.default_rng(seed)
    picks = set(rng.integers(0, nc, size=min(samples, nc)).tolist()) | {0, nc - 1}
    ends = np.append(offs[1:], stream.size - payload_start)
    for c in sorted(picks):
        ref = oracle.encode(words[c * C:(c + 1) * C], C)
        body = ref[32 + 8:]
        got = stream[payload_start + offs[c]:payload_start + ends[c]]
        assert got.tobytes() == body.tobytes(), f"chunk {c}"
