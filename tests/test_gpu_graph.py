"""Compress and decompress captured in a CUDA graph and replayed on new data.

Each compress launch tags its workspace entries (the tile aggregates of the decoupled
look-back, Rhu et al., "Compressing DMA Engine", section V.B: offsets from prefix sums)
with an epoch that it draws on the device, so a replayed launch never reads an entry
of an earlier replay: every replay must equal the oracle byte for byte.
"""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
from tests.gpu_util import ensure_lib, sh

pytestmark = pytest.mark.gpu


def _words(rng, n, d):
    w = rng.integers(1, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    w[rng.random(n) >= d] = 0
    return w


def _permute_in_windows(rng, w):
    """The same number of non-zero words in every window, in other places and values:
    the stream keeps its size, its bytes change."""
    n = w.size - w.size % 32
    v = w[:n].reshape(-1, 32).copy()
    idx = np.argsort(rng.random(v.shape), axis=1)
    v = np.take_along_axis(v, idx, axis=1)
    v[v != 0] = rng.integers(1, 2**32, size=int((v != 0).sum()), dtype=np.uint64).astype(np.uint32)
    out = w.copy()
    out[:n] = v.reshape(-1)
    return out


def test_compress_graph_replays_equal_the_oracle():
    ensure_lib()
    rng = np.random.default_rng(7)
    C, n = 4096, 3_000_017
    x = torch.zeros(n, dtype=torch.int32, device="cuda")
    cap = zvc.zvc_size_bound(n, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))

    def comp(stream):
        return zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), stream)

    assert comp(sh()) == zvc.ZVC_OK  # loads the kernel outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert comp(s.cuda_stream) == zvc.ZVC_OK
    for d in (0.5, 0.05, 0.9, 0.3, 0.0, 1.0):
        w = _words(rng, n, d)
        x.copy_(torch.from_numpy(w.view(np.int32)).cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode(w, C)
        S = int(size.item())
        assert S == ref.size, d
        assert np.array_equal(out[:S].cpu().numpy(), ref), d
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK


def test_compress_and_decompress_in_one_graph():
    ensure_lib()
    rng = np.random.default_rng(8)
    C, n = 1024, 1_500_001
    w = _words(rng, n, 0.4)
    x = torch.from_numpy(w.view(np.int32)).cuda()
    y = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    cap = zvc.zvc_size_bound(n, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
    dws = zvc.new_workspace(zvc.ZVC_WORKSPACE_ALIGN)
    assert zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                            ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    S = int(size.item())
    assert zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, dws.data_ptr(), dws.numel(),
                              sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert zvc.zvc_compress(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), s.cuda_stream) == zvc.ZVC_OK
        assert zvc.zvc_decompress(out.data_ptr(), S, y.data_ptr(), n, C, dws.data_ptr(),
                                  dws.numel(), s.cuda_stream) == zvc.ZVC_OK
    for _ in range(4):
        w = _permute_in_windows(rng, w)
        x.copy_(torch.from_numpy(w.view(np.int32)).cuda())
        y.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode(w, C)
        assert int(size.item()) == S == ref.size
        assert np.array_equal(out[:S].cpu().numpy(), ref)
        assert torch.equal(y, x)
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(dws.data_ptr(), sh()) == zvc.ZVC_OK


def test_batched_compress_graph_replays_equal_the_oracle():
    ensure_lib()
    rng = np.random.default_rng(9)
    C = 4096
    ns = [70_001, 1_000_000, 4_097, 2_500_000]
    xs = [torch.zeros(k, dtype=torch.int32, device="cuda") for k in ns]
    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_batch_workspace_size(ns, C))
    ptrs = [x.data_ptr() for x in xs]

    def comp(stream):
        return zvc.zvc_compress_batched(ptrs, ns, C, out.data_ptr(), cap, size.data_ptr(),
                                        ws.data_ptr(), ws.numel(), stream)

    assert comp(sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert comp(s.cuda_stream) == zvc.ZVC_OK
    for d in (0.3, 0.7, 0.02):
        ws_ = [_words(rng, k, d) for k in ns]
        for x, w in zip(xs, ws_):
            x.copy_(torch.from_numpy(w.view(np.int32)).cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode_batch(ws_, C)
        S = int(size.item())
        assert S == ref.size and np.array_equal(out[:S].cpu().numpy(), ref), d
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK


def test_compress16_graph_replays_equal_the_oracle():
    ensure_lib()
    rng = np.random.default_rng(10)
    C, n = 1024, 1_000_003
    x = torch.zeros(n, dtype=torch.int16, device="cuda")
    cap = zvc.zvc_size_bound16(n, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))

    def comp(stream):
        return zvc.zvc_compress16(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                  ws.data_ptr(), ws.numel(), stream)

    assert comp(sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert comp(s.cuda_stream) == zvc.ZVC_OK
    for d in (0.4, 0.02, 1.0):
        w = rng.integers(1, 2**16, size=n, dtype=np.uint32).astype(np.uint16)
        w[rng.random(n) >= d] = 0
        x.copy_(torch.from_numpy(w.view(np.int16)).cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode16(w, C)
        S = int(size.item())
        assert S == ref.size and np.array_equal(out[:S].cpu().numpy(), ref), d
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK


def test_static_compress_graph_replays_equal_the_oracle():
    """zvc_compress_static captured and replayed: its epoch counter lives in the library's
    static scratch, and every replay still equals the oracle."""
    ensure_lib()
    rng = np.random.default_rng(11)
    C, n = 4096, 900_001
    x = torch.zeros(n, dtype=torch.int32, device="cuda")
    cap = zvc.zvc_size_bound(n, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")

    def comp(stream):
        return zvc.zvc_compress_static(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                       stream)

    assert comp(sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert comp(s.cuda_stream) == zvc.ZVC_OK
    for d in (0.25, 0.75):
        w = _words(rng, n, d)
        x.copy_(torch.from_numpy(w.view(np.int32)).cuda())
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode(w, C)
        S = int(size.item())
        assert S == ref.size and np.array_equal(out[:S].cpu().numpy(), ref), d
    assert zvc.zvc_compress_static_get_error(sh()) == zvc.ZVC_OK


def test_batched_and_16bit_decompress_graph_replays_restore_the_input():
    """Batched and 16-bit decompress captured and replayed on streams of new data of the same
    size (the words moved within their windows): every replay restores its input."""
    ensure_lib()
    rng = np.random.default_rng(12)
    C = 4096
    ns = [300_017, 65_536, 1_000_000]
    ws_ = [_words(rng, k, 0.35) for k in ns]
    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ws = zvc.new_workspace(zvc.ZVC_WORKSPACE_ALIGN)
    ys = [torch.full((k,), -1, dtype=torch.int32, device="cuda") for k in ns]
    ref = oracle.encode_batch(ws_, C)
    out[:ref.size].copy_(torch.from_numpy(ref).cuda())
    S = ref.size

    def dec(stream):
        return zvc.zvc_decompress_batched(out.data_ptr(), S, [y.data_ptr() for y in ys], ns, C,
                                          ws.data_ptr(), ws.numel(), stream)

    assert dec(sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert dec(s.cuda_stream) == zvc.ZVC_OK
    for _ in range(3):
        ws_ = [_permute_in_windows(rng, w) for w in ws_]
        ref = oracle.encode_batch(ws_, C)
        assert ref.size == S
        out[:S].copy_(torch.from_numpy(ref).cuda())
        g.replay()
        torch.cuda.synchronize()
        for w, y in zip(ws_, ys):
            assert np.array_equal(y.cpu().numpy().view(np.uint32), w)
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK

    # 16-bit: the same, one stream
    n = 777_777
    w16 = rng.integers(1, 2**16, size=n, dtype=np.uint32).astype(np.uint16)
    w16[rng.random(n) >= 0.4] = 0
    ref16 = oracle.encode16(w16, C)
    S16 = ref16.size
    out16 = torch.from_numpy(ref16).cuda()
    y16 = torch.full((n,), -1, dtype=torch.int16, device="cuda")

    def dec16(stream):
        return zvc.zvc_decompress16(out16.data_ptr(), S16, y16.data_ptr(), n, C, ws.data_ptr(),
                                    ws.numel(), stream)

    assert dec16(sh()) == zvc.ZVC_OK
    torch.cuda.synchronize()
    g16 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g16, stream=s):
        assert dec16(s.cuda_stream) == zvc.ZVC_OK
    for _ in range(3):
        m = n - n % 32
        v = w16[:m].reshape(-1, 32)
        v = np.take_along_axis(v, np.argsort(rng.random(v.shape), axis=1), axis=1)
        w16 = np.concatenate([v.reshape(-1), w16[m:]])
        ref16 = oracle.encode16(w16, C)
        assert ref16.size == S16
        out16.copy_(torch.from_numpy(ref16).cuda())
        g16.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y16.cpu().numpy().view(np.uint16), w16)
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
