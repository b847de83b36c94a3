"""Seeded random combinations, each checked in full against the oracle.

Rhu et al., "Compressing DMA Engine", section V.A: every GPU stream must equal the oracle's
bytes, and decompression must restore every word. Each case draws the number of tensors
(1: a single stream; 2-6: one batched call, empty tensors among them), the chunk size, every
tensor's length (log-uniform up to 300,000 words, so ragged tiles, windows and chunks are
the rule) and its zero structure (i.i.d. at a random density, or blocks of non-zero words
at a random block size), so that the launch paths meet in combinations no hand-written
case lists.
"""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
from tests.gpu_util import ensure_lib, sh

pytestmark = pytest.mark.gpu

CHUNKS = [32, 64, 96, 128, 512, 1024, 2048, 4096, 8192, 32768]


def _tensor(rng, n):
    w = rng.integers(1, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    if rng.random() < 0.5:  # i.i.d.
        w[rng.random(n) >= rng.random()] = 0
    else:  # blocks of non-zero words in a zero map
        blk = int(rng.choice([1, 7, 32, 100, 1024, 5000]))
        keep = np.repeat(rng.random(n // blk + 1) < rng.random(), blk)[:n]
        w[~keep] = 0
    return w


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    T = 1 if rng.random() < 0.5 else int(rng.integers(2, 7))
    C = int(rng.choice(CHUNKS))
    ns = []
    for _ in range(T):
        n = 0 if (T > 1 and rng.random() < 0.15) else int(np.exp(rng.uniform(0, np.log(300_000))))
        ns.append(n)
    return rng, T, C, ns


@pytest.mark.parametrize("seed", range(60))
def test_random_case_equals_the_oracle(seed):
    ensure_lib()
    rng, T, C, ns = _case(seed)
    words = [_tensor(rng, n) for n in ns]
    xs = [torch.from_numpy(w.view(np.int32)).cuda() if w.size else
          torch.empty(0, dtype=torch.int32, device="cuda") for w in words]
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    if T == 1:
        n = ns[0]
        cap = zvc.zvc_size_bound(n, C)
        ws = zvc.new_workspace(max(zvc.zvc_workspace_size(n, C), zvc.ZVC_WORKSPACE_ALIGN))
        out = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device="cuda")
        assert zvc.zvc_compress(xs[0].data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
        ref = oracle.encode(words[0], C)
    else:
        cap = zvc.zvc_batch_size_bound(ns, C)
        ws = zvc.new_workspace(max(zvc.zvc_batch_workspace_size(ns, C), zvc.ZVC_WORKSPACE_ALIGN))
        out = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device="cuda")
        assert zvc.zvc_compress_batched([x.data_ptr() for x in xs], ns, C, out.data_ptr(), cap,
                                        size.data_ptr(), ws.data_ptr(), ws.numel(),
                                        sh()) == zvc.ZVC_OK
        ref = oracle.encode_batch(words, C)
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    S = int(size.item())
    host = out.cpu().numpy()
    assert S == ref.size, (seed, T, C, ns)
    assert np.array_equal(host[:S], ref), (seed, T, C, ns)
    assert (host[S:] == 0xEE).all()  # nothing written past the stream

    ys = [torch.full((n,), -1, dtype=torch.int32, device="cuda") for n in ns]
    if T == 1:
        st = zvc.zvc_decompress(out.data_ptr(), S, ys[0].data_ptr(), ns[0], C, ws.data_ptr(),
                                ws.numel(), sh())
    else:
        st = zvc.zvc_decompress_batched(out.data_ptr(), S, [y.data_ptr() for y in ys], ns, C,
                                        ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    for x, y in zip(xs, ys):
        assert torch.equal(x, y), (seed, T, C, ns)


@pytest.mark.parametrize("seed", range(30))
def test_random_16bit_case_equals_the_oracle(seed):
    """The same draws for the 16-bit calls (single streams)."""
    ensure_lib()
    rng = np.random.default_rng(5000 + seed)
    C = int(rng.choice(CHUNKS))
    n = int(np.exp(rng.uniform(0, np.log(300_000))))
    w = rng.integers(1, 2**16, size=n, dtype=np.uint32).astype(np.uint16)
    if rng.random() < 0.5:
        w[rng.random(n) >= rng.random()] = 0
    else:
        blk = int(rng.choice([1, 7, 32, 100, 1024, 5000]))
        keep = np.repeat(rng.random(n // blk + 1) < rng.random(), blk)[:n]
        w[~keep] = 0
    x = torch.from_numpy(w.view(np.int16)).cuda()
    cap = zvc.zvc_size_bound16(n, C)
    out = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
    assert zvc.zvc_compress16(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                              ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    ref = oracle.encode16(w, C)
    S = int(size.item())
    host = out.cpu().numpy()
    assert S == ref.size and np.array_equal(host[:S], ref), (seed, C, n)
    assert (host[S:] == 0xEE).all()
    y = torch.full((n,), -1, dtype=torch.int16, device="cuda")
    assert zvc.zvc_decompress16(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(),
                                sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert torch.equal(x, y), (seed, C, n)
