"""ZVC on 16-bit words (bf16 / fp16) on the GPU, checked against the 16-bit oracle.

The rule of Rhu et al., "Compressing DMA Engine", section V.A (32 values, a 32-bit mask,
the non-zero values) on 2-byte words: GPU streams must equal the oracle's byte for byte,
decompression must restore every word bit for bit (and decode the oracle's streams), and a
corrupt stream must get the oracle's verdict. Windows sit on 2-byte boundaries, so the
cases cover every chunk size class, ragged tails, unaligned bases and pieces.
"""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests.gpu_util import ensure_lib, sh

pytestmark = pytest.mark.gpu


def rand16(rng, n, d):
    w = rng.integers(1, 2**16, size=n, dtype=np.uint32).astype(np.uint16)
    w[rng.random(n) >= d] = 0
    if n > 3:  # -0.0, a NaN and a denormal: non-zero bit patterns
        w[n // 3], w[n // 2], w[n - 1] = 0x8000, 0x7FC0, 0x0001
    return w


def compress16(words, C, in_off=0, out_off=0):
    """GPU compress of host uint16 words; in_off / out_off shift the device input (in
    2-byte units) and the output (in bytes, a multiple of 4) inside larger buffers.
    Returns the stream bytes; checks that nothing outside the stream was written."""
    ensure_lib()
    n = words.size
    x = torch.zeros(n + in_off + 8, dtype=torch.int16, device="cuda")
    if n:
        x[in_off:in_off + n] = torch.from_numpy(words.view(np.int16)).cuda()
    cap = zvc.zvc_size_bound16(n, C)
    out = torch.full((cap + out_off + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
    st = zvc.zvc_compress16(x.data_ptr() + 2 * in_off, n, C, out.data_ptr() + out_off, cap,
                            size.data_ptr(), ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    s = int(size.item())
    host = out.cpu().numpy()
    assert (host[:out_off] == 0xEE).all() and (host[out_off + s:] == 0xEE).all()
    return host[out_off:out_off + s].copy()


def decompress16(stream, n, C, out_off=0):
    """GPU decompress of host stream bytes into n uint16 words (out_off units into a larger
    buffer). Returns (status or latched error, words)."""
    ensure_lib()
    d_in = torch.from_numpy(np.array(stream, dtype=np.uint8, copy=True)).cuda()
    y = torch.full((n + out_off + 16,), -1, dtype=torch.int16, device="cuda")
    ws = zvc.new_workspace(zvc.ZVC_WORKSPACE_ALIGN)
    st = zvc.zvc_decompress16(d_in.data_ptr(), d_in.numel(), y.data_ptr() + 2 * out_off, n, C,
                              ws.data_ptr(), ws.numel(), sh())
    if st != zvc.ZVC_OK:
        return st, None
    err = zvc.zvc_get_error(ws.data_ptr(), sh())
    host = y.cpu().numpy().view(np.uint16)
    if err == zvc.ZVC_OK:  # nothing outside the output range is written
        assert (host[:out_off] == 0xFFFF).all() and (host[out_off + n:] == 0xFFFF).all()
    return err, host[out_off:out_off + n].copy()


@pytest.mark.parametrize("C", [32, 96, 1024, 4096, 32768])
@pytest.mark.parametrize("n", [0, 1, 31, 33, 4095, 4097, 100_003])
def test_odd_sizes_equal_the_oracle(n, C):
    rng = np.random.default_rng(n * 7 + C)
    for d in (0.0, 0.3, 1.0):
        w = rand16(rng, n, d)
        ref = oracle.encode16(w, C)
        got = compress16(w, C)
        assert np.array_equal(got, ref), (n, C, d)
        err, back = decompress16(ref, n, C)
        assert err == zvc.ZVC_OK and np.array_equal(back, w), (n, C, d)


@pytest.mark.parametrize("in_off,out_off", [(1, 4), (3, 8), (7, 12), (0, 0)])
def test_unaligned_bases(in_off, out_off):
    rng = np.random.default_rng(in_off)
    for C in (64, 4096):
        w = rand16(rng, 300_001, 0.45)
        ref = oracle.encode16(w, C)
        assert np.array_equal(compress16(w, C, in_off=in_off, out_off=out_off), ref)
        err, back = decompress16(ref, w.size, C, out_off=in_off)
        assert err == zvc.ZVC_OK and np.array_equal(back, w)


@pytest.mark.parametrize("density", [0.0, 0.05, 0.35, 0.6, 1.0])
def test_bf16_relu_activation_full_bytes(density):
    """A bf16 ReLU map of GoogLeNet's 56x56 stage at batch 64 (12.8 M words), every byte."""
    ensure_lib()
    g = torch.Generator(device="cuda").manual_seed(int(density * 100) + 16)
    thr = 0.0 if density in (0.0, 1.0) else float(torch.distributions.Normal(0, 1).icdf(
        torch.tensor(1.0 - density)))
    x = torch.randn((64, 64, 56, 56), generator=g, device="cuda")
    if density == 0.0:
        x = torch.zeros_like(x)
    elif density == 1.0:
        x = x.abs() + 1.0
    else:
        x = torch.relu(x - thr)
    xb = x.to(torch.bfloat16).contiguous()
    w = xb.view(torch.int16).cpu().numpy().view(np.uint16).reshape(-1)
    C = 4096
    ref = oracle.encode16(w, C)
    n = w.size
    cap = zvc.zvc_size_bound16(n, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, C))
    assert zvc.zvc_compress16(xb.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(),
                              ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    S = int(size.item())
    assert np.array_equal(out[:S].cpu().numpy(), ref)
    y = torch.empty_like(xb)
    assert zvc.zvc_decompress16(out.data_ptr(), S, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(),
                                sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert torch.equal(y.view(torch.int16), xb.view(torch.int16))


def test_dense_chunks_among_empty_ones_are_staged_in_pieces():
    """The decompress buffer is sized from the mean chunk: dense chunks among empty ones
    are staged in several pieces, from unaligned (2 mod 4) chunk starts."""
    rng = np.random.default_rng(9)
    C = 4096
    parts = []
    for k in range(64):
        d = 1.0 if k % 16 == 5 else 0.0
        parts.append(rand16(rng, C if k != 63 else C - 37, d))
    w = np.concatenate(parts)
    w[7] = 0x0101  # chunk 0 holds one value: every later chunk starts 2 mod 4
    ref = oracle.encode16(w, C)
    assert np.array_equal(compress16(w, C), ref)
    err, back = decompress16(ref, w.size, C)
    assert err == zvc.ZVC_OK and np.array_equal(back, w)


def test_random_corruption_agrees_with_oracle():
    ensure_lib()
    rng = np.random.default_rng(61)
    seen = {zvc.ZVC_OK: 0, zvc.ZVC_ERR_CORRUPT: 0}
    for trial in range(300):
        n = int(rng.integers(1, 20_000))
        C = int(rng.choice([32, 64, 1024, 4096]))
        w = rand16(rng, n, float(rng.random()))
        s = oracle.encode16(w, C)
        t = s.copy()
        for _ in range(int(rng.integers(1, 4))):
            i = int(rng.integers(0, t.size))
            t[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, owords = oracle.decode16(t, n, C)
        gst, gwords = decompress16(t, n, C)
        if ost == oracle.OK:
            assert gst == zvc.ZVC_OK and np.array_equal(gwords, owords), trial
        else:
            assert gst == zvc.ZVC_ERR_CORRUPT, (trial, ost, gst)
        seen[gst] += 1
    assert seen[zvc.ZVC_ERR_CORRUPT] > 50 and seen[zvc.ZVC_OK] > 10


def test_a_32_bit_stream_is_not_a_16_bit_stream():
    ensure_lib()
    w = np.arange(1, 5000, dtype=np.uint32)
    s32 = oracle.encode(w, 4096)
    # sizes a 16-bit stream of 4999 words can have exclude the 32-bit stream's; pad it to a
    # size in range so that the header itself must be rejected on the device
    s16 = oracle.encode16(w.astype(np.uint16), 4096)
    t = np.zeros(s16.size, np.uint8)
    t[:32] = s32[:32]
    err, _ = decompress16(t, w.size, 4096)
    assert err == zvc.ZVC_ERR_CORRUPT
    assert decompress16(s32, w.size, 4096)[0] == zvc.ZVC_ERR_CORRUPT
