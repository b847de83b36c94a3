"""Corrupt input and device-side waits, on the GPU, without faulting it: every failure is
made on the host (bytes flipped in a valid stream, wrong sizes) or by a wait on a flag
that nothing sets; the kernels report through the latched error word and the context
stays usable afterwards."""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
from tests.gpu_util import ensure_lib, gpu_compress, gpu_decompress, sh

pytestmark = pytest.mark.gpu


def _rand(rng, n, d):
    w = rng.integers(1, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    w[rng.random(n) >= d] = 0
    return w


def _gpu_status(stream, n, C):
    st, err, words = gpu_decompress(stream, n, C)
    return (st if st != zvc.ZVC_OK else err), words


def test_random_corruption_agrees_with_oracle():
    ensure_lib()
    rng = np.random.default_rng(21)
    seen = {zvc.ZVC_OK: 0, zvc.ZVC_ERR_CORRUPT: 0}
    for trial in range(400):
        n = int(rng.integers(1, 20_000))
        C = int(rng.choice([32, 64, 1024, 4096]))
        w = _rand(rng, n, float(rng.random()))
        s = oracle.encode(w, C)
        t = s.copy()
        for _ in range(int(rng.integers(1, 4))):
            i = int(rng.integers(0, t.size))
            t[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, owords = oracle.decode(t, n, C)
        gst, gwords = _gpu_status(t, n, C)
        if ost == oracle.OK:
            assert gst == zvc.ZVC_OK and np.array_equal(gwords, owords), trial
        else:
            assert gst == zvc.ZVC_ERR_CORRUPT, (trial, ost, gst)
        seen[gst] += 1
    assert seen[zvc.ZVC_ERR_CORRUPT] > 50 and seen[zvc.ZVC_OK] > 10


def test_corrupt_chunks_staged_in_pieces_agree_with_oracle():
    """Flipped bits in dense chunks among empty ones, whose decompression is staged in
    several pieces (the CTA buffer is sized from the mean chunk): the status and, when the
    stream still decodes, the words must be the oracle's."""
    ensure_lib()
    rng = np.random.default_rng(25)
    C = 4096
    seen = {zvc.ZVC_OK: 0, zvc.ZVC_ERR_CORRUPT: 0}
    for trial in range(120):
        dens = [0.0] * 10 + [1.0, float(rng.random()), 1.0] + [0.0] * 10
        w = np.concatenate([_rand(rng, C, d) for d in dens])
        n = w.size - int(rng.integers(0, 100))
        w = w[:n]
        s = oracle.encode(w, C)
        table_end = 32 + 8 * (-(-n // C))
        starts = np.frombuffer(s[32:table_end].tobytes(), "<u8").astype(np.int64)
        lo, hi = table_end + int(starts[10]), table_end + int(starts[13])  # the dense chunks
        t = s.copy()
        for _ in range(int(rng.integers(1, 3))):
            if rng.random() < 0.5:  # a mask of chunk 10 or 12 (all windows full: 33 words)
                c = int(rng.choice([10, 12]))
                i = table_end + int(starts[c]) + 4 * 33 * int(rng.integers(0, C // 32))
                i += int(rng.integers(0, 4))
            else:
                i = int(rng.integers(lo, hi))
            t[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, owords = oracle.decode(t, n, C)
        gst, gwords = _gpu_status(t, n, C)
        if ost == oracle.OK:
            assert gst == zvc.ZVC_OK and np.array_equal(gwords, owords), trial
        else:
            assert gst == zvc.ZVC_ERR_CORRUPT, (trial, ost, gst)
        seen[gst] += 1
    assert seen[zvc.ZVC_ERR_CORRUPT] > 20 and seen[zvc.ZVC_OK] > 5, seen


def test_corrupt_short_chunks_agree_with_oracle():
    """Flipped bits in a stream of 8192 sparse chunks, decompressed by CTAs that hold several
    chunks each (one warp walking them all): status and words must be the oracle's."""
    ensure_lib()
    rng = np.random.default_rng(26)
    C = 4096
    n = 8192 * C
    w = _rand(rng, n, 0.03)
    s = oracle.encode(w, C)
    table_end = 32 + 8 * (n // C)
    seen = {zvc.ZVC_OK: 0, zvc.ZVC_ERR_CORRUPT: 0}
    for trial in range(8):
        t = s.copy()
        for _ in range(int(rng.integers(1, 4))):
            i = int(rng.integers(table_end, t.size))
            t[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, owords = oracle.decode(t, n, C)
        gst, gwords = _gpu_status(t, n, C)
        if ost == oracle.OK:
            assert gst == zvc.ZVC_OK and np.array_equal(gwords, owords), trial
        else:
            assert gst == zvc.ZVC_ERR_CORRUPT, (trial, ost, gst)
        seen[gst] += 1
    assert seen[zvc.ZVC_ERR_CORRUPT] >= 3, seen


def test_size_and_parameter_mismatches():
    rng = np.random.default_rng(22)
    w = _rand(rng, 50_000, 0.4)
    s = oracle.encode(w, 4096)
    assert _gpu_status(s[:-4], w.size, 4096)[0] == zvc.ZVC_ERR_CORRUPT
    assert _gpu_status(np.concatenate([s, s[-4:]]), w.size, 4096)[0] == zvc.ZVC_ERR_CORRUPT
    assert _gpu_status(s, w.size - 1, 4096)[0] == zvc.ZVC_ERR_CORRUPT
    assert _gpu_status(s, w.size, 1024)[0] == zvc.ZVC_ERR_CORRUPT
    tail = oracle.encode(np.array([0, 0, 7], np.uint32), 32)
    bad = tail.copy()
    bad[40] |= 0x08  # mask bit 3 names element 3 of a 3-element tensor
    assert oracle.decode(bad, 3, 32)[0] == oracle.ERR_CORRUPT
    assert _gpu_status(bad, 3, 32)[0] == zvc.ZVC_ERR_CORRUPT


def test_error_latches_until_read_and_context_survives():
    ensure_lib()
    rng = np.random.default_rng(23)
    w = _rand(rng, 10_000, 0.5)
    s = oracle.encode(w, 1024)
    bad = s.copy()
    bad[32 + 8 * 10] ^= 0x01
    ws = zvc.new_workspace(256)
    out = torch.empty(w.size, dtype=torch.int32, device="cuda")
    for stream_bytes in (bad, s):  # corrupt first, then a good stream
        d = torch.from_numpy(stream_bytes).cuda()
        assert zvc.zvc_decompress(d.data_ptr(), d.numel(), out.data_ptr(), w.size, 1024,
                                  ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_ERR_CORRUPT
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    st, back, err = gpu_compress(torch.from_numpy(w.view(np.int32)).cuda(), 1024)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK and np.array_equal(back, s)


def test_wait_limit_gives_up_and_reports():
    ensure_lib()
    ws = zvc.new_workspace(4096)
    st = zvc.zvc_selftest_wait_timeout(ws.data_ptr(), ws.numel(), 20_000_000, sh())  # 20 ms
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_ERR_TIMEOUT
    # the device is still usable
    x = torch.arange(1, 100_001, dtype=torch.int32, device="cuda")
    st, got, err = gpu_compress(x, 4096)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert np.array_equal(got, oracle.encode(x.cpu().numpy(), 4096))


def test_batched_corruption():
    ensure_lib()
    rng = np.random.default_rng(24)
    ws_ = [_rand(rng, n, 0.5) for n in (1000, 0, 5000)]
    b = oracle.encode_batch(ws_, 1024)
    last = int(np.frombuffer(b[32:40].tobytes(), "<u8")[0])  # tensor_off[2]
    # batch magic, T, total, tensor_off[0], tensor_off[1], stream 0 magic, stream 2 n
    for off, bit in ((0, 0), (4, 1), (8, 0), (16, 2), (24, 3), (40, 4), (last + 16, 0)):
        t = b.copy()
        t[off] ^= np.uint8(1 << bit)
        assert oracle.decode_batch(t, [1000, 0, 5000], 1024)[0] == oracle.ERR_CORRUPT
        d = torch.from_numpy(t).cuda()
        outs = [torch.empty(max(w.size, 1), dtype=torch.int32, device="cuda") for w in ws_]
        ws = zvc.new_workspace(256)
        st = zvc.zvc_decompress_batched(d.data_ptr(), d.numel(), [o.data_ptr() for o in outs],
                                        [1000, 0, 5000], 1024, ws.data_ptr(), ws.numel(), sh())
        if st == zvc.ZVC_OK:
            st = zvc.zvc_get_error(ws.data_ptr(), sh())
        assert st == zvc.ZVC_ERR_CORRUPT, off
