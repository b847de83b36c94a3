"""RLE, the comparison codec (Rhu et al., "Compressing DMA Engine", section V.A: RLE exploits
runs of zeros and non-zeros; section VII.A: its ratio depends on the activation layout,
ZVC's does not): the GPU stream must equal the RLE oracle's byte for byte and decode back
bit for bit; corrupt streams must get the oracle's verdict."""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests import golden_io
from tests.gpu_util import ensure_lib, sh, words_of

pytestmark = pytest.mark.gpu


def gpu_rle(words, window):
    ensure_lib()
    x = torch.as_tensor(np.asarray(words, dtype=np.uint32).view(np.int32)).cuda()
    n = x.numel()
    cap = zvc.zvc_rle_size_bound(n, window)
    out = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_rle_workspace_size(n, window))
    st = zvc.zvc_rle_compress(x.data_ptr(), n, window, out.data_ptr(), cap, size.data_ptr(),
                              ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    s = int(size.item())
    host = out.cpu().numpy()
    assert (host[s:] == 0xEE).all()  # nothing written past the stream
    return host[:s]


def gpu_unrle(stream, n, window):
    """Returns (status, words): status is the call's, else the latched one."""
    ensure_lib()
    d = torch.as_tensor(np.array(stream, dtype=np.uint8, copy=True)).cuda()
    y = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
    ws = zvc.new_workspace(256)
    st = zvc.zvc_rle_decompress(d.data_ptr(), d.numel(), y.data_ptr(), n, window, ws.data_ptr(),
                                ws.numel(), sh())
    if st == zvc.ZVC_OK:
        st = zvc.zvc_get_error(ws.data_ptr(), sh())
    return st, y[:n].cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("name", golden_io.all_rle())
def test_hand_derived_bytes(name):
    g = golden_io.load_rle(name)
    got = gpu_rle(g["input"], g["window"])
    assert got.tobytes() == g["expected"]
    st, back = gpu_unrle(np.frombuffer(g["expected"], np.uint8), g["n"], g["window"])
    assert st == zvc.ZVC_OK and np.array_equal(back, g["input"])


def _words(rng, n, density, run):
    if run:  # alternating runs of random lengths up to `run`
        w, i, on = np.zeros(n, dtype=np.uint32), 0, rng.random() < density
        while i < n:
            k = int(rng.integers(1, run + 1))
            if on:
                w[i:i + k] = rng.integers(1, 2**32, size=min(k, n - i), dtype=np.uint64)
            i, on = i + k, not on
        return w
    return (rng.integers(1, 2**32, size=n, dtype=np.uint64) * (rng.random(n) < density)).astype(np.uint32)


@pytest.mark.parametrize("window", [32, 96, 1024, 4096])
def test_matches_the_oracle(window):
    rng = np.random.default_rng(window)
    for n in (1, 31, 33, window - 1, window, window + 1, 3 * window + 5, 100_003):
        for density, run in ((0.0, 0), (1.0, 0), (0.5, 0), (0.3, 0), (0.6, 50), (0.5, 2000)):
            w = _words(rng, n, density, run)
            got = gpu_rle(w, window)
            ref = oracle.rle_encode(w, window)
            assert np.array_equal(got, ref), (n, density, run)
            st, back = gpu_unrle(got, n, window)
            assert st == zvc.ZVC_OK and np.array_equal(back, w), (n, density, run)


def test_alexnet_layer_in_two_layouts():
    x = workloads.alexnet_stack(device="cuda", batch=16)[0]  # 16 x 96 x 55 x 55
    for t in (x, x.permute(0, 2, 3, 1).contiguous()):  # NCHW, NHWC
        w = words_of(t)
        got = gpu_rle(w, 1024)
        assert np.array_equal(got, oracle.rle_encode(w, 1024))
        st, back = gpu_unrle(got, w.size, 1024)
        assert st == zvc.ZVC_OK and np.array_equal(back, w)


def test_empty_and_header_only_streams():
    assert gpu_rle(np.zeros(0, np.uint32), 1024).tobytes() == oracle.rle_encode(
        np.zeros(0, np.uint32), 1024).tobytes()
    s = oracle.rle_encode(np.zeros(0, np.uint32), 1024)
    assert gpu_unrle(s, 0, 1024)[0] == zvc.ZVC_OK
    bad = s.copy()
    bad[0] ^= 1
    assert gpu_unrle(bad, 0, 1024)[0] == zvc.ZVC_ERR_CORRUPT


def test_corrupt_streams_get_the_oracle_verdict():
    rng = np.random.default_rng(5)
    n, window = 5000, 96
    w = _words(rng, n, 0.5, 40)
    s = oracle.rle_encode(w, window)
    for _ in range(200):
        bad = s.copy()
        i = int(rng.integers(0, bad.size))
        bad[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        ost, oback = oracle.rle_decode(bad, n, window)
        gst, gback = gpu_unrle(bad, n, window)
        if ost == oracle.OK:
            assert gst == zvc.ZVC_OK and np.array_equal(gback, oback), i
        else:
            assert gst == zvc.ZVC_ERR_CORRUPT, i


def test_host_checks():
    ensure_lib()
    assert zvc.zvc_rle_size_bound(10, 33) == 0
    assert zvc.zvc_rle_size_bound(10, zvc.ZVC_RLE_MAX_WINDOW + 32) == 0
    x = torch.ones(64, dtype=torch.int32, device="cuda")
    out = torch.empty(1024, dtype=torch.uint8, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_rle_workspace_size(64, 32))
    size = torch.zeros(2, dtype=torch.int64, device="cuda")
    # output not 8-byte aligned
    assert zvc.zvc_rle_compress(x.data_ptr(), 64, 32, out.data_ptr() + 4, 512, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_ERR_INVALID_ARG
    assert zvc.zvc_rle_compress(x.data_ptr(), 64, 32, out.data_ptr(), 16, size.data_ptr(),
                                ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_ERR_BUFFER_TOO_SMALL
