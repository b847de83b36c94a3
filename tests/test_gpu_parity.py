"""GPU parity on small and ragged inputs: the sm_103a kernels, called through the C ABI,
must produce the oracle's bytes exactly and decode the oracle's streams to the exact
input words (ZVC is lossless; Rhu et al., "Compressing DMA Engine", section V.A)."""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests import golden_io
from tests.gpu_util import ensure_lib, gpu_compress, gpu_decompress, sh, words_of

pytestmark = pytest.mark.gpu


def _dev_words(w: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(w.view(np.int32).copy()).cuda()


def _random_words(rng, n, density):
    w = rng.integers(1, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    w[rng.random(n) >= density] = 0
    return w


def _assert_parity(w: np.ndarray, C: int, **kw):
    st, got, err = gpu_compress(_dev_words(w), C, **kw)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    ref = oracle.encode(w, C)
    assert got.size == ref.size, (w.size, C)
    assert np.array_equal(got, ref), (w.size, C, int(np.flatnonzero(got != ref)[0]))
    st, err, back = gpu_decompress(ref, w.size, C)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert np.array_equal(back, w), (w.size, C)


@pytest.mark.parametrize("name", golden_io.all_single())
def test_golden_vectors(name):
    g = golden_io.load(name)
    st, got, err = gpu_compress(_dev_words(g["input"]), g["chunk_elems"]) if g["n"] else \
        gpu_compress(torch.empty(0, dtype=torch.int32, device="cuda"), g["chunk_elems"])
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert got.tobytes() == g["expected"]
    st, err, back = gpu_decompress(np.frombuffer(g["expected"], np.uint8), g["n"], g["chunk_elems"])
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert np.array_equal(back, g["input"])


SIZES = [1, 2, 31, 32, 33, 127, 128, 129, 4095, 4096, 4097, 8191, 8192, 12_293, 65_536 + 17,
         100_003, 1_000_003]


@pytest.mark.parametrize("C", [32, 64, 96, 128, 256, 512, 1024, 2048, 4096, 8192, 16384, 32768])
def test_random_ragged_sizes(C):
    rng = np.random.default_rng(C)
    for n in SIZES:
        for d in (0.0, 0.07, 0.5, 1.0):
            _assert_parity(_random_words(rng, n, d), C)


def test_special_bit_patterns_are_nonzero():
    w = np.zeros(4097, np.uint32)
    w[[0, 31, 32, 4095, 4096]] = [0x80000000, 0x7FC00000, 0x00000001, 0xFF800000, 0x80000001]
    _assert_parity(w, 4096)
    _assert_parity(w, 32)


@pytest.mark.parametrize("n", workloads.ODD_SIZES)
def test_odd_activation_sizes(n):
    x = workloads.odd_case(n, device="cuda")[0]
    _assert_parity(words_of(x), 4096)
    _assert_parity(words_of(x), 1024)


@pytest.mark.parametrize("pad", [4, 8, 12])
def test_unaligned_destination(pad):
    rng = np.random.default_rng(pad)
    for n in (5, 4096 * 3 + 77, 100_003):
        _assert_parity(_random_words(rng, n, 0.4), 4096, out_pad_bytes=pad)


@pytest.mark.parametrize("off", [1, 2, 3])
def test_unaligned_source_and_output(off):
    rng = np.random.default_rng(10 + off)
    n = 4096 * 5 + 33
    w = _random_words(rng, n, 0.3)
    big = torch.zeros(n + 8, dtype=torch.int32, device="cuda")
    big[off:off + n] = _dev_words(w)
    st, got, err = gpu_compress(big[off:off + n], 4096)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert np.array_equal(got, oracle.encode(w, 4096))
    st, err, back = gpu_decompress(oracle.encode(w, 4096), n, 4096, out_offset_words=off)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK and np.array_equal(back, w)


def _chunkwise_words(rng, C, densities):
    return np.concatenate([_random_words(rng, C, d) for d in densities])


CHUNK_PATTERNS = ([0.0] * 30 + [1.0] + [0.0] * 30, [1.0] + [0.0] * 40, [0.0] * 40 + [1.0],
                  [0.0, 0.9, 0.0, 0.3, 1.0, 0.0, 0.0, 0.6] * 4, [0.05] * 20 + [0.97, 1.0])


@pytest.mark.parametrize("C", [4096, 16384])
def test_chunks_longer_than_the_mean(C):
    """Dense chunks among sparse ones. A decompressing CTA's chunk buffer is sized from the
    stream's mean chunk, so these chunks are staged and walked in several pieces, each
    starting at a window of its own 16-byte phase."""
    rng = np.random.default_rng(C + 7)
    for pattern in CHUNK_PATTERNS:
        w = _chunkwise_words(rng, C, pattern)
        for cut in (0, 37, C // 2 + 5):
            _assert_parity(w[:w.size - cut], C)


@pytest.mark.parametrize("off", [1, 2, 3])
def test_chunks_longer_than_the_mean_unaligned(off):
    rng = np.random.default_rng(30 + off)
    w = _chunkwise_words(rng, 4096, [0.0] * 12 + [1.0, 0.8] + [0.0] * 12)
    n = w.size
    s = oracle.encode(w, 4096)
    # the stream at a 4-byte offset from 16-byte alignment, so every piece's phase moves
    raw = torch.zeros(s.size + 16, dtype=torch.uint8, device="cuda")
    raw[4 * off:4 * off + s.size] = torch.from_numpy(s.copy()).cuda()
    out = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    ws = zvc.new_workspace(zvc.ZVC_WORKSPACE_ALIGN)
    st = zvc.zvc_decompress(raw.data_ptr() + 4 * off, s.size, out.data_ptr(), n, 4096,
                            ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK and zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert np.array_equal(out.cpu().numpy().view(np.uint32), w)


@pytest.mark.parametrize("cut", [0, 4096 * 3 + 101])
def test_many_short_chunks(cut):
    """8192 sparse chunks (3% non-zero): a launch of more than two waves of short chunks,
    where a decompressing CTA holds several chunks and one warp walks them all."""
    rng = np.random.default_rng(40 + cut)
    w = _random_words(rng, 8192 * 4096 - cut, 0.03)
    w[: 4096 * 2] = _random_words(rng, 4096 * 2, 1.0)  # two dense chunks among them
    st, err, back = gpu_decompress(oracle.encode(w, 4096), w.size, 4096)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert np.array_equal(back, w)


def test_single_relu_config_bit_exact():
    x = workloads.single_relu(device="cuda")[0]
    w = words_of(x)
    _assert_parity(w, 4096)
    _assert_parity(w, 1024)  # the paper's 4 KB compression window


def test_deterministic_and_workspace_reuse():
    rng = np.random.default_rng(3)
    w = _random_words(rng, 3_000_000, 0.45)
    x = _dev_words(w)
    ws = zvc.new_workspace(zvc.zvc_workspace_size(w.size, 4096))
    outs = [gpu_compress(x, 4096, ws=ws)[1] for _ in range(4)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    assert np.array_equal(outs[0], oracle.encode(w, 4096))


def test_round_trip_on_device_of_gpu_stream():
    x = workloads.odd_case(2_000_000 + 3, device="cuda", density=0.3)[0]
    out, size = zvc.compress(x, 4096)
    y = zvc.decompress(out, int(size.item()), x.numel(), 4096)
    torch.cuda.synchronize()
    assert torch.equal(x.view(torch.int32), y.view(torch.int32))


# ------------------------------------------------------------------ batches
def _gpu_compress_batched(xs, C):
    ensure_lib()
    ns = [x.numel() for x in xs]
    cap = zvc.zvc_batch_size_bound(ns, C)
    buf = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_batch_workspace_size(ns, C))
    st = zvc.zvc_compress_batched([x.data_ptr() for x in xs], ns, C, buf.data_ptr(), cap,
                                  size.data_ptr(), ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    s = int(size.item())
    host = buf.cpu().numpy()
    assert (host[s:] == 0xEE).all()
    return host[:s].copy()


def _gpu_decompress_batched(stream, ns, C):
    d_in = torch.from_numpy(stream).cuda()
    outs = [torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda") for n in ns]
    ws = zvc.new_workspace(256)
    st = zvc.zvc_decompress_batched(d_in.data_ptr(), d_in.numel(), [o.data_ptr() for o in outs],
                                    ns, C, ws.data_ptr(), ws.numel(), sh())
    err = zvc.zvc_get_error(ws.data_ptr(), sh()) if st == zvc.ZVC_OK else None
    return st, err, [o.cpu().numpy().view(np.uint32)[:n] for o, n in zip(outs, ns)]


@pytest.mark.parametrize("C", [1024, 4096])
def test_batched_many_short_chunks_with_empty_tensors(C):
    """A batch of sparse tensors with empty ones among them, large enough that a
    decompressing CTA holds several chunks: the header checks of the empty tensors run in
    lanes of a walker warp that also walks chunks."""
    rng = np.random.default_rng(50 + C)
    ns = [(12000 if C == 1024 else 8000) * C + 77, 0, 1000, 0, 3 * C, 5 * C + 1]  # > 2 waves
    ws_ = [_random_words(rng, n, 0.03) for n in ns]
    ws_[4][: C] = _random_words(rng, C, 1.0)  # a dense chunk staged in pieces
    ref = oracle.encode_batch(ws_, C)
    st, err, backs = _gpu_decompress_batched(ref, ns, C)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    for w, b in zip(ws_, backs):
        assert np.array_equal(b, w)
    got = _gpu_compress_batched([_dev_words(w) if w.size else
                                 torch.empty(0, dtype=torch.int32, device="cuda") for w in ws_], C)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name", golden_io.all_batch())
def test_golden_batch(name):
    g = golden_io.load(name)
    xs = [_dev_words(w) if w.size else torch.empty(0, dtype=torch.int32, device="cuda")
          for w in g["inputs"]]
    got = _gpu_compress_batched(xs, g["chunk_elems"])
    assert got.tobytes() == g["expected"]
    st, err, backs = _gpu_decompress_batched(np.frombuffer(g["expected"], np.uint8).copy(), g["ns"],
                                             g["chunk_elems"])
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert all(np.array_equal(a, b) for a, b in zip(backs, g["inputs"]))


@pytest.mark.parametrize("C", [32, 1024, 4096])
def test_batched_mixed_sizes(C):
    rng = np.random.default_rng(C + 1)
    sizes = [0, 1, 4096, 0, 33, 70_001, 4096 * 7, 5, 0, 200_000]
    ws_ = [_random_words(rng, n, float(rng.uniform(0.05, 0.95))) for n in sizes]
    xs = [_dev_words(w) if w.size else torch.empty(0, dtype=torch.int32, device="cuda") for w in ws_]
    got = _gpu_compress_batched(xs, C)
    ref = oracle.encode_batch(ws_, C)
    assert np.array_equal(got, ref)
    st, err, backs = _gpu_decompress_batched(ref, sizes, C)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert all(np.array_equal(a, b) for a, b in zip(backs, ws_))


def test_batched_empty_and_max_batch():
    got = _gpu_compress_batched([], 4096)
    assert np.array_equal(got, oracle.encode_batch([], 4096))
    st, err, _ = _gpu_decompress_batched(got, [], 4096)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    rng = np.random.default_rng(99)
    ws_ = [_random_words(rng, int(rng.integers(0, 300)), 0.5) for _ in range(zvc.ZVC_MAX_BATCH)]
    xs = [_dev_words(w) if w.size else torch.empty(0, dtype=torch.int32, device="cuda") for w in ws_]
    got = _gpu_compress_batched(xs, 64)
    assert np.array_equal(got, oracle.encode_batch(ws_, 64))
    st, err, backs = _gpu_decompress_batched(got, [w.size for w in ws_], 64)
    assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
    assert all(np.array_equal(a, b) for a, b in zip(backs, ws_))
