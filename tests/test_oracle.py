"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: hand-derived byte vectors,
the closed-form size, an independent pure-Python brute-force codec, exact round trip,
layout invariants the paper states, and corruption detection. Core rule: Rhu et al.,
"Compressing DMA Engine", section V.A (32-word windows, a 32-bit mask, the non-zero
words appended; an all-zero window is a single mask, i.e. 32x).
"""
import struct

import numpy as np
import pytest

import oracle
from tests import golden_io
from tests.zvc_tiny import tiny_decode, tiny_encode, tiny_encode_batch


def closed_form_size(words: np.ndarray, chunk_elems: int) -> int:
    """S = 32 + 8*ceil(n/C) + 4*ceil(n/32) + 4*nnz, nnz counted with numpy."""
    n = words.size
    nnz = int(np.count_nonzero(words.view(np.uint32)))
    return 32 + 8 * (-(-n // chunk_elems)) + 4 * (-(-n // 32)) + 4 * nnz


def random_words(rng, n, density):
    w = rng.integers(1, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    w[rng.random(n) >= density] = 0
    return w


# ------------------------------------------------------------------ golden vectors
@pytest.mark.parametrize("name", golden_io.all_single())
def test_golden_single(name, oracle_lib):
    g = golden_io.load(name)
    got = oracle.encode(g["input"], g["chunk_elems"], lib=oracle_lib)
    assert got.tobytes() == g["expected"]
    assert tiny_encode(g["input"].tolist(), g["chunk_elems"]) == g["expected"]
    st, back = oracle.decode(np.frombuffer(g["expected"], np.uint8), g["n"], g["chunk_elems"],
                             lib=oracle_lib)
    assert st == oracle.OK
    assert np.array_equal(back, g["input"])
    assert len(g["expected"]) == closed_form_size(g["input"], g["chunk_elems"])


@pytest.mark.parametrize("name", golden_io.all_batch())
def test_golden_batch(name, oracle_lib):
    g = golden_io.load(name)
    got = oracle.encode_batch(g["inputs"], g["chunk_elems"], lib=oracle_lib)
    assert got.tobytes() == g["expected"]
    assert tiny_encode_batch([x.tolist() for x in g["inputs"]], g["chunk_elems"]) == g["expected"]
    st, backs = oracle.decode_batch(np.frombuffer(g["expected"], np.uint8), g["ns"],
                                    g["chunk_elems"], lib=oracle_lib)
    assert st == oracle.OK
    for a, b in zip(backs, g["inputs"]):
        assert np.array_equal(a, b)


# ------------------------------------------------------- brute force vs the oracle
@pytest.mark.parametrize("chunk_elems", [32, 64, 1024, 4096])
def test_tiny_codec_agrees_for_all_small_n(chunk_elems, oracle_lib):
    rng = np.random.default_rng(chunk_elems)
    for n in range(0, 301):
        density = [0.0, 0.1, 0.5, 0.9, 1.0][n % 5]
        w = random_words(rng, n, density)
        if n > 3:  # the special bit patterns that must count as non-zero
            w[rng.integers(0, n, 3)] = [0x80000000, 0x7FC00000, 0x00000001]
        ref = tiny_encode(w.tolist(), chunk_elems)
        got = oracle.encode(w, chunk_elems, lib=oracle_lib)
        assert got.tobytes() == ref, (n, chunk_elems)
        st, back = oracle.decode(got, n, chunk_elems, lib=oracle_lib)
        assert st == oracle.OK and np.array_equal(back, w)
        assert tiny_decode(ref, n, chunk_elems) == w.tolist()


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("n,chunk_elems", [(0, 4096), (1, 32), (4095, 4096), (4097, 4096),
                                           (200_704, 4096), (100_003, 1024), (77_777, 96)])
@pytest.mark.parametrize("density", [0.0, 0.05, 0.5, 1.0])
def test_closed_form_size_and_round_trip(n, chunk_elems, density, oracle_lib):
    rng = np.random.default_rng(n + int(density * 100))
    w = random_words(rng, n, density)
    s = oracle.encode(w, chunk_elems, lib=oracle_lib)
    assert s.size == closed_form_size(w, chunk_elems)
    assert s.size <= oracle.size_bound(n, chunk_elems, lib=oracle_lib)
    st, back = oracle.decode(s, n, chunk_elems, lib=oracle_lib)
    assert st == oracle.OK and np.array_equal(back, w)


def test_all_zero_is_32x_per_window(oracle_lib):
    # section V.A: a window of 32 zeros is one all-zero 32-bit mask.
    n, c = 32 * 4096, 4096
    s = oracle.encode(np.zeros(n, np.uint32), c, lib=oracle_lib)
    payload = s.size - 32 - 8 * (n // c)
    assert payload * 32 == 4 * n
    assert not s[32 + 8 * (n // c):].any()


def test_all_dense_is_worst_case(oracle_lib):
    n, c = 10_000, 4096
    w = np.arange(1, n + 1, dtype=np.uint32)
    s = oracle.encode(w, c, lib=oracle_lib)
    assert s.size == oracle.size_bound(n, c, lib=oracle_lib)
    assert s.size == 32 + 8 * 3 + 4 * (-(-n // 32)) + 4 * n


def test_relu_activations_round_trip(oracle_lib):
    import workloads
    x = workloads.single_relu(device="cpu")[0].numpy()
    w = x.view(np.uint32).reshape(-1)
    s = oracle.encode(w, 4096, lib=oracle_lib)
    assert s.size == closed_form_size(w, 4096)
    ratio = 4 * w.size / s.size
    assert 1.7 < ratio < 2.0  # about half zeros: 4n / (4n/32 + 2n) ~ 1.88
    st, back = oracle.decode(s, w.size, 4096, lib=oracle_lib)
    assert st == oracle.OK and np.array_equal(back, w)


# ------------------------------------------------------------------ invariants
def test_size_independent_of_order_within_window(oracle_lib):
    # section VII.A: ZVC's ratio does not depend on how activations are arranged; within
    # a window a permutation keeps the mask's popcount and therefore the size.
    rng = np.random.default_rng(7)
    w = random_words(rng, 32 * 500, 0.4)
    p = w.reshape(-1, 32).copy()
    for row in p:
        rng.shuffle(row)
    a = oracle.encode(w, 1024, lib=oracle_lib)
    b = oracle.encode(p.reshape(-1), 1024, lib=oracle_lib)
    assert a.size == b.size


def test_each_extra_nonzero_adds_four_bytes(oracle_lib):
    rng = np.random.default_rng(8)
    w = random_words(rng, 5000, 0.3)
    base = oracle.encode(w, 1024, lib=oracle_lib).size
    zeros = np.flatnonzero(w == 0)[:50]
    for k, i in enumerate(zeros, 1):
        w[i] = 0xABCD
        assert oracle.encode(w, 1024, lib=oracle_lib).size == base + 4 * k


def test_chunk_table_is_prefix_of_chunk_sizes(oracle_lib):
    rng = np.random.default_rng(9)
    n, c = 50_000, 1024
    w = random_words(rng, n, 0.35)
    s = oracle.encode(w, c, lib=oracle_lib)
    nc = -(-n // c)
    offs = np.frombuffer(s[32:32 + 8 * nc].tobytes(), dtype="<u8")
    payload = int(np.frombuffer(s[24:32].tobytes(), "<u8")[0])
    sizes = []
    for k in range(nc):
        blk = w[k * c:(k + 1) * c]
        sizes.append(4 * (-(-blk.size // 32)) + 4 * int(np.count_nonzero(blk)))
    assert offs[0] == 0 and np.all(np.diff(offs.astype(np.int64)) > 0)
    assert np.array_equal(offs, np.cumsum([0] + sizes[:-1]))
    assert sum(sizes) == payload


def test_chunk_size_changes_only_the_table(oracle_lib):
    # section VII.A reports a 4 KB window and similar results for larger windows; with
    # ZVC the payload is the same for every chunk size, only the offset table differs.
    rng = np.random.default_rng(10)
    n = 1 << 18
    w = random_words(rng, n, 0.38)
    sizes = {c: oracle.encode(w, c, lib=oracle_lib).size for c in (1024, 4096, 16384)}
    for c, s in sizes.items():
        assert s - 8 * (n // c) == sizes[1024] - 8 * (n // 1024)


# ------------------------------------------------------------------ corruption
def _good_stream(oracle_lib, n=3000, c=1024, density=0.4, seed=11):
    rng = np.random.default_rng(seed)
    w = random_words(rng, n, density)
    return w, oracle.encode(w, c, lib=oracle_lib)


def test_rejects_bad_headers_and_parameters(oracle_lib):
    w, s = _good_stream(oracle_lib)
    n, c = w.size, 1024
    assert oracle.decode(s, n, c, lib=oracle_lib)[0] == oracle.OK
    for off in (0, 4, 6, 8, 12, 16, 24):  # every header field
        t = s.copy()
        t[off] ^= 0x01
        assert oracle.decode(t, n, c, lib=oracle_lib)[0] == oracle.ERR_CORRUPT, off
    assert oracle.decode(s, n + 1, c, lib=oracle_lib)[0] == oracle.ERR_CORRUPT
    assert oracle.decode(s, n, 2048, lib=oracle_lib)[0] == oracle.ERR_CORRUPT
    assert oracle.decode(s[:-4], n, c, lib=oracle_lib)[0] == oracle.ERR_CORRUPT
    assert oracle.decode(np.concatenate([s, s[-4:]]), n, c, lib=oracle_lib)[0] == oracle.ERR_CORRUPT
    assert oracle.decode(s[:31], n, c, lib=oracle_lib)[0] == oracle.ERR_CORRUPT
    assert oracle.decode(s, n, 48, lib=oracle_lib)[0] == oracle.ERR_INVALID_ARG
    with pytest.raises(oracle.OracleError):
        oracle.encode(w, 0, lib=oracle_lib)


def test_flipped_mask_bit_is_detected(oracle_lib):
    w, s = _good_stream(oracle_lib)
    payload_start = 32 + 8 * 3
    first_mask = payload_start  # chunk 0, window 0
    for bit in range(32):
        t = s.copy()
        t[first_mask + bit // 8] ^= 1 << (bit % 8)
        st, back = oracle.decode(t, w.size, 1024, lib=oracle_lib)
        # one more or one fewer word per window shifts every later mask, so the chunk
        # cannot end where the table says
        assert st == oracle.ERR_CORRUPT


def test_bad_offset_table_is_detected(oracle_lib):
    w, s = _good_stream(oracle_lib)
    for k, delta in ((0, 4), (1, 4), (1, -4), (2, 8)):
        t = s.copy()
        v = int(np.frombuffer(t[32 + 8 * k:40 + 8 * k].tobytes(), "<u8")[0]) + delta
        t[32 + 8 * k:40 + 8 * k] = np.frombuffer(struct.pack("<Q", v % 2**64), np.uint8)
        assert oracle.decode(t, w.size, 1024, lib=oracle_lib)[0] == oracle.ERR_CORRUPT


def test_tail_mask_bits_beyond_n_are_rejected(oracle_lib):
    w = np.zeros(33, np.uint32)
    w[32] = 5
    s = oracle.encode(w, 32, lib=oracle_lib)
    t = s.copy()
    # last window: its mask is at payload offset 4; element 33 does not exist
    t[32 + 16 + 4] |= 0x02
    t_words = tiny_decode(t.tobytes(), 33, 32)
    assert t_words is None
    assert oracle.decode(t, 33, 32, lib=oracle_lib)[0] == oracle.ERR_CORRUPT


def test_random_corruption_never_disagrees_with_tiny_decoder(oracle_lib):
    rng = np.random.default_rng(12)
    for trial in range(300):
        n = int(rng.integers(1, 200))
        c = int(rng.choice([32, 64, 96]))
        w = random_words(rng, n, float(rng.random()))
        s = oracle.encode(w, c, lib=oracle_lib)
        t = s.copy()
        for _ in range(int(rng.integers(1, 4))):
            i = int(rng.integers(0, t.size))
            t[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        st, back = oracle.decode(t, n, c, lib=oracle_lib)
        ref = tiny_decode(t.tobytes(), n, c)
        if ref is None:
            assert st == oracle.ERR_CORRUPT, trial
        else:
            assert st == oracle.OK and back.tolist() == ref, trial


# ------------------------------------------------------------------ batches
def test_batch_is_table_plus_streams(oracle_lib):
    rng = np.random.default_rng(13)
    xs = [random_words(rng, n, d) for n, d in ((0, 0.5), (1, 1.0), (5000, 0.3), (4096, 0.0),
                                               (12_345, 0.9))]
    b = oracle.encode_batch(xs, 1024, lib=oracle_lib)
    T = len(xs)
    magic, t, total = struct.unpack_from("<IIQ", b.tobytes(), 0)
    assert (magic, t, total) == (0x4243565A, T, b.size)
    offs = struct.unpack_from(f"<{T + 1}Q", b.tobytes(), 16)
    assert offs[0] == 16 + 8 * (T + 1) and offs[-1] == b.size
    for i, x in enumerate(xs):
        assert b[offs[i]:offs[i + 1]].tobytes() == oracle.encode(x, 1024, lib=oracle_lib).tobytes()
    assert b.tobytes() == tiny_encode_batch([x.tolist() for x in xs], 1024)
    st, backs = oracle.decode_batch(b, [x.size for x in xs], 1024, lib=oracle_lib)
    assert st == oracle.OK
    assert all(np.array_equal(a, x) for a, x in zip(backs, xs))
    bad = b.copy()
    bad[8] ^= 1
    assert oracle.decode_batch(bad, [x.size for x in xs], 1024, lib=oracle_lib)[0] == oracle.ERR_CORRUPT


def test_empty_batch(oracle_lib):
    b = oracle.encode_batch([], 4096, lib=oracle_lib)
    assert b.tobytes() == struct.pack("<IIQQ", 0x4243565A, 0, 24, 24)
    assert oracle.decode_batch(b, [], 4096, lib=oracle_lib)[0] == oracle.OK
