"""Pins for the 16-bit ZVC oracle (no GPU).

ZVC on bf16 / fp16 activation words is a reading beyond the pages: Rhu et al.,
"Compressing DMA Engine", section V.A gives the rule (32 values, a 32-bit zero/non-zero
mask, the non-zero values appended) for the 32-bit activations the paper evaluates; here
the values are 2 bytes. The oracle is checked against things other than itself:
hand-derived byte vectors, an independent pure-Python codec, the closed-form size, the
pinned 32-bit oracle on zero-extended words (same masks, same values, half the value
bytes), exact round trip, layout invariants and corruption detection.
"""
import struct

import numpy as np
import pytest

import oracle
from tests import golden_io
from tests.zvc_tiny import tiny_decode16, tiny_encode16


@pytest.fixture(scope="module")
def z16():
    return oracle.z16_load()


def closed_form16(words: np.ndarray, chunk_elems: int) -> int:
    """S = 32 + 8*ceil(n/C) + 4*ceil(n/32) + 2*nnz, nnz counted with numpy."""
    n = words.size
    return (32 + 8 * (-(-n // chunk_elems)) + 4 * (-(-n // 32))
            + 2 * int(np.count_nonzero(words.view(np.uint16))))


def random16(rng, n, density):
    w = rng.integers(1, 2**16, size=n, dtype=np.uint32).astype(np.uint16)
    w[rng.random(n) >= density] = 0
    return w


def windows_of(stream: bytes, n: int, chunk_elems: int, word_bytes: int):
    """(chunk offsets, [(mask, [values])] per window) of a valid stream."""
    nc = -(-n // chunk_elems)
    offs = [struct.unpack_from("<Q", stream, 32 + 8 * c)[0] for c in range(nc)]
    pos = 32 + 8 * nc
    fmt = "<H" if word_bytes == 2 else "<I"
    wins = []
    for _ in range(-(-n // 32)):
        (m,) = struct.unpack_from("<I", stream, pos)
        pos += 4
        vals = []
        for i in range(32):
            if m >> i & 1:
                vals.append(struct.unpack_from(fmt, stream, pos)[0])
                pos += word_bytes
        wins.append((m, vals))
    assert pos == len(stream)
    return offs, wins


# ------------------------------------------------------------------ golden vectors
@pytest.mark.parametrize("name", golden_io.all_z16())
def test_golden16(name, z16):
    g = golden_io.load_z16(name)
    got = oracle.encode16(g["input"], g["chunk_elems"], lib=z16)
    assert got.tobytes() == g["expected"]
    st, back = oracle.decode16(np.frombuffer(g["expected"], np.uint8), g["n"], g["chunk_elems"],
                               lib=z16)
    assert st == oracle.OK and np.array_equal(back, g["input"])


# ------------------------------------------------------------------ independent codec
@pytest.mark.parametrize("chunk_elems", [32, 64, 1024, 4096])
def test_tiny_codec_agrees_for_all_small_n(chunk_elems, z16):
    rng = np.random.default_rng(chunk_elems)
    for n in range(0, 301):
        w = random16(rng, n, [0.0, 0.1, 0.5, 1.0][n % 4])
        ref = tiny_encode16(w.tolist(), chunk_elems)
        got = oracle.encode16(w, chunk_elems, lib=z16)
        assert got.tobytes() == ref, n
        st, back = oracle.decode16(got, n, chunk_elems, lib=z16)
        assert st == oracle.OK and np.array_equal(back, w), n
        assert tiny_decode16(ref, n, chunk_elems) == w.tolist()


# ------------------------------------------------------------------ the 32-bit oracle
@pytest.mark.parametrize("n,chunk_elems", [(1, 32), (100, 64), (4097, 1024), (70_001, 4096)])
def test_same_masks_and_values_as_the_32_bit_oracle(n, chunk_elems, z16, oracle_lib):
    """Zero-extended to 32 bits, the same words have the same zero pattern, so the pinned
    32-bit oracle gives the same masks and the same values in the same order; only each
    value's width differs (4 bytes against 2), and with it every chunk offset."""
    rng = np.random.default_rng(n)
    w16 = random16(rng, n, 0.3)
    w16[::7] = 0x8000  # -0.0 in bf16 and fp16: non-zero bits
    s16 = oracle.encode16(w16, chunk_elems, lib=z16).tobytes()
    s32 = oracle.encode(w16.astype(np.uint32), chunk_elems, lib=oracle_lib).tobytes()
    o16, win16 = windows_of(s16, n, chunk_elems, 2)
    o32, win32 = windows_of(s32, n, chunk_elems, 4)
    assert win16 == win32
    wpc = chunk_elems // 32
    for c in range(len(o16)):
        before = win16[:c * wpc]
        nz = sum(len(v) for _, v in before)
        assert o16[c] == 4 * len(before) + 2 * nz
        assert o32[c] == 4 * len(before) + 4 * nz
    assert struct.unpack_from("<H", s16, 6)[0] == 2 and struct.unpack_from("<H", s32, 6)[0] == 4


# ------------------------------------------------------------------ closed form, round trip
@pytest.mark.parametrize("n,chunk_elems", [(0, 4096), (1, 32), (4095, 4096), (4097, 4096),
                                           (100_003, 1024), (65_536, 32768)])
@pytest.mark.parametrize("density", [0.0, 0.05, 0.5, 1.0])
def test_closed_form_size_and_round_trip(n, chunk_elems, density, z16):
    w = random16(np.random.default_rng(n + int(density * 100)), n, density)
    s = oracle.encode16(w, chunk_elems, lib=z16)
    assert s.size == closed_form16(w, chunk_elems)
    st, back = oracle.decode16(s, n, chunk_elems, lib=z16)
    assert st == oracle.OK and np.array_equal(back, w)


def test_all_zero_window_is_16x(z16):
    n = 32 * 1000
    s = oracle.encode16(np.zeros(n, np.uint16), 32 * 1000, lib=z16)
    assert s.size - 32 - 8 == 4 * 1000  # 64 bytes of data per window -> one 4-byte mask


def test_all_dense_is_worst_case(z16):
    n = 10_000
    w = np.arange(1, n + 1, dtype=np.uint16)
    s = oracle.encode16(w, 4096, lib=z16)
    assert s.size == oracle.size_bound16(n, 4096, lib=z16)
    assert s.size == 32 + 8 * 3 + 4 * (-(-n // 32)) + 2 * n


def test_size_independent_of_order_within_window(z16):
    """Section VII.A: ZVC's ratio does not depend on how values are laid out inside a
    window (only the mask changes)."""
    rng = np.random.default_rng(3)
    w = random16(rng, 32 * 64, 0.4)
    p = w.reshape(-1, 32)[:, rng.permutation(32)].reshape(-1)
    assert oracle.encode16(w, 1024, lib=z16).size == oracle.encode16(p, 1024, lib=z16).size


def test_each_extra_nonzero_adds_two_bytes(z16):
    w = np.zeros(4096, np.uint16)
    base = oracle.encode16(w, 4096, lib=z16).size
    for k, i in enumerate([0, 31, 32, 4095, 100], start=1):
        w[i] = 0x0101
        assert oracle.encode16(w, 4096, lib=z16).size == base + 2 * k


# ------------------------------------------------------------------ corruption
def test_rejects_bad_headers_and_parameters(z16):
    w = random16(np.random.default_rng(5), 1000, 0.3)
    s = oracle.encode16(w, 64, lib=z16)
    for off in (0, 4, 6, 8, 12, 16, 24):
        bad = s.copy()
        bad[off] ^= 1
        assert oracle.decode16(bad, 1000, 64, lib=z16)[0] == oracle.ERR_CORRUPT, off
    assert oracle.decode16(s, 1001, 64, lib=z16)[0] == oracle.ERR_CORRUPT
    assert oracle.decode16(s, 1000, 32, lib=z16)[0] == oracle.ERR_CORRUPT
    assert oracle.decode16(s[:-2], 1000, 64, lib=z16)[0] == oracle.ERR_CORRUPT
    # a 32-bit stream of the same words is not a 16-bit stream (word_bytes differs)
    assert oracle.decode16(oracle.encode(w.astype(np.uint32), 64), 1000, 64, lib=z16)[0] == \
        oracle.ERR_CORRUPT


def test_tail_mask_bits_beyond_n_are_rejected(z16):
    w = np.ones(40, np.uint16)
    s = oracle.encode16(w, 64, lib=z16)
    # the second window covers elements 32..39: set its bit 8 (element 40, past n)
    off = 32 + 8 + 4 + 64
    bad = s.copy()
    bad[off + 1] |= 0x01
    assert oracle.decode16(bad, 40, 64, lib=z16)[0] == oracle.ERR_CORRUPT


def test_random_corruption_never_disagrees_with_tiny_decoder(z16):
    rng = np.random.default_rng(11)
    for t in range(300):
        n = int(rng.integers(1, 400))
        C = int(rng.choice([32, 64, 128]))
        w = random16(rng, n, float(rng.choice([0.05, 0.3, 0.9])))
        s = oracle.encode16(w, C, lib=z16)
        bad = s.copy()
        for _ in range(int(rng.integers(1, 3))):
            bad[int(rng.integers(0, bad.size))] ^= 1 << int(rng.integers(0, 8))
        if t % 5 == 0:
            bad = bad[:int(rng.integers(0, bad.size))]
        st, back = oracle.decode16(bad, n, C, lib=z16)
        ref = tiny_decode16(bad.tobytes(), n, C)
        if ref is None:
            assert st == oracle.ERR_CORRUPT, t
        else:
            assert st == oracle.OK and back.tolist() == ref, t
