"""Pins for the RLE oracle (oracle/rle_oracle.c), the layout-dependent comparison codec of
Rhu et al., "Compressing DMA Engine" (section V.A: RLE exploits runs of zeros and non-zeros,
so it depends on how values are laid out; section VII.A: ZVC's ratio is independent of the
layout, RLE's is not). Each pin checks the oracle against something other than itself:
hand-derived bytes, an independent brute-force codec, a closed form, a property."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle
from tests import golden_io


# ------------------------------------------------------------------ independent codec
def brute_encode(words, window):
    """Plain-Python RLE with the same layout, written from the format description."""
    n = len(words)
    nw = -(-n // window)
    payload, offs = bytearray(), []
    for w in range(nw):
        offs.append(len(payload))
        seg = [int(x) for x in words[w * window:(w + 1) * window]]
        i = 0
        while i < len(seg):
            z = 0
            while i < len(seg) and seg[i] == 0:
                z, i = z + 1, i + 1
            lit = []
            while i < len(seg) and seg[i] != 0:
                lit.append(seg[i])
                i += 1
            payload += struct.pack("<HH", z, len(lit)) + b"".join(struct.pack("<I", v) for v in lit)
    head = struct.pack("<IHHIIQQ", 0x31454C52, 1, 4, window, 0, n, len(payload))
    return head + b"".join(struct.pack("<Q", o) for o in offs) + bytes(payload)


def brute_decode(stream, n, window):
    """Returns the words, or None if the stream is not valid for (n, window)."""
    s = bytes(stream)
    if len(s) < 32:
        return None
    magic, ver, wb, win, res, nn, payload = struct.unpack_from("<IHHIIQQ", s, 0)
    nw = -(-n // window)
    if (magic, ver, wb, win, res, nn) != (0x31454C52, 1, 4, window, 0, n):
        return None
    if len(s) < 32 + 8 * nw or len(s) - 32 - 8 * nw != payload:
        return None
    offs = list(struct.unpack_from(f"<{nw}Q", s, 32)) + [payload]
    base = 32 + 8 * nw
    out = []
    for w in range(nw):
        a, b = offs[w], offs[w + 1]
        if (w == 0 and a != 0) or a > b or b > payload or (a | b) % 4:
            return None
        length = min(window, n - w * window)
        got, pos = [], base + a
        while len(got) < length:
            if pos + 4 > base + b:
                return None
            z, lit = struct.unpack_from("<HH", s, pos)
            pos += 4
            if z + lit == 0 or z + lit > length - len(got) or pos + 4 * lit > base + b:
                return None
            got += [0] * z + list(struct.unpack_from(f"<{lit}I", s, pos))
            pos += 4 * lit
        if pos != base + b:
            return None
        out += got
    return np.array(out, dtype=np.uint32)


def closed_form(words, window):
    w = np.asarray(words, dtype=np.uint32)
    n = w.size
    nw = -(-n // window)
    nz = w != 0
    idx = np.arange(n)
    # a record starts at each window's first word and at each zero after a non-zero in the
    # same window
    trans = int(np.sum((~nz[1:]) & nz[:-1] & (idx[1:] % window != 0))) if n > 1 else 0
    return 32 + 8 * nw + 4 * (nw + trans) + 4 * int(nz.sum())


def _random_words(rng, n, density, clustered):
    if clustered:  # runs: alternate zero and non-zero runs of random lengths
        w, i, on = np.zeros(n, dtype=np.uint32), 0, rng.random() < density
        while i < n:
            k = int(rng.integers(1, 40))
            if on:
                w[i:i + k] = rng.integers(1, 2**32, size=min(k, n - i), dtype=np.uint64)
            i += k
            on = not on
        return w
    keep = rng.random(n) < density
    return (rng.integers(1, 2**32, size=n, dtype=np.uint64) * keep).astype(np.uint32)


# ------------------------------------------------------------------ pins
@pytest.mark.parametrize("name", golden_io.all_rle())
def test_hand_derived_bytes(name):
    g = golden_io.load_rle(name)
    got = oracle.rle_encode(g["input"], g["window"])
    assert got.tobytes() == g["expected"]
    st, back = oracle.rle_decode(np.frombuffer(g["expected"], np.uint8), g["n"], g["window"])
    assert st == oracle.OK and np.array_equal(back, g["input"])


@pytest.mark.parametrize("window", [32, 64, 96, 1024])
def test_brute_force_agrees_on_small_inputs(window):
    rng = np.random.default_rng(window)
    for n in list(range(0, 70)) + [127, 128, 129, 300, 1025, 2100]:
        for density in (0.0, 0.3, 0.7, 1.0):
            for clustered in (False, True):
                w = _random_words(rng, n, density, clustered)
                got = oracle.rle_encode(w, window)
                assert got.tobytes() == brute_encode(w, window), (n, density, clustered)
                assert got.size == closed_form(w, window)
                assert got.size <= oracle.rle_size_bound(n, window)
                st, back = oracle.rle_decode(got, n, window)
                assert st == oracle.OK and np.array_equal(back, w)


def test_alternating_window_meets_the_bound():
    w = np.zeros(1024, dtype=np.uint32)
    w[0::2] = 7  # N Z N Z ...: a record per non-zero
    assert oracle.rle_encode(w, 1024).size == oracle.rle_size_bound(1024, 1024)


def test_signed_zero_nan_and_denormals_are_payload():
    w = np.array([0x80000000, 0, 0x7FC00000, 0, 1], dtype=np.uint32)
    s = oracle.rle_encode(w, 32)
    assert s.size == closed_form(w, 32) == 32 + 8 + 4 * 3 + 4 * 3
    st, back = oracle.rle_decode(s, 5, 32)
    assert st == oracle.OK and np.array_equal(back, w)


def test_layout_moves_rle_but_not_zvc():
    """The pages' finding: the same values in another order change RLE's size, not ZVC's."""
    rng = np.random.default_rng(3)
    c, h, w = 16, 32, 32
    # clustered along the spatial axes (NCHW-contiguous blobs)
    x = np.zeros((c, h, w), dtype=np.uint32)
    for k in range(c):
        r0, c0 = rng.integers(0, h - 12), rng.integers(0, w - 12)
        x[k, r0:r0 + 12, c0:c0 + 12] = rng.integers(1, 2**32, size=(12, 12), dtype=np.uint64)
    nchw = x.reshape(-1)
    nhwc = np.ascontiguousarray(x.transpose(1, 2, 0)).reshape(-1)
    assert oracle.encode(nchw, 1024).size == oracle.encode(nhwc, 1024).size
    r_nchw, r_nhwc = oracle.rle_encode(nchw, 1024).size, oracle.rle_encode(nhwc, 1024).size
    assert r_nchw < r_nhwc  # long runs in NCHW rows, short runs across channels
    assert r_nchw == closed_form(nchw, 1024) and r_nhwc == closed_form(nhwc, 1024)


def test_corruption_verdicts_match_the_brute_force_decoder():
    rng = np.random.default_rng(9)
    w = _random_words(rng, 700, 0.5, True)
    s = oracle.rle_encode(w, 64)
    for _ in range(300):
        bad = s.copy()
        i = int(rng.integers(0, bad.size))
        bad[i] ^= np.uint8(1 << int(rng.integers(0, 8)))
        st, back = oracle.rle_decode(bad, 700, 64)
        ref = brute_decode(bad, 700, 64)
        if ref is None:
            assert st == oracle.ERR_CORRUPT, i
        else:
            assert st == oracle.OK and np.array_equal(back, ref), i
    assert oracle.rle_decode(s[:-1], 700, 64)[0] == oracle.ERR_CORRUPT
    assert oracle.rle_decode(s, 701, 64)[0] == oracle.ERR_CORRUPT
    assert oracle.rle_decode(s, 700, 32)[0] == oracle.ERR_CORRUPT


MUTANTS = {
    "runs cross windows": ("const uint64_t end = begin + window < n ? begin + window : n;\n    uint64_t i = begin;\n    while (i < end) {  /* one record per iteration */",
                           "const uint64_t end = n;\n    uint64_t i = begin;\n    while (i < end && i < begin + window) {  /* one record per iteration */"),
    "sign-insensitive zero": ("while (i < end && x[i] == 0) {", "while (i < end && (x[i] & 0x7FFFFFFFu) == 0) {"),
    "table from stream start": ("put_u64(out + 32 + 8 * w, pos - payload_at);", "put_u64(out + 32 + 8 * w, pos);"),
    "counts swapped": ("put_u16(out + head, (uint16_t)zeros);\n      put_u16(out + head + 2, (uint16_t)literals);",
                       "put_u16(out + head, (uint16_t)literals);\n      put_u16(out + head + 2, (uint16_t)zeros);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_a_mutated_oracle(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._RLE_SRC).read()
    a, b = MUTANTS[name]
    assert src.count(a) == 1, name
    path = tmp_path / "m.c"
    path.write_text(src.replace(a, b))
    lib_path = str(tmp_path / "libm.so")
    oracle.build(str(path), lib_path)
    lib = oracle.rle_load(lib_path)
    caught = False
    for gname in golden_io.all_rle():
        g = golden_io.load_rle(gname)
        try:
            caught |= oracle.rle_encode(g["input"], g["window"], lib=lib).tobytes() != g["expected"]
        except oracle.OracleError:
            caught = True
    w = np.array([0x80000000, 0, 5, 0, 0, 6] * 20, dtype=np.uint32)
    try:
        caught |= oracle.rle_encode(w, 32, lib=lib).tobytes() != brute_encode(w, 32)
    except oracle.OracleError:
        caught = True
    assert caught, name
