"""Parser for the hand-derived vectors in tests/golden (syntax in tests/golden/README.md)."""
import os
import re

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _parse_words(spec: str, n: int, dtype=np.uint32) -> np.ndarray:
    w = np.zeros(n, dtype=dtype)
    for tok in spec.split():
        i, v = tok.split("=")
        w[int(i)] = int(v, 16)
    return w


def load(name: str, directory: str = GOLDEN_DIR) -> dict:
    path = os.path.join(directory, name)
    keys = {}
    hex_bytes = []
    in_expected = False
    with open(path) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if in_expected:
                hex_bytes.extend(line.split())
                continue
            m = re.match(r"^([a-z_0-9]+):\s*(.*)$", line)
            if not m:
                raise ValueError(f"{name}: bad line {raw!r}")
            k, v = m.group(1), m.group(2)
            if k == "expected":
                in_expected = True
                if v:
                    hex_bytes.extend(v.split())
            else:
                keys[k] = v
    expected = bytes(int(b, 16) for b in hex_bytes)
    if "window" in keys:  # an RLE vector
        n = int(keys["n"])
        return {"name": name, "n": n, "window": int(keys["window"]),
                "input": _parse_words(keys.get("input", ""), n), "expected": expected}
    c = int(keys["chunk_elems"])
    if keys.get("word_bytes") == "2":  # a 16-bit ZVC vector
        n = int(keys["n"])
        return {"name": name, "n": n, "chunk_elems": c, "word_bytes": 2,
                "input": _parse_words(keys.get("input", ""), n, np.uint16), "expected": expected}
    if "batch" in keys:
        ns = [int(s) for s in keys["batch"].split(",")]
        inputs = [_parse_words(keys.get(f"input{k}", ""), n) for k, n in enumerate(ns)]
        return {"name": name, "batch": True, "ns": ns, "chunk_elems": c, "inputs": inputs,
                "expected": expected}
    n = int(keys["n"])
    return {"name": name, "batch": False, "n": n, "chunk_elems": c,
            "input": _parse_words(keys.get("input", ""), n), "expected": expected}


def all_single():
    return sorted(f for f in os.listdir(GOLDEN_DIR)
                  if f.endswith(".txt") and not load(f)["batch"])


def all_batch():
    return sorted(f for f in os.listdir(GOLDEN_DIR) if f.endswith(".txt") and load(f)["batch"])


RLE_DIR = os.path.join(GOLDEN_DIR, "rle")


def all_rle():
    return sorted(f for f in os.listdir(RLE_DIR) if f.endswith(".txt"))


def load_rle(name: str) -> dict:
    return load(name, RLE_DIR)


Z16_DIR = os.path.join(GOLDEN_DIR, "zvc16")


def all_z16():
    return sorted(f for f in os.listdir(Z16_DIR) if f.endswith(".txt"))


def load_z16(name: str) -> dict:
    return load(name, Z16_DIR)
