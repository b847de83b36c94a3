"""The C-ABI library builds for sm_103a, loads, and exports every function include/zvc.h
declares; its host-only size functions and argument checks work without a GPU (no
compute call is made here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import activation_sparsity_compression_gb300 as zvc
from activation_sparsity_compression_gb300 import build as zbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    zbuild.build()
    return zvc.lib()


def test_every_declared_function_is_exported(lib):
    names = zvc.header_functions()
    assert "zvc_compress" in names and "zvc_prefetch" in names and len(names) >= 16
    for name in names:
        assert hasattr(lib, name), name
        assert name in zvc._SIGS, f"binding lacks {name}"


def test_library_targets_sm103a():
    txt = open(os.path.join(ROOT, "activation_sparsity_compression_gb300", "build.py")).read()
    assert "arch=compute_103a,code=sm_103a" in txt


def test_size_bound_matches_closed_form_and_oracle(lib, oracle_lib):
    import oracle
    for n in (0, 1, 31, 32, 33, 4095, 4096, 4097, 200_704, 2**28, 3_030_000_000):
        for c in (32, 1024, 4096, 32768):
            expect = 32 + 8 * (-(-n // c)) + 4 * (-(-n // 32)) + 4 * n
            assert zvc.zvc_size_bound(n, c) == expect
            assert oracle.size_bound(n, c, lib=oracle_lib) == expect


def test_invalid_chunk_sizes_rejected(lib):
    for c in (0, 16, 33, 48 + 1, 32768 + 32, 2**31):
        assert zvc.zvc_size_bound(100, c) == 0
        assert zvc.zvc_workspace_size(100, c) == 0


def test_batch_bound_and_workspace(lib):
    ns = [0, 1, 5000, 4096 * 3]
    expect = 16 + 8 * 5 + sum(zvc.zvc_size_bound(n, 4096) for n in ns)
    assert zvc.zvc_batch_size_bound(ns, 4096) == expect
    ws = zvc.zvc_batch_workspace_size(ns, 4096)
    assert ws % 256 == 0 and ws >= 512 + 8 * (0 + 1 + 2 + 3) + 8 * 4
    assert zvc.zvc_batch_size_bound([1] * 513, 4096) == 0  # over ZVC_MAX_BATCH


def test_offload_plan_is_whole_chunks(lib):
    for n in (1, 4096, 8_306_688, 37_171_200, 205_520_896, 2**28):
        seg = zvc.zvc_offload_segment_elems(n, 4096)
        S = -(-n // seg)
        # ceil(n / 2^25) equal segments of whole chunks, the last one possibly shorter
        assert seg % 4096 == 0 and seg <= 1 << 25
        assert S == max(1, -(-n // (1 << 25))) and (S - 1) * seg < n <= S * seg
        bound = 16 + 8 * (S + 1) + sum(
            zvc.zvc_size_bound(min(seg, n - k * seg), 4096) for k in range(S))
        assert zvc.zvc_offload_host_bound(n, 4096) == bound
        assert zvc.zvc_offload_workspace_size(n, 4096) >= 3 * zvc.zvc_size_bound(min(seg, n), 4096)


def test_host_side_argument_checks_need_no_gpu(lib):
    # every one of these is rejected before any CUDA call
    ws = 0x10000
    assert zvc.zvc_compress(0x1000, 10, 33, 0x2000, 1 << 20, 0, ws, 1 << 20, 0) == zvc.ZVC_ERR_INVALID_ARG
    assert zvc.zvc_compress(0x1001, 10, 32, 0x2000, 1 << 20, 0, ws, 1 << 20, 0) == zvc.ZVC_ERR_INVALID_ARG
    assert zvc.zvc_compress(0x1000, 10, 32, 0x2000, 1 << 20, 0, ws + 8, 1 << 20, 0) == zvc.ZVC_ERR_INVALID_ARG
    assert zvc.zvc_compress(0x1000, 10, 32, 0x2000, 10, 0, ws, 1 << 20, 0) == zvc.ZVC_ERR_BUFFER_TOO_SMALL
    assert zvc.zvc_compress(0x1000, 10, 32, 0x2000, 1 << 20, 0, ws, 16, 0) == zvc.ZVC_ERR_BUFFER_TOO_SMALL
    # sizes no stream of n words can have are corrupt without reading the stream
    assert zvc.zvc_decompress(0x1000, 30, 0x2000, 10, 32, ws, 1 << 20, 0) == zvc.ZVC_ERR_CORRUPT
    assert zvc.zvc_decompress(0x1000, 43, 0x2000, 1, 32, ws, 1 << 20, 0) == zvc.ZVC_ERR_CORRUPT
    assert zvc.zvc_decompress(0x1000, 10_000, 0x2000, 10, 32, ws, 1 << 20, 0) == zvc.ZVC_ERR_CORRUPT
    assert zvc.zvc_selftest_wait_timeout(ws, 1 << 20, 0, 0) == zvc.ZVC_ERR_INVALID_ARG
    h = np.zeros(64, np.uint8)
    assert zvc.zvc_prefetch(h.ctypes.data, 64, 0x2000, 10, 32, ws, 1 << 30, 0) == zvc.ZVC_ERR_CORRUPT
    assert zvc.zvc_status_string(zvc.ZVC_ERR_CORRUPT) == "ZVC_ERR_CORRUPT"


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "activation_sparsity_compression_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "zvc_oracle" not in text and "zvco_" not in text, f


def test_offload_hooks_reject_an_unknown_placement():
    from activation_sparsity_compression_gb300.offload import ActivationOffload
    with pytest.raises(ValueError):
        ActivationOffload(where="disk")


def test_every_declaration_cites_its_passage():
    """The comment above each function declared in include/zvc.h names the paper's
    section it follows, or says that the paper has no counterpart."""
    text = open(zvc.HEADER_PATH).read()
    names = zvc.header_functions()
    for name in names:
        m = re.search(r"^(?:const\s+)?[a-z_0-9]+\s*\*?\s*" + name + r"\s*\(", text, re.M)
        assert m, name
        # the last comment block that opens a line above the declaration (a trailing
        # comment on a #define line is not one)
        blocks = [c for c in re.finditer(r"^/\*.*?\*/", text, re.M | re.S) if c.end() <= m.start()]
        comment = blocks[-1].group(0).lower()
        assert ("section" in comment) or ("no counterpart" in comment), name
