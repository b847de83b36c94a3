"""zvc_compress_static: compression for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their device memory is owned by a
manager that forbids side allocations, or they must avoid cudaMalloc because it
synchronises the device and fails once memory is fully reserved. zvc_compress_static
keeps its scratch in a static device array inside the library instead. Its output must
equal zvc_compress's byte for byte (compression is exact integer work) and the oracle's,
call after call, although every call reuses the same scratch. This file is named to be
collected last.
"""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests.gpu_util import ensure_lib, gpu_compress, sh, words_of

pytestmark = pytest.mark.gpu


def _static_compress(x, C):
    n = x.numel()
    cap = zvc.zvc_size_bound(n, C)
    out = torch.full((cap + 64,), 0xEE, dtype=torch.uint8, device=x.device)
    size = torch.zeros(1, dtype=torch.int64, device=x.device)
    st = zvc.zvc_compress_static(x.data_ptr(), n, C, out.data_ptr(), cap, size.data_ptr(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_compress_static_get_error(sh()) == zvc.ZVC_OK  # nothing latched
    s = int(size.item())
    host = out.cpu().numpy()
    assert (host[s:] == 0xEE).all()  # nothing written past the stream
    return host[:s]


@pytest.mark.parametrize("C", [32, 1024, 4096, 32768])
def test_static_scratch_matches_workspace_compress_on_consecutive_calls(C):
    ensure_lib()
    inputs = [workloads.odd_case(3_000_017, device="cuda", density=0.4)[0],
              workloads.odd_case(1_234_567, device="cuda", density=0.8)[0]]
    for x in inputs:  # two calls in a row, each through the shared static scratch
        st, ref, err = gpu_compress(x, C)
        assert st == zvc.ZVC_OK and err == zvc.ZVC_OK
        got = _static_compress(x, C)
        assert got.size == ref.size
        assert np.array_equal(got, ref)
        assert np.array_equal(got, oracle.encode(words_of(x), C))


def test_static_scratch_near_its_tile_capacity():
    """A map of ZVC_STATIC_MAX_ELEMS - 5 words fills all but the last of the scratch's
    tile status words; compressed twice in a row, each time equal to the oracle."""
    ensure_lib()
    C = 32768
    n = zvc.ZVC_STATIC_MAX_ELEMS - 5
    x = workloads.odd_case(n, device="cuda", density=0.1)[0]
    ref = oracle.encode(words_of(x), C)
    for _ in range(2):
        got = _static_compress(x, C)
        assert got.size == ref.size
        assert np.array_equal(got, ref)


def test_static_scratch_rejects_sizes_beyond_its_limit():
    ensure_lib()
    too_big = zvc.ZVC_STATIC_MAX_ELEMS + 1
    out_cap = zvc.zvc_size_bound(too_big, 4096)
    # rejected on the host before any device work, so the pointers are never touched
    assert zvc.zvc_compress_static(0x1000, too_big, 4096, 0x2000, out_cap, 0, sh()) == \
        zvc.ZVC_ERR_INVALID_ARG
