"""Offload / prefetch (Rhu et al., "Compressing DMA Engine", section V.D: activations are
offloaded to host memory in forward propagation and prefetched before backward
propagation with cudaMemcpyAsync; cDMA compresses them on the way). The pinned host
buffer must hold exactly the batch the oracle builds over the same segments, and the
prefetch must restore the tensor bit for bit."""
import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests.gpu_util import ensure_lib, sh, words_of

pytestmark = pytest.mark.gpu


def _offload(x, C):
    ensure_lib()
    n = x.numel()
    cap = zvc.zvc_offload_host_bound(n, C)
    h = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    ws = zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C))
    st, size = zvc.zvc_offload(x.data_ptr(), n, C, h.data_ptr(), cap, ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    torch.cuda.synchronize()
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    return h, size, ws


def _prefetch(h, size, n, C, ws):
    y = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    st = zvc.zvc_prefetch(h.data_ptr(), size, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    return y


@pytest.mark.parametrize("n", [1, 4097, 1_000_003, 5_000_000, 9_437_184 + 11])
def test_offload_equals_oracle_batch_and_prefetch_restores(n):
    C = 4096
    x = workloads.odd_case(n, device="cuda", density=0.4)[0]
    h, size, ws = _offload(x, C)
    w = words_of(x)
    seg = zvc.zvc_offload_segment_elems(n, C)
    segs = [w[k:k + seg] for k in range(0, n, seg)]
    ref = oracle.encode_batch(segs, C)
    assert size == ref.size
    assert np.array_equal(h[:size].numpy(), ref)
    y = _prefetch(h, size, n, C, ws)
    assert torch.equal(y, x.view(torch.int32))


def test_offload_empty_tensor():
    h, size, ws = _offload(torch.empty(0, dtype=torch.float32, device="cuda"), 4096)
    assert np.array_equal(h[:size].numpy(), oracle.encode_batch([], 4096))
    _prefetch(h, size, 0, 4096, ws)


def test_prefetch_rejects_a_bad_table_on_the_host():
    n, C = 3_000_000, 4096
    x = workloads.odd_case(n, device="cuda", density=0.3)[0]
    h, size, ws = _offload(x, C)
    y = torch.empty(n, dtype=torch.int32, device="cuda")
    for off in (0, 4, 8, 16, 24):
        bad = h.clone().pin_memory()
        bad[off] ^= 1
        assert zvc.zvc_prefetch(bad.data_ptr(), size, y.data_ptr(), n, C, ws.data_ptr(),
                                ws.numel(), sh()) == zvc.ZVC_ERR_CORRUPT


def test_prefetch_latches_corrupt_segment():
    n, C = 3_000_000, 4096
    x = workloads.odd_case(n, device="cuda", density=0.3)[0]
    h, size, ws = _offload(x, C)
    seg0 = int(np.frombuffer(h[16:24].numpy().tobytes(), "<u8")[0])
    bad = h.clone().pin_memory()
    bad[seg0 + 32 + 8 * 10] ^= 0x10  # chunk_off[10] of the first segment, off by 16 bytes
    y = torch.empty(n, dtype=torch.int32, device="cuda")
    assert zvc.zvc_prefetch(bad.data_ptr(), size, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(),
                            sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_ERR_CORRUPT


def test_offload_join_makes_the_host_batch_complete_on_the_callers_stream():
    ensure_lib()
    n, C = 5_000_000, 4096
    x = workloads.odd_case(n, device="cuda", density=0.4)[0]
    cap = zvc.zvc_offload_host_bound(n, C)
    h = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    ws = zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    st, size = zvc.zvc_offload(x.data_ptr(), n, C, h.data_ptr(), cap, ws.data_ptr(), ws.numel(),
                               s.cuda_stream)
    assert st == zvc.ZVC_OK
    assert zvc.zvc_offload_join(s.cuda_stream) == zvc.ZVC_OK
    s.synchronize()  # this stream only: the join put the copies on it
    seg = zvc.zvc_offload_segment_elems(n, C)
    w = words_of(x)
    ref = oracle.encode_batch([w[k:k + seg] for k in range(0, n, seg)], C)
    assert size == ref.size
    assert np.array_equal(h[:size].numpy(), ref)


def test_offload_rejects_a_host_buffer_off_8_byte_alignment():
    ensure_lib()
    n, C = 100_000, 4096
    x = workloads.odd_case(n, device="cuda")[0]
    cap = zvc.zvc_offload_host_bound(n, C)
    h = torch.empty(cap + 8, dtype=torch.uint8, pin_memory=True)
    ws = zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C))
    st, _ = zvc.zvc_offload(x.data_ptr(), n, C, h.data_ptr() + 4, cap, ws.data_ptr(), ws.numel(),
                            sh())
    assert st == zvc.ZVC_ERR_INVALID_ARG
