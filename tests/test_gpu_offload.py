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


def test_offload_and_prefetch_from_two_threads_at_once():
    """An offload on one thread (its own stream and workspace) and prefetches of another
    tensor on a second thread run at the same time: the library's per-device lock is
    held only around its copy-stream enqueues, never while a call waits for a kernel.
    Every host batch equals the oracle's, every restored tensor is bit-exact."""
    import threading

    ensure_lib()
    C = 4096
    n_a, n_b = 70_000_011, 40_000_003  # 3 and 2 offload segments
    xa = workloads.odd_case(n_a, device="cuda", density=0.35)[0]
    xb = workloads.odd_case(n_b, device="cuda", density=0.55)[0]
    hb, size_b, ws_b = _offload(xb, C)
    cap_a = zvc.zvc_offload_host_bound(n_a, C)
    ha = [torch.empty(cap_a, dtype=torch.uint8, pin_memory=True) for _ in range(3)]
    ws_a = zvc.new_workspace(zvc.zvc_offload_workspace_size(n_a, C))
    ys = [torch.full((n_b,), -1, dtype=torch.int32, device="cuda") for _ in range(3)]
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    results = {}
    start = threading.Barrier(2)

    def offloader():
        torch.cuda.set_device(0)
        start.wait()
        out = []
        for h in ha:
            out.append(zvc.zvc_offload(xa.data_ptr(), n_a, C, h.data_ptr(), cap_a,
                                       ws_a.data_ptr(), ws_a.numel(), sa.cuda_stream))
        results["a"] = out

    def prefetcher():
        torch.cuda.set_device(0)
        start.wait()
        results["b"] = [zvc.zvc_prefetch(hb.data_ptr(), size_b, y.data_ptr(), n_b, C,
                                         ws_b.data_ptr(), ws_b.numel(), sb.cuda_stream)
                        for y in ys]

    threads = [threading.Thread(target=offloader), threading.Thread(target=prefetcher)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert zvc.zvc_offload_join(sa.cuda_stream) == zvc.ZVC_OK
    torch.cuda.synchronize()
    assert zvc.zvc_get_error(ws_a.data_ptr(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws_b.data_ptr(), sh()) == zvc.ZVC_OK
    assert all(st == zvc.ZVC_OK for st, _ in results["a"])
    assert all(st == zvc.ZVC_OK for st in results["b"])
    seg = zvc.zvc_offload_segment_elems(n_a, C)
    w = words_of(xa)
    ref = oracle.encode_batch([w[k:k + seg] for k in range(0, n_a, seg)], C)
    for h, (_, size) in zip(ha, results["a"]):
        assert size == ref.size
        assert np.array_equal(h[:size].numpy(), ref)
    for y in ys:
        assert torch.equal(y, xb.view(torch.int32))


def test_offload_of_more_segments_than_staging_buffers():
    """Five segments through three staging buffers, each reused: the batch equals the
    oracle's and restores bit for bit, and a second offload through the same workspace
    gives the same bytes."""
    C = 4096
    n = 4 * (1 << 25) + 12_345
    x = workloads.odd_case(n, device="cuda", density=0.1)[0]
    h, size, ws = _offload(x, C)
    seg = zvc.zvc_offload_segment_elems(n, C)
    assert -(-n // seg) == 5
    w = words_of(x)
    ref = oracle.encode_batch([w[k:k + seg] for k in range(0, n, seg)], C)
    assert size == ref.size
    assert np.array_equal(h[:size].numpy(), ref)
    y = _prefetch(h, size, n, C, ws)
    assert torch.equal(y, x.view(torch.int32))
    h2, size2, _ = _offload(x, C)
    assert size2 == size and torch.equal(h2[:size], h[:size])


@pytest.mark.parametrize("shift", [8, 16, 24])
def test_offload_and_prefetch_through_a_host_base_off_16_bytes(shift):
    """A host buffer at any 8-byte aligned base: the batch lands exactly in place and
    restores, and nothing outside it is written."""
    ensure_lib()
    C = 1024
    n = 2_000_003
    x = workloads.odd_case(n, device="cuda", density=0.45)[0]
    cap = zvc.zvc_offload_host_bound(n, C)
    buf = torch.full((cap + 64,), 0xAB, dtype=torch.uint8, pin_memory=True)
    ws = zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C))
    st, size = zvc.zvc_offload(x.data_ptr(), n, C, buf.data_ptr() + shift, cap, ws.data_ptr(),
                               ws.numel(), sh())
    assert st == zvc.ZVC_OK
    assert zvc.zvc_offload_join(sh()) == zvc.ZVC_OK  # the copies, on the library's stream
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    host = buf.numpy()
    assert (host[:shift] == 0xAB).all() and (host[shift + size:] == 0xAB).all()
    ref = oracle.encode_batch([words_of(x)], C)
    assert np.array_equal(host[shift:shift + size], ref)
    y = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    assert zvc.zvc_prefetch(buf.data_ptr() + shift, size, y.data_ptr(), n, C, ws.data_ptr(),
                            ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert torch.equal(y, x.view(torch.int32))


def test_prefetch_from_pageable_host_memory():
    """A batch in ordinary (pageable) host memory restores too, at either 8-byte phase."""
    C = 4096
    n = 40_000_003  # two segments
    x = workloads.odd_case(n, device="cuda", density=0.3)[0]
    h, size, ws = _offload(x, C)
    pageable = torch.empty(size + 4, dtype=torch.uint8)
    assert not pageable.is_pinned()
    for off in (0, 4):
        pageable[off:off + size] = h[:size]
        y = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        assert zvc.zvc_prefetch(pageable.data_ptr() + off, size, y.data_ptr(), n, C,
                                ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
        assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
        assert torch.equal(y, x.view(torch.int32))
