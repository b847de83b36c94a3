"""The five benchmark workloads at full size on the GPU.

Every stream is compared with the oracle byte for byte: the single ReLU map, the AlexNet
stack, the VGG conv1_2 map, every case of the 1 GiB density sweep and all 57 streams of
the GoogLeNet batch (with the batch's header and offset table). Each is also checked by
properties that hold at any size (closed-form size, header, chunk table against
per-chunk non-zero counts) and by a bit-exact round trip through the GPU decoder. The
oracle encodes independent tensors on a thread pool (its calls release the GIL).
"""
import concurrent.futures
import os
import struct

import numpy as np
import pytest
import torch

import activation_sparsity_compression_gb300 as zvc
import oracle
import workloads
from tests.gpu_util import ensure_lib, sh, words_of

pytestmark = pytest.mark.gpu
C = 4096


def _compress(x, chunk_elems=C):
    ensure_lib()
    n = x.numel()
    cap = zvc.zvc_size_bound(n, chunk_elems)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_workspace_size(n, chunk_elems))
    assert zvc.zvc_compress(x.data_ptr(), n, chunk_elems, out.data_ptr(), cap, size.data_ptr(),
                            ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    return out[:int(size.item())]


def _decompress_equal(stream_dev, x, chunk_elems=C):
    y = torch.empty_like(x)
    ws = zvc.new_workspace(256)
    assert zvc.zvc_decompress(stream_dev.data_ptr(), stream_dev.numel(), y.data_ptr(), x.numel(),
                              chunk_elems, ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert torch.equal(y.view(torch.int32), x.view(torch.int32))


def check_device_stream(stream, x, chunk_elems, samples, seed=0):
    """Property checks and sampled oracle chunks for a stream held on the device."""
    n = x.numel()
    w = x.reshape(-1).view(torch.int32)
    nc = -(-n // chunk_elems)
    nz = w != 0
    nnz = int(nz.sum())
    assert stream.numel() == 32 + 8 * nc + 4 * (-(-n // 32)) + 4 * nnz
    hdr = stream[:32].cpu().numpy().tobytes()
    payload_start = 32 + 8 * nc
    assert hdr == struct.pack("<IHHIIQQ", 0x3143565A, 1, 4, 32, chunk_elems, n,
                              stream.numel() - payload_start)
    offs = stream[32:payload_start].cpu().numpy().view("<u8").astype(np.int64)
    full = (n // chunk_elems) * chunk_elems
    per = nz[:full].view(-1, chunk_elems).sum(1, dtype=torch.int64) * 4 + 4 * (chunk_elems // 32)
    if full < n:
        t = nz[full:]
        per = torch.cat([per, torch.tensor([4 * (-(-t.numel() // 32)) + 4 * int(t.sum())],
                                           device=per.device)])
    expect = torch.cumsum(per, 0) - per
    assert np.array_equal(offs, expect.cpu().numpy())
    rng = np.random.default_rng(seed)
    picks = set(rng.integers(0, nc, size=min(samples, nc)).tolist()) | {0, nc - 1}
    ends = np.append(offs[1:], stream.numel() - payload_start)
    for c in sorted(picks):
        chunk_words = w[c * chunk_elems:(c + 1) * chunk_elems].cpu().numpy().view(np.uint32)
        ref = oracle.encode(chunk_words, chunk_elems)[40:]
        got = stream[payload_start + offs[c]:payload_start + ends[c]].cpu().numpy()
        assert got.tobytes() == ref.tobytes(), f"chunk {c}"


def test_alexnet_stack_full_bytes():
    for l, x in enumerate(workloads.alexnet_stack(device="cuda")):
        s = _compress(x)
        ref = oracle.encode(words_of(x), C)
        assert np.array_equal(s.cpu().numpy(), ref), l
        _decompress_equal(s, x)
        d = workloads.ALEXNET_LAYERS[l][3]
        assert abs(float((x != 0).float().mean()) - d) < 0.003  # the layer's stated density


def test_vgg_conv12_full_bytes_and_host_round_trip():
    x = workloads.vgg_conv12(device="cuda")[0]
    s = _compress(x)
    w = words_of(x)
    ref = oracle.encode(w, C)
    assert np.array_equal(s.cpu().numpy(), ref)
    ratio = 4 * x.numel() / s.numel()
    assert 2.4 < ratio < 2.9  # about 35% non-zero in blobs
    # compress -> pinned host -> prefetch -> decompress, the configuration's full pipeline
    n = x.numel()
    cap = zvc.zvc_offload_host_bound(n, C)
    h = torch.empty(cap, dtype=torch.uint8, pin_memory=True)
    ws = zvc.new_workspace(zvc.zvc_offload_workspace_size(n, C))
    st, size = zvc.zvc_offload(x.data_ptr(), n, C, h.data_ptr(), cap, ws.data_ptr(), ws.numel(), sh())
    assert st == zvc.ZVC_OK
    y = torch.empty(n, dtype=torch.int32, device="cuda")
    assert zvc.zvc_prefetch(h.data_ptr(), size, y.data_ptr(), n, C, ws.data_ptr(), ws.numel(),
                            sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    assert torch.equal(y, x.view(-1).view(torch.int32))


RATIO_4096 = {0.0: 31.5, 0.01: 24.0, 0.05: 12.2, 0.10: 7.59, 0.25: 3.55, 0.50: 1.88,
              0.75: 1.28, 0.90: 1.07, 1.0: 0.969}


@pytest.mark.parametrize("structure", ["iid", "block"])
@pytest.mark.parametrize("density", workloads.SWEEP_DENSITIES)
def test_density_sweep_full(density, structure):
    x = workloads.density_sweep(density, structure, device="cuda")[0]
    s = _compress(x)
    check_device_stream(s, x, C, samples=4, seed=int(density * 100))
    ref = oracle.encode(words_of(x), C)  # the whole 1 GiB map, every byte
    assert np.array_equal(s.cpu().numpy(), ref)
    del ref
    _decompress_equal(s, x)
    if structure == "iid":
        assert abs(4 * x.numel() / s.numel() / RATIO_4096[density] - 1) < 0.01


def test_googlenet_batch_full():
    ensure_lib()
    xs = workloads.googlenet_batch(device="cuda")
    assert len(xs) == 57
    ns = [x.numel() for x in xs]
    cap = zvc.zvc_batch_size_bound(ns, C)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    ws = zvc.new_workspace(zvc.zvc_batch_workspace_size(ns, C))
    assert zvc.zvc_compress_batched([x.data_ptr() for x in xs], ns, C, out.data_ptr(), cap,
                                    size.data_ptr(), ws.data_ptr(), ws.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(ws.data_ptr(), sh()) == zvc.ZVC_OK
    total = int(size.item())
    T = len(xs)
    head = out[:16 + 8 * (T + 1)].cpu().numpy().tobytes()
    magic, t, tot = struct.unpack_from("<IIQ", head, 0)
    assert (magic, t, tot) == (0x4243565A, T, total)
    offs = struct.unpack_from(f"<{T + 1}Q", head, 16)
    assert offs[0] == 16 + 8 * (T + 1) and offs[-1] == total
    for i, x in enumerate(xs):
        check_device_stream(out[offs[i]:offs[i + 1]], x, C, samples=1, seed=i)
    # every byte of the batch against the oracle: stream i at offs[i] is the oracle's
    # encoding of tensor i, so the offset table is the prefix of the oracle's sizes
    workers = max(1, min(16, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        pending = {}
        for i, x in enumerate(xs):
            pending[i] = pool.submit(oracle.encode, words_of(x), C)
            if len(pending) >= workers or i == T - 1:
                for j in sorted(pending):
                    ref = pending.pop(j).result()
                    assert offs[j + 1] - offs[j] == ref.size, j
                    got = out[offs[j]:offs[j + 1]].cpu().numpy()
                    assert np.array_equal(got, ref), f"tensor {j}"
    ys = [torch.empty_like(x) for x in xs]
    wsd = zvc.new_workspace(256)
    assert zvc.zvc_decompress_batched(out.data_ptr(), total, [y.data_ptr() for y in ys], ns, C,
                                      wsd.data_ptr(), wsd.numel(), sh()) == zvc.ZVC_OK
    assert zvc.zvc_get_error(wsd.data_ptr(), sh()) == zvc.ZVC_OK
    for x, y in zip(xs, ys):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
