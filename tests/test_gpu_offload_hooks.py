"""Activation offload during training (Rhu et al., "Compressing DMA Engine", section V.D:
vDNN offloads the maps a layer's backward pass needs and prefetches them before it; cDMA
compresses them on the way). ZVC is lossless, so a training step whose saved activations
went through the compress -> host (or HBM) -> decompress round trip must produce the very
same gradients, bit for bit, as one that kept them."""
import pytest
import torch

from activation_sparsity_compression_gb300.offload import ActivationOffload
from tests.gpu_util import ensure_lib

pytestmark = pytest.mark.gpu


def _cnn():
    torch.manual_seed(0)
    nn = torch.nn
    return nn.Sequential(
        nn.Conv2d(3, 32, 3, padding=1), nn.ReLU(),
        nn.Conv2d(32, 64, 3, padding=1), nn.ReLU(), nn.MaxPool2d(2),
        nn.Conv2d(64, 64, 3, padding=1), nn.ReLU(),
        nn.Flatten(), nn.Linear(64 * 32 * 32, 10)).cuda()


def _step(model, x, off):
    model.zero_grad(set_to_none=True)
    if off is None:
        loss = model(x).square().sum()
    else:
        with off:
            loss = model(x).square().sum()
    loss.backward()
    torch.cuda.synchronize()
    return [p.grad.clone() for p in model.parameters()]


@pytest.mark.parametrize("where", ["host", "device"])
def test_offloaded_activations_give_bit_identical_gradients(where):
    ensure_lib()
    torch.backends.cudnn.deterministic = True
    torch.backends.cudnn.benchmark = False
    model = _cnn()
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn(16, 3, 64, 64, device="cuda", generator=g)
    ref = _step(model, x, None)
    off = ActivationOffload(where=where, min_elems=1024)
    for _ in range(3):  # buffers and workspaces are reused across passes
        got = _step(model, x, off)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    off.check_errors()
    # at least the input image, the three ReLU outputs (each saved by the ReLU and by the
    # next layer, compressed once) and the pooled map went through the codec, every pass
    assert off.stats["packed"] >= 3 * 5
    assert off.stats["bytes_stored"] < off.stats["bytes_in"]  # post-ReLU maps compress


def test_retained_graph_can_be_unpacked_twice():
    ensure_lib()
    torch.backends.cudnn.deterministic = True
    torch.backends.cudnn.benchmark = False
    model = _cnn()
    x = torch.randn(4, 3, 64, 64, device="cuda")
    off = ActivationOffload(where="host", min_elems=1024)
    with off:
        loss = model(x).square().sum()
    loss.backward(retain_graph=True)
    first = [p.grad.clone() for p in model.parameters()]
    model.zero_grad(set_to_none=True)
    loss.backward()
    torch.cuda.synchronize()
    for a, p in zip(first, model.parameters()):
        assert torch.equal(a, p.grad)
    off.check_errors()


@pytest.mark.parametrize("max_pending", [0, 1, 4])
def test_worker_queue_depth_keeps_gradients_identical(max_pending):
    """Host mode offloads on a worker thread with at most max_pending tensors queued; the
    depth changes only how far the training loop runs ahead, never the result."""
    ensure_lib()
    torch.backends.cudnn.deterministic = True
    torch.backends.cudnn.benchmark = False
    model = _cnn()
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(8, 3, 64, 64, device="cuda", generator=g)
    ref = _step(model, x, None)
    off = ActivationOffload(where="host", min_elems=1024, max_pending=max_pending)
    for _ in range(2):
        got = _step(model, x, off)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    off.check_errors()
    off.close()
    assert off._worker is None


def test_worker_failure_surfaces_on_unpack():
    """An offload that fails on the worker thread raises when autograd unpacks the tensor,
    on the training loop's thread."""
    ensure_lib()
    model = _cnn()
    x = torch.randn(2, 3, 64, 64, device="cuda")
    off = ActivationOffload(where="host", min_elems=1024)

    def broken(h, t, produced, cap):
        raise RuntimeError("planted offload failure")

    off._offload_one = broken
    with off:
        loss = model(x).square().sum()
    with pytest.raises(RuntimeError, match="planted offload failure"):
        loss.backward()
    off.close()
