"""Seeded synthetic activation maps (post-ReLU fp32), shared by tests and the benchmark.

The activations of the ImageNet CNNs in Rhu et al., "Compressing DMA Engine" (section
VI set-up: AlexNet, OverFeat, NiN, VGG, SqueezeNet, GoogLeNet) need datasets and trained
weights that are not available here, so these generators stand in for them with the
shapes and non-zero densities the paper reports (section IV: roughly 50% to 90% zeros,
49.4% average sparsity for AlexNet, up to 93%). Nothing in this module encodes or
decodes anything; it only draws numbers.

Every generator takes ``device``: on a GPU the draws come from a seeded CUDA generator,
on the CPU from a seeded CPU generator. The two give different values for the same
seed; parity tests therefore copy the device tensor to the host before handing it to
the oracle. A ``batch`` argument shrinks the batch dimension (keeping the per-element
distribution) so that CPU runs stay small.
"""
from __future__ import annotations

from dataclasses import dataclass
from statistics import NormalDist

import numpy as np
import torch

CHUNK_ELEMS = 4096
_PHI_INV = NormalDist().inv_cdf


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def _randn(shape, device, g):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


# ---------------------------------------------------------------- config 1
def single_relu(device="cuda", seed: int = 0):
    """1x64x56x56 ReLU(x), x ~ N(0,1) i.i.d.: about half the words are zero."""
    g = _gen(device, seed)
    return [torch.relu_(_randn((1, 64, 56, 56), device, g))]


# ---------------------------------------------------------------- config 2
ALEXNET_LAYERS = [  # (C, H, W, non-zero density)
    (96, 55, 55, 0.60),
    (256, 27, 27, 0.45),
    (384, 13, 13, 0.35),
    (384, 13, 13, 0.30),
    (256, 13, 13, 0.20),
]


def alexnet_biases(c: int, d: float, seed: int):
    """Per-channel biases of one layer: b_c = mu + 0.5 * Phi^-1((p(c) + 0.5) / C) with p a
    seeded permutation of the channels and mu = sqrt(1.25) * Phi^-1(d). The biases are the
    C mid-quantiles of N(mu, 0.5^2), so the channel average of Phi(b_c), the layer's
    non-zero fraction, is E[Phi(mu + 0.5 Z)] = Phi(mu / sqrt(1.25)) = d up to the
    midpoint-rule error, while each channel keeps its own density."""
    rng = np.random.default_rng(seed)
    mu = (1.25 ** 0.5) * _PHI_INV(d)
    q = [(k + 0.5) / c for k in rng.permutation(c)]
    return [mu + 0.5 * _PHI_INV(v) for v in q]


def alexnet_stack(device="cuda", batch: int = 128, seed: int = 1):
    """Five AlexNet conv activations ReLU(x + b_c), x ~ N(0,1), with the per-channel
    biases of alexnet_biases (layer l draws from seed + l)."""
    out = []
    for l, (c, h, w, d) in enumerate(ALEXNET_LAYERS):
        g = _gen(device, seed + l)
        b = torch.tensor(alexnet_biases(c, d, seed + l), dtype=torch.float32,
                         device=device).view(1, c, 1, 1)
        x = _randn((batch, c, h, w), device, g)
        out.append(torch.relu_(x.add_(b)))
    return out


# ---------------------------------------------------------------- config 3
def vgg_conv12(device="cuda", batch: int = 64, seed: int = 2):
    """64x64x224x224: a 5x5 box blur (zero padded, divide by 25) of N(0,1) per plane,
    then ReLU(z - t) with t = 0.2 * Phi^-1(0.65): in the interior z ~ N(0, 1/25), so about
    35% of the words are non-zero, in spatially clustered blobs."""
    g = _gen(device, seed)
    x = _randn((batch * 64, 1, 224, 224), device, g)
    z = torch.nn.functional.avg_pool2d(x, 5, stride=1, padding=2, count_include_pad=True)
    del x
    t = 0.2 * _PHI_INV(0.65)
    return [torch.relu_(z.sub_(t)).view(batch, 64, 224, 224)]


# ---------------------------------------------------------------- config 4
SWEEP_DENSITIES = [0.0, 0.01, 0.05, 0.10, 0.25, 0.50, 0.75, 0.90, 1.0]
SWEEP_N = 1 << 28


def density_sweep(density: float, structure: str, device="cuda", n: int = SWEEP_N,
                  seed: int = 3):
    """Flat buffer of n words with non-zero fraction ``density``. ``iid``: each word is
    non-zero with probability d. ``block``: each aligned 1024-word block is entirely
    non-zero with probability d, else entirely zero. Non-zero values are |N(0,1)| with
    any value whose bits are all zero replaced by 1.0, so that the drawn mask is exact."""
    g = _gen(device, seed)
    v = _randn((n,), device, g).abs_()
    v[v == 0] = 1.0
    if structure == "iid":
        keep = torch.rand((n,), generator=g, device=device) < density
    elif structure == "block":
        nb = -(-n // 1024)
        keep = (torch.rand((nb,), generator=g, device=device) < density)
        keep = keep.repeat_interleave(1024)[:n]
    else:
        raise ValueError(structure)
    return [v.mul_(keep)]


# ---------------------------------------------------------------- config 5
GOOGLENET_STAGES = [  # (spatial size, tensor count, channel choices)
    (112, 3, [64]),
    (56, 9, [64, 128, 192]),
    (28, 15, list(range(128, 481, 32))),
    (14, 20, list(range(160, 833, 32))),
    (7, 10, list(range(256, 1025, 32))),
]


@dataclass
class TensorSpec:
    shape: tuple
    density: float


def googlenet_specs(batch: int = 256, seed: int = 4):
    """The 57-tensor shape list: per tensor, draw its channel count uniformly from its
    stage's choices, then its density uniformly in [5%, 60%], both from
    numpy.random.default_rng(seed), in stage order."""
    rng = np.random.default_rng(seed)
    specs = []
    for hw, count, choices in GOOGLENET_STAGES:
        for _ in range(count):
            c = int(rng.choice(choices))
            d = float(rng.uniform(0.05, 0.60))
            specs.append(TensorSpec((batch, c, hw, hw), d))
    return specs


def googlenet_batch(device="cuda", batch: int = 256, seed: int = 4):
    """57 tensors ReLU(x - Phi^-1(1 - d_i)), x ~ N(0,1); tensor i draws from seed*1000+i."""
    out = []
    for i, s in enumerate(googlenet_specs(batch, seed)):
        g = _gen(device, seed * 1000 + i)
        x = _randn(s.shape, device, g)
        out.append(torch.relu_(x.sub_(_PHI_INV(1.0 - s.density))))
    return out


# ---------------------------------------------------------------- odd sizes
ODD_SIZES = [1, 31, 33, 4095, 4097, 1_000_003]


def odd_case(n: int, device="cuda", seed: int = 5, density: float = 0.5):
    """A flat ReLU(x - Phi^-1(1-d)) buffer of n words with -0.0, NaN and a denormal
    planted at fixed positions when they fit (all three are non-zero bit patterns)."""
    g = _gen(device, seed + n)
    x = torch.relu_(_randn((n,), device, g).sub_(_PHI_INV(1.0 - density)))
    w = x.view(torch.int32)
    for pos, bits in ((n // 3, -2**31), (n // 2, 0x7FC00000), (n - 1, 1)):
        if 0 <= pos < n:
            w[pos] = bits
    return [x]


CONFIGS = {
    "single_relu": single_relu,
    "alexnet_stack": alexnet_stack,
    "vgg_conv12": vgg_conv12,
    "googlenet_batch": googlenet_batch,
}
