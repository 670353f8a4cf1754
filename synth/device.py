"""Seeded synthetic tensors generated directly on a CUDA device.

Used by the benchmark, whose full-size workloads (billions of weights) are
too large to draw on the host.  Each tensor has its own torch Generator keyed
by (seed, tags...) through the same tag hashing as generators.py; outlier
channels come from the host-side seeded shuffle, so a tensor's outlier set
does not depend on the device.  Values are drawn in float32 and rounded to
bf16 (round to nearest even).
"""
from __future__ import annotations

import numpy as np
import torch

from .generators import outlier_channels, sub_rng, _tag_int


def _gen(device, seed, *tags) -> torch.Generator:
    key = np.random.SeedSequence([int(seed) & 0xFFFFFFFF] + [_tag_int(t) for t in tags])
    g = torch.Generator(device=device)
    g.manual_seed(int(key.generate_state(1, dtype=np.uint64)[0] & 0x7FFFFFFFFFFFFFFF))
    return g


def activations(M, K, *, dist="normal", n_outliers=0, outlier_scale=1.0, seed=0, tags=(),
                device="cuda", out=None):
    g = _gen(device, seed, "dact", M, K, *tags)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if dist == "student_t4":
        # Student-t(4) = Z / sqrt(chi2_4 / 4), chi2_4 = -2 ln(U1 U2)
        u = torch.rand((2, M, K), generator=g, device=device, dtype=torch.float32).clamp_min_(1e-30)
        chi2 = -2.0 * torch.log(u[0] * u[1])
        x = x / torch.sqrt(chi2 / 4.0)
    elif dist != "normal":
        raise ValueError(dist)
    if n_outliers > 0:
        ch = outlier_channels(K, n_outliers, sub_rng(seed, "dact_out", M, K, *tags))
        x[:, torch.from_numpy(ch).to(device)] *= outlier_scale
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


def weights(N, K, *, std=0.02, spike_frac=0.0, spike_scale=1.0, seed=0, tags=(), device="cuda"):
    g = _gen(device, seed, "dw", N, K, *tags)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std
    if spike_frac > 0:
        mask = torch.rand((N, K), generator=g, device=device, dtype=torch.float32) < spike_frac
        w = torch.where(mask, w * spike_scale, w)
    return w.to(torch.bfloat16)
