"""Seeded synthetic inputs with the shapes and distributions of the workloads.

This module only draws random numbers; it holds none of the quantisation or
attention arithmetic.  The tests feed the same tensors to the CUDA library and
to the CPU oracle, and the benchmark uses the same recipes at full size.

Recipes (one per workload):

* tiny decode: K, V, q fp32 ~ N(0, 1); per (tensor, head) four channels chosen
  at random are multiplied by 20 (outliers).
* heavy-tailed decode (32K / 262K contexts, batched paged decode, prefill):
  bf16 values where, per (layer, tensor, head), a seeded subset of 13 of 256
  channels (5 %) is Student-t(nu = 3) x 10 and the rest N(0, 1).  Student-t is
  drawn as Z / sqrt(chi2_3 / 3) with chi2_3 a sum of three squared normals.
* fp8 latent rows: 576 values (512 latent + 64 rope) ~ N(0, 1) times one
  log-normal(0, 1) magnitude per row; queries N(0, 1) fp32.
* ragged batch: lengths ~ Uniform{1024 .. 65536}; page ids a seeded
  permutation of all pages the batch needs.
"""
from __future__ import annotations

import hashlib

import torch


def sub_seed(*keys) -> int:
    """A stable 63-bit seed derived from a tuple of keys."""
    h = hashlib.sha256(repr(keys).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(device, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(*keys))
    return g


def outlier_normal(shape, n_out, scale, device, *keys):
    """fp32 N(0,1) with n_out seeded channels (last dim) per leading index of
    dim -2 multiplied by `scale`.  shape = (..., heads, D)."""
    g = generator(device, "outlier_normal", *keys)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    heads, D = shape[-2], shape[-1]
    for h in range(heads):
        ch = torch.randperm(D, generator=g, device=device)[:n_out]
        x[..., h, ch] *= scale
    return x


def heavy_tailed(shape, device, *keys, frac=0.05, nu=3, scale=10.0, dtype=torch.bfloat16, subset=None):
    """Values with 95 % N(0,1) channels and 5 % Student-t(nu) x scale channels.
    shape = (..., heads, D).  The heavy channel subset of each head is drawn from
    `subset` (a tuple of keys; default: the value keys), so a cache filled in
    chunks keeps one subset per (layer, tensor, head)."""
    g = generator(device, "heavy_tailed", *keys)
    gs = generator("cpu", "heavy_subset", *(subset if subset is not None else keys))
    heads, D = shape[-2], shape[-1]
    n_heavy = int(round(frac * D))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    lead = shape[:-2]
    for h in range(heads):
        ch = torch.randperm(D, generator=gs)[:n_heavy].to(device)
        z = torch.randn(lead + (n_heavy,), generator=g, device=device, dtype=torch.float32)
        chi = torch.zeros_like(z)
        for _ in range(nu):
            w = torch.randn(lead + (n_heavy,), generator=g, device=device, dtype=torch.float32)
            chi += w * w
        t = z / torch.sqrt(chi / nu)
        x[..., h, ch] = t * scale
    return x.to(dtype)


def latent_rows(n, width, device, *keys):
    """fp32 rows ~ N(0,1) * exp(N(0,1)), one log-normal magnitude per row."""
    g = generator(device, "latent_rows", *keys)
    x = torch.randn((n, width), generator=g, device=device, dtype=torch.float32)
    mag = torch.exp(torch.randn((n, 1), generator=g, device=device, dtype=torch.float32))
    return x * mag


def normal(shape, device, *keys, dtype=torch.float32):
    g = generator(device, "normal", *keys)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def ragged_lengths(n, lo, hi, *keys):
    """n integer lengths ~ Uniform{lo .. hi} (host tensor, int64)."""
    g = generator("cpu", "ragged_lengths", *keys)
    return torch.randint(lo, hi + 1, (n,), generator=g)


def page_permutation(n_pages, *keys):
    """A seeded permutation of page ids 0 .. n_pages-1 (host tensor, int64)."""
    g = generator("cpu", "page_permutation", *keys)
    return torch.randperm(n_pages, generator=g)


def distinct_sorted(n, upper, *keys):
    """n distinct integers from [0, upper), sorted ascending (host tensor, int64)."""
    g = generator("cpu", "distinct_sorted", *keys)
    return torch.sort(torch.randperm(upper, generator=g)[:n]).values


def sign_mask(n, *keys):
    """n random signs as a bit mask: [n / 32] int32 words, bit i of word i / 32 set
    with probability 1/2 (host tensor; the bits of each word are uniform)."""
    g = generator("cpu", "sign_mask", *keys)
    bits = torch.randint(0, 2, (n // 32, 32), generator=g, dtype=torch.int64)
    words = (bits << torch.arange(32, dtype=torch.int64)).sum(1)
    return torch.where(words >= 2**31, words - 2**32, words).to(torch.int32)
