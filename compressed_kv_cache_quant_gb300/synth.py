"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

Random numbers and workload shapes only: nothing here computes any step of
the method.  Every tensor comes from a torch.Generator seeded from
(BASE_SEED + config id, tensor id...), so the same call gives the same bytes
on the same device type.  The CPU oracle and the GPU library receive the
same bytes (the oracle a host copy of what the GPU got).

Distributions (the workloads' stated shapes): K, V ~ N(0, 1) fp16; per
(layer, kv head) four seeded K channels scaled by 10 (outlier channels);
queries ~ N(0, 1) fp16, fresh per step.  No public dataset is used.
"""
from __future__ import annotations

import torch

BASE_SEED = 0xC0FFEE
MASK64 = (1 << 64) - 1


def mix(*ids):
    """A 63-bit seed from a tuple of integers (splitmix64 folding)."""
    s = 0x9E3779B97F4A7C15
    for v in ids:
        s = (s + (int(v) & MASK64) + 0x9E3779B97F4A7C15) & MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        s = z ^ (z >> 31)
    return s & ((1 << 63) - 1)


def generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed, device="cpu", scale=1.0, dtype=torch.float16):
    g = generator(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def outlier_channels(seed, n_kv, n_out=4, d=128):
    """Seeded outlier channel ids per kv head (a [n_kv][n_out] int64 tensor)."""
    g = generator(seed, "cpu")
    return torch.stack([torch.randperm(d, generator=g)[:n_out] for _ in range(n_kv)])


def kv_rows(T, n_kv, seed, device="cpu", n_out=4, factor=10.0, d=128):
    """K, V fp16 [T][n_kv][d] ~ N(0,1); K's outlier channels scaled by `factor`."""
    K = normal((T, n_kv, d), mix(seed, 1), device, dtype=torch.float32)
    if n_out:
        ch = outlier_channels(mix(seed, 3), n_kv, n_out, d)
        for h in range(n_kv):
            K[:, h, ch[h].to(device)] *= factor
    V = normal((T, n_kv, d), mix(seed, 2), device)
    return K.to(torch.float16), V


def queries(shape, seed, device="cpu"):
    return normal(shape, mix(seed, 4), device)


def h2o_hot_positions(seed, T, n_hot=64):
    """Hot key positions and Zipf(1.2) weights for power-law query affinity."""
    g = generator(mix(seed, 5), "cpu")
    pos = torch.randperm(T, generator=g)[:n_hot]
    w = torch.arange(1, n_hot + 1, dtype=torch.float64) ** -1.2
    return pos, w / w.sum()


def h2o_queries(K_hot_rows, w, n_q, seed, device="cpu", n_pick=4, gain=2.0, noise=0.5):
    """q_h = gain * mean(K[hot picks]) + noise * N(0,1): queries with a
    power-law preference for a few hot keys (heavy hitters).
    K_hot_rows: [n_hot][d] fp16 rows of the hot positions."""
    g = generator(mix(seed, 6), "cpu")
    d = K_hot_rows.shape[-1]
    out = torch.empty((n_q, d), dtype=torch.float32)
    for i in range(n_q):
        pick = torch.multinomial(w, n_pick, replacement=True, generator=g)
        out[i] = gain * K_hot_rows[pick].float().mean(0)
    out += noise * torch.randn((n_q, d), generator=g)
    return out.to(torch.float16).to(device)


def lengths_uniform(B, lo, hi, seed):
    """B sequence lengths drawn uniformly from [lo, hi]."""
    g = generator(mix(seed, 7), "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g)


def h2o_query_bank(K_hot, n_q, seed, n_pick=4, gain=2.0, noise=0.5, zipf=1.2):
    """The power-law queries of ``h2o_queries`` for many key sets at once.

    K_hot: fp16 [N][n_hot][d] rows of each set's hot positions (any device).
    Returns fp16 [N][n_q][d] on that device: every query averages n_pick hot rows
    drawn with Zipf(zipf) weights over the hot ranks, times gain, plus noise *
    N(0, 1).  Draws come from one generator (seeded by `seed`) on K_hot's device."""
    N, n_hot, d = K_hot.shape
    dev = K_hot.device
    g = generator(mix(seed, 8), dev)
    w = torch.arange(1, n_hot + 1, dtype=torch.float64, device=dev) ** -zipf
    cdf = torch.cumsum(w / w.sum(), 0)
    u = torch.rand((N, n_q * n_pick), generator=g, device=dev, dtype=torch.float64)
    picks = torch.searchsorted(cdf, u).clamp_(max=n_hot - 1)        # inverse-CDF draws of the hot ranks
    rows = torch.gather(K_hot.float(), 1, picks[..., None].expand(N, n_q * n_pick, d))
    q = gain * rows.view(N, n_q, n_pick, d).mean(2)
    q += noise * torch.randn((N, n_q, d), generator=g, device=dev)
    return q.to(torch.float16)
