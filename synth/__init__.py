"""Seeded synthetic KV-cache inputs, shared by the tests, the benchmark and
the smoke check.  This module holds input generation only -- none of the
codec's arithmetic -- so the oracle and the CUDA library can both be fed
from it without sharing any method code.

Workload shapes follow the pages' settings (Llama-3.1-8B-like: 8 KV heads,
head_dim 128; Qwen2.5-7B-like: 28 layers x 4 KV heads) and the ablation
page's synthetic regimes (heavy-tailed Student-t marginals, low-rank spiked
covariance, outlier channels).  Every array is a pure function of its seed.

Generators:
  tiny_gaussian   zero-mean Gaussian, covariance Q diag(lam) Q^T,
                  lam_i = i^-1.5, Q random orthogonal (per head)
  spiked_t        rank-16 spiked covariance (strengths log-spaced 50 -> 5)
                  plus identity, 4 outlier channels scaled x20, multivariate
                  Student-t (nu = 4) scale mixture with that covariance
  rwht_signs      seeded +-1 vectors
  queries         N(0, 1/d) query vectors
"""
from __future__ import annotations

import numpy as np

ROLE_K, ROLE_V, ROLE_Q, ROLE_SIGNS = 0, 1, 2, 3


def rng(seed: int, *stream: int) -> np.random.Generator:
    """Independent PCG64 stream for (seed, *stream)."""
    return np.random.default_rng([int(seed), *[int(s) for s in stream]])


def random_orthogonal(g: np.random.Generator, d: int) -> np.ndarray:
    """Haar-random orthogonal matrix: QR of a Gaussian, R's diagonal made
    positive."""
    A = g.standard_normal((d, d))
    Q, R = np.linalg.qr(A)
    return Q * np.sign(np.diag(R))[None, :]


# ---------------------------------------------------------------- Tiny
def tiny_cov(seed: int, H: int = 2, d: int = 64, role: int = ROLE_K):
    """Per-head (Q, lam) of the Tiny regime."""
    lam = np.arange(1, d + 1, dtype=np.float64) ** -1.5
    return [(random_orthogonal(rng(seed, role, h, 0), d), lam) for h in range(H)]


def tiny_gaussian(seed: int = 0, T: int = 256, H: int = 2, d: int = 64,
                  role: int = ROLE_K) -> np.ndarray:
    """x[T, H, d] float32, x_t = Q diag(sqrt(lam)) z_t per head."""
    x = np.zeros((T, H, d), dtype=np.float64)
    for h, (Q, lam) in enumerate(tiny_cov(seed, H, d, role)):
        z = rng(seed, role, h, 1).standard_normal((T, d))
        x[:, h, :] = (z * np.sqrt(lam)[None, :]) @ Q.T
    return x.astype(np.float32)


# ---------------------------------------------------------------- spiked + t
def spiked_cov(seed: int, h: int, d: int = 128, role: int = ROLE_K, rank: int = 16,
               s_hi: float = 50.0, s_lo: float = 5.0, n_out: int = 4,
               out_scale: float = 20.0) -> np.ndarray:
    """Population covariance of one head: S (U diag(s) U^T + I) S with U a
    random d x rank orthonormal frame, s log-spaced s_hi -> s_lo, and S
    scaling n_out random channels by out_scale."""
    g = rng(seed, role, h, 0)
    U = random_orthogonal(g, d)[:, :rank]
    s = np.geomspace(s_hi, s_lo, rank)
    cov = (U * s[None, :]) @ U.T + np.eye(d)
    scale = np.ones(d)
    scale[g.choice(d, size=n_out, replace=False)] = out_scale
    return cov * scale[:, None] * scale[None, :]


def spiked_t(seed: int, T: int, H: int, d: int = 128, role: int = ROLE_K,
             nu: float = 4.0, t0: int = 0) -> np.ndarray:
    """x[T, H, d] float32 from the multivariate-t scale mixture
    x = sqrt((nu-2)/w) L z, w ~ chi2(nu), z ~ N(0, I), L L^T = cov.
    Tokens t0 .. t0+T-1 of the (seed, role) sequence (row-blocked streams so
    a slice can be regenerated on its own)."""
    x = np.zeros((T, H, d), dtype=np.float32)
    for h in range(H):
        L = np.linalg.cholesky(spiked_cov(seed, h, d, role))
        blk = 4096
        for b0 in range((t0 // blk) * blk, t0 + T, blk):
            g = rng(seed, role, h, 1, b0 // blk)
            z = g.standard_normal((blk, d))
            w = g.chisquare(nu, size=blk)
            xb = (z @ L.T) * np.sqrt((nu - 2.0) / w)[:, None]
            lo, hi = max(b0, t0), min(b0 + blk, t0 + T)
            if lo < hi:
                x[lo - t0: hi - t0, h, :] = xb[lo - b0: hi - b0]
    return x


def spiked_t_torch(seed: int, T: int, H: int, d: int = 128, role: int = ROLE_K,
                   nu: float = 4.0, device="cuda", dtype=None, out=None,
                   batch_index: int = 0):
    """Same law as ``spiked_t`` drawn on a torch device (different random
    stream: used for caches too large to draw on the host).  Returns a
    [T, H, d] tensor in ``dtype`` (bf16 by default), or fills ``out``."""
    import torch
    dtype = dtype or torch.bfloat16
    if out is None:
        out = torch.empty((T, H, d), device=device, dtype=dtype)
    gen = torch.Generator(device=device)
    for h in range(H):
        L = torch.tensor(np.linalg.cholesky(spiked_cov(seed, h, d, role)),
                         device=device, dtype=torch.float32)
        gen.manual_seed(int(seed) * 1_000_003 + role * 10_007 + h * 101 + batch_index * 7_919 + 17)
        blk = 1 << 16
        for b0 in range(0, T, blk):
            n = min(blk, T - b0)
            z = torch.randn((n, d), device=device, generator=gen)
            w = (torch.randn((n, int(nu)), device=device, generator=gen) ** 2).sum(1)
            xb = (z @ L.T) * torch.sqrt((nu - 2.0) / w)[:, None]
            out[b0: b0 + n, h, :] = xb.to(dtype)
    return out


# ---------------------------------------------------------------- misc
def rwht_signs(seed: int, H: int, d: int = 128) -> np.ndarray:
    """int8 [H, d] of +-1."""
    g = rng(seed, ROLE_SIGNS)
    return (g.integers(0, 2, size=(H, d)) * 2 - 1).astype(np.int8)


def queries(seed: int, B: int, Hq: int, d: int = 128) -> np.ndarray:
    """q[B, Hq, d] float32 ~ N(0, 1/d) (std 1/sqrt(d))."""
    g = rng(seed, ROLE_Q)
    return (g.standard_normal((B, Hq, d)) / np.sqrt(d)).astype(np.float32)


def to_bf16_exact(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even) and return the
    rounded values as float32 (exact bf16 values)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
