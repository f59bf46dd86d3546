"""Helpers shared by the GPU parity tests: move an oracle plan onto the
device (the oracle's plan is the one both sides use, so code parity is
decided on identical inputs), compare codes within the boundary band, and
the relative-L2 measure of the tolerances.

Tolerances (from the workload statement):
  allocation          bit-exact
  codes               bit-exact except where the oracle's pre-quantization
                      value lies within 1e-5 relative of a decision boundary
                      (relative to the channel's clip range 3 sigma, i.e.
                      |y - tau| <= 3e-5 sigma), and such flips < 1e-4 of entries
  reconstruction      relative L2 <= 1e-3
  attention output    relative L2 <= 2e-3
"""
import numpy as np
import torch

BAND_SIGMA = 3e-5          # 1e-5 x the +-3 sigma clip range, in units of sigma
FLIP_FRAC = 1e-4
REC_TOL = 1e-3
ATTN_TOL = 2e-3


def gpu_plan(spx, oplan, device="cuda"):
    """Device copy of an oracle plan, finalized by the library."""
    H, d = oplan.bits.shape
    p = spx.Plan(H, d, basis=oplan.basis_kind, quant=oplan.quant, device=device)
    if oplan.basis is not None:
        p.basis_mat.copy_(torch.from_numpy(np.asarray(oplan.basis, dtype=np.float32)))
        p.eigvals.copy_(torch.from_numpy(np.asarray(oplan.eigvals, dtype=np.float32)))
    if oplan.signs is not None:
        p.signs.copy_(torch.from_numpy(np.asarray(oplan.signs, dtype=np.int8)))
    p.bits.copy_(torch.from_numpy(np.asarray(oplan.bits, dtype=np.uint8)))
    p.max_rec_bits = int(oplan.rec_bits().max())
    spx.spectra_plan_finalize(p)
    return p


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def compare_codes(orc, oplan, h, enc, gpu_stream, T):
    """Unpack the GPU stream with the oracle's unpacker; every mismatch must
    sit inside the boundary band.  Returns (mismatches, entries)."""
    got = orc.unpack(np.ascontiguousarray(gpu_stream[: orc.stream_bytes(T, int(oplan.rec_bits()[h]))]),
                     T, oplan.bits[h])
    want = enc["codes"]
    live = oplan.bits[h] > 0
    diff = (got != want) & live[None, :]
    if diff.any():
        margin = orc.decision_margin(oplan, h, enc)
        assert np.all(margin[diff] <= BAND_SIGMA), (
            f"head {h}: {int(diff.sum())} code flips, worst margin {margin[diff].max():.3g} sigma")
        assert np.all(np.abs(got[diff] - want[diff]) <= 1)
    return int(diff.sum()), int(live.sum()) * T


def bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def ks_same_distribution(a, b, alpha=0.01):
    """Two-sample Kolmogorov-Smirnov test of the ablation page's validation
    methodology ("Technisch Overzicht ...", "Experimentele Opstelling": a
    systematic difference between two implementations against seed
    variance).  Returns (no systematic difference at level alpha, p-value)."""
    import scipy.stats
    p = float(scipy.stats.ks_2samp(np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)).pvalue)
    return p > alpha, p
