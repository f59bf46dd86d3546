"""Pins of the oracle against what the pages and mathematics fix (CPU only).

Each test ties one oracle routine to something other than itself: a closed
form, a textbook table, a library routine (LAPACK, scipy), brute force, or a
worked example written out by hand under tests/golden/.  A plausible slip in
the oracle (a dropped term, a wrong sign or index, a transposed operand)
fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.special
import scipy.stats

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- Gram
def test_gram_planted_hadamard_columns_exact(orc):
    """X = H_n[:, :d] diag(s), n >= d: G = X^T X / n = diag(s^2) exactly
    (Hadamard columns are orthogonal with squared norm n; s dyadic so every
    partial sum is exact)."""
    n, d = 64, 16
    s = (np.arange(d) + 1) / 8.0
    X = scipy.linalg.hadamard(n)[:, :d] * s[None, :]
    G = orc.gram(X)
    assert np.array_equal(G, np.diag(s * s))


def test_gram_matches_library(orc):
    x = synth.tiny_gaussian(3, T=200, H=1, d=24)[:, 0, :].astype(np.float64)
    np.testing.assert_allclose(orc.gram(x), x.T @ x / 200, rtol=1e-13, atol=1e-15)


def test_gram_uncentred(orc):
    """A constant offset shows up in G (no mean is removed): x = c for all t
    gives G = c c^T."""
    c = np.array([1.0, -2.0, 0.5])
    G = orc.gram(np.tile(c, (7, 1)))
    np.testing.assert_allclose(G, np.outer(c, c), rtol=0, atol=1e-15)


# ---------------------------------------------------------------- Jacobi
def test_jacobi_planted_diagonal_recovers_axes(orc):
    """Planted diagonal covariance: the eigenbasis is the coordinate axes
    (|Q| is a permutation matrix), eigenvalues reproduced exactly, sorted
    descending."""
    g = np.random.default_rng(1)
    d = 32
    lam = g.permutation(np.linspace(0.1, 5.0, d))
    lam_o, Q, sweeps = orc.jacobi_eigh(np.diag(lam))
    assert sweeps == 0
    assert np.array_equal(lam_o, np.sort(lam)[::-1])
    P = np.abs(Q)
    assert np.array_equal(P, P.round()) and np.array_equal(P.sum(0), np.ones(d))
    assert np.array_equal(P.sum(1), np.ones(d))
    for c in range(d):                       # axis i holds eigenvalue lam[i]
        i = int(np.argmax(P[:, c]))
        assert lam[i] == lam_o[c] and Q[i, c] == 1.0


def test_jacobi_planted_rotation(orc):
    """G = R diag(lam) R^T with a random orthogonal R: the basis recovers R's
    columns up to sign, eigenvalues to 1e-12 relative."""
    g = synth.rng(5)
    d = 48
    R = synth.random_orthogonal(g, d)
    lam = np.geomspace(100.0, 0.01, d)
    G = (R * lam[None, :]) @ R.T
    G = 0.5 * (G + G.T)
    lam_o, Q, _ = orc.jacobi_eigh(G)
    np.testing.assert_allclose(lam_o, lam, rtol=1e-11, atol=1e-12 * lam[0])
    overlap = np.abs(np.sum(Q * R, axis=0))
    np.testing.assert_allclose(overlap, 1.0, atol=1e-10)


@pytest.mark.parametrize("seed,d", [(0, 64), (1, 128)])
def test_jacobi_vs_lapack(orc, seed, d):
    """Residual, orthogonality, eigenvalues vs numpy.linalg.eigh (LAPACK),
    eigenvectors with relative gap > 1e-6 equal up to sign; sort and sign
    readings hold."""
    x = synth.spiked_t(seed, 512, 1, d)[:, 0, :].astype(np.float64)
    G = orc.gram(x)
    lam, Q, _ = orc.jacobi_eigh(G)
    gf = np.linalg.norm(G)
    assert np.linalg.norm(G @ Q - Q * lam[None, :]) <= 1e-12 * gf
    assert np.linalg.norm(Q.T @ Q - np.eye(d)) <= 1e-12
    w, U = np.linalg.eigh(G)
    w, U = w[::-1], U[:, ::-1]
    np.testing.assert_allclose(lam, w, rtol=0, atol=1e-12 * w[0])
    gaps = np.minimum(np.abs(np.diff(np.r_[np.inf, w])), np.abs(np.diff(np.r_[w, -np.inf])))
    for c in np.nonzero(gaps > 1e-6 * w[0])[0]:
        assert abs(abs(Q[:, c] @ U[:, c]) - 1.0) < 1e-8
    assert np.all(np.diff(lam) <= 0)
    for c in range(d):
        i = int(np.argmax(np.abs(Q[:, c])))
        assert Q[i, c] > 0


def test_jacobi_sign_tie_lowest_row(orc):
    """Sign reading on a tie: eigenvector (1, -1)/sqrt2 has equal magnitudes;
    the lowest row wins, so row 0 is made positive."""
    G = np.array([[1.0, -1.0], [-1.0, 1.0]])      # eigvals 2 (1,-1), 0 (1,1)
    lam, Q, _ = orc.jacobi_eigh(G)
    np.testing.assert_allclose(lam, [2.0, 0.0], atol=1e-15)
    assert Q[0, 0] > 0 and Q[1, 0] < 0 and Q[0, 1] > 0 and Q[1, 1] > 0


# ---------------------------------------------------------------- allocation
def test_alloc_worked_example(orc):
    rows = _golden_lines("alloc_worked_example.txt")
    lam = np.array([float(v) for v in rows[0][1:]])
    for r in rows[1:]:
        R = int(r[0])
        assert list(orc.alloc(lam, R)) == [int(v) for v in r[1:]], R


@pytest.mark.parametrize("B", [0.0, 0.25, 1.0, 1.33, 2.0, 4.0, 7.99, 8.0])
def test_alloc_hits_budget_exactly(orc, B):
    g = np.random.default_rng(2)
    for d in (16, 64, 128):
        lam = np.sort(g.gamma(0.5, 2.0, d))[::-1]
        R = orc.total_bits(B, d)
        bits = orc.alloc(lam, R)
        assert int(bits.astype(int).sum()) == R
        assert bits.max() <= 8


def test_total_bits_readings(orc):
    assert orc.total_bits(2.0, 64) == 128
    assert orc.total_bits(2.0, 128) == 256
    assert orc.total_bits(4.0, 128) == 512
    assert orc.total_bits(1.33, 128) == 170
    assert orc.total_bits(16.0, 128) == 1024        # saturates at 8 bits
    with pytest.raises(ValueError):
        orc.total_bits(-1.0, 128)


def test_alloc_sixteen_bits_saturates(orc):
    lam = np.geomspace(10, 1e-3, 32)
    assert np.all(orc.alloc(lam, orc.total_bits(16.0, 32)) == 8)


def _dp_min_distortion(lam, R):
    """Brute force: min sum_c lam_c 4^-b_c over integer b in [0,8], sum b = R
    (dynamic programming over channels)."""
    best = {0: 0.0}
    for l in lam:
        nxt = {}
        for used, v in best.items():
            for b in range(9):
                if used + b <= R:
                    val = v + l * 4.0 ** -b
                    if val < nxt.get(used + b, np.inf):
                        nxt[used + b] = val
        best = nxt
    return best[R]


def test_alloc_optimal_vs_bruteforce_2x16x32(orc):
    """On 2 heads x d=16 x 32 tokens: greedy reaches the DP minimum of the
    high-rate distortion sum lam_c 4^-b_c for every budget 0..128."""
    x = synth.spiked_t(11, 32, 2, 16)
    lam_all, _ = orc.calibrate(x)
    for h in range(2):
        lam = lam_all[h].astype(np.float32).astype(np.float64)
        for R in range(0, 129):
            bits = orc.alloc(lam, R)
            got = float(np.sum(lam * 4.0 ** -bits.astype(float)))
            want = _dp_min_distortion(np.maximum(lam, 0), R)
            assert got <= want * (1 + 1e-12) + 1e-300, (h, R)


def test_alloc_no_improving_swap(orc):
    """Optimality certificate: moving one bit from channel j (b_j > 0) to
    channel i (b_i < 8) never lowers the distortion."""
    lam = synth.tiny_cov(0, 1, 64)[0][1]
    for R in (0, 17, 128, 300, 512):
        b = orc.alloc(lam, R).astype(int)
        gain = np.where(b < 8, lam * 4.0 ** -b * 0.75, -np.inf)       # add 1 bit
        loss = np.where(b > 0, lam * 4.0 ** -(b - 1) * 0.75, np.inf)  # remove 1
        assert gain.max() <= loss.min() * (1 + 1e-12)


def test_alloc_population_tiny(orc):
    """Tiny regime population spectrum lam_i = i^-1.5, d = 64, 2 bits/value.
    Against the textbook continuous reverse water-filling
    b = max(0, log2(lam/theta)/2) with sum b = R: every integer width is
    within one bit of the continuous one."""
    d = 64
    lam = np.arange(1, d + 1, dtype=float) ** -1.5
    bits = orc.alloc(lam, orc.total_bits(2.0, d)).astype(int)
    assert bits.sum() == 128
    lo, hi = 1e-12, 10.0
    for _ in range(200):
        th = np.sqrt(lo * hi)
        s = np.maximum(0.0, 0.5 * np.log2(lam / th)).sum()
        lo, hi = (th, hi) if s > 128 else (lo, th)
    cont = np.maximum(0.0, 0.5 * np.log2(lam / th))
    assert np.all(np.abs(bits - cont) <= 1.0)
    assert np.all(np.diff(bits) <= 0)             # energy-ordered widths
    # regression value of the reading (greedy integer water-filling)
    want = [6, 5, 4, 4, 4, 4] + [3] * 9 + [2] * 25 + [1] * 24
    assert list(bits) == want


def test_alloc_permutation_equivariant(orc):
    g = np.random.default_rng(9)
    lam = g.uniform(0.1, 10, 40)
    perm = g.permutation(40)
    b1 = orc.alloc(lam, 90)
    b2 = orc.alloc(lam[perm], 90)
    assert np.array_equal(b1[perm], b2)


def test_zero_bit_channels_dropped(orc):
    """Steep spectrum lam_i = 10^-i at 0.5 bits/value: tail channels get 0
    bits and reconstruct to exactly 0 in those latent coordinates."""
    d = 16
    lam = 10.0 ** -np.arange(d)
    bits = orc.alloc(lam, orc.total_bits(0.5, d))
    assert bits[-1] == 0 and bits[0] > 0 and bits.sum() == 8
    plan = orc.Plan(orc.BASIS_EIGEN, orc.QUANT_UNIFORM, bits[None, :],
                    basis=np.eye(d)[None], eigvals=lam[None, :])
    x = np.random.default_rng(0).standard_normal((50, d)) * np.sqrt(lam)[None, :]
    enc = orc.encode_head(plan, 0, x)
    xh = orc.decode_head(plan, 0, enc["stream"], 50)
    assert np.all(xh[:, bits == 0] == 0.0)


# ---------------------------------------------------------------- quantizers
def test_uniform_worked_example(orc):
    rows = _golden_lines("uniform_worked_example.txt")
    y = np.array([[float(r[0])] for r in rows])
    lam, bits = np.array([1.0]), np.array([2], dtype=np.uint8)
    codes = np.zeros(y.shape, dtype=np.int32)
    orc.lib().orc_quant_uniform(y, len(rows), 1, lam, bits, codes)
    yh = np.zeros(y.shape)
    orc.lib().orc_dequant_uniform(codes, len(rows), 1, lam, bits, yh)
    assert list(codes[:, 0]) == [int(r[1]) for r in rows]
    assert list(yh[:, 0]) == [float(r[2]) for r in rows]


@pytest.mark.parametrize("b", [1, 2, 3, 5, 8])
def test_uniform_nearest_level_inside_clip(orc, b):
    """Inside +-3 sigma the code is the nearest of the 2^b midrise levels;
    outside, the extreme level."""
    sig = 1.7
    y = np.linspace(-4 * sig, 4 * sig, 20001)[:, None]
    codes = np.zeros(y.shape, dtype=np.int32)
    orc.lib().orc_quant_uniform(np.ascontiguousarray(y), len(y), 1, np.array([sig * sig]),
                                np.array([b], dtype=np.uint8), codes)
    L = 1 << b
    levels = -3 * sig + (np.arange(L) + 0.5) * 6 * sig / L
    dist = np.abs(y - levels[None, :])
    near = dist.argmin(1)
    tie = np.sort(dist, 1)[:, 1] - np.sort(dist, 1)[:, 0] < 1e-9
    ok = ~tie
    assert np.array_equal(codes[ok, 0], near[ok])


def test_uniform_gaussian_mse_analytic(orc):
    """Empirical MSE of the 2-bit uniform quantizer on N(0, sigma^2) equals
    the integral of (y - recon(y))^2 phi (scipy quadrature), within Monte
    Carlo error."""
    sig, b = 1.3, 2
    L = 1 << b
    delta = 6 * sig / L
    levels = -3 * sig + (np.arange(L) + 0.5) * delta
    edges = np.r_[-np.inf, -3 * sig + np.arange(1, L) * delta, np.inf]
    want = sum(scipy.integrate.quad(lambda v, r=levels[k]: (v - r) ** 2 *
                                    scipy.stats.norm.pdf(v, scale=sig), edges[k], edges[k + 1])[0]
               for k in range(L))
    y = np.random.default_rng(4).standard_normal((400000, 1)) * sig
    codes = np.zeros(y.shape, dtype=np.int32)
    yh = np.zeros(y.shape)
    lam, bits = np.array([sig * sig]), np.array([b], dtype=np.uint8)
    orc.lib().orc_quant_uniform(y, len(y), 1, lam, bits, codes)
    orc.lib().orc_dequant_uniform(codes, len(y), 1, lam, bits, yh)
    got = float(((y - yh) ** 2).mean())
    assert abs(got - want) < 0.01 * want


def test_lloyd_max_closed_form_and_max_tables(orc):
    """1 bit: +-sqrt(2/pi); Max (1960) Gaussian tables for 2-4 bits."""
    levels, _ = orc.lloyd_max_tables()
    assert abs(levels[0, 1] - np.sqrt(2 / np.pi)) < 1e-12
    np.testing.assert_allclose(levels[1, 2:4], [0.4528, 1.510], atol=6e-4)
    np.testing.assert_allclose(levels[2, 4:8], [0.2451, 0.7560, 1.344, 2.152], atol=6e-4)
    np.testing.assert_allclose(levels[3, 8:16], [0.1284, 0.3881, 0.6568, 0.9424, 1.256,
                                                 1.618, 2.069, 2.733], atol=6e-4)
    assert abs(orc.codebook_mse(1) - (1 - 2 / np.pi)) < 1e-12
    assert abs(orc.codebook_mse(2) - 0.1175) < 1e-4
    assert abs(orc.codebook_mse(3) - 0.03454) < 1e-5
    assert abs(orc.codebook_mse(4) - 0.009497) < 1e-5


def test_lloyd_max_structure_and_panter_dite(orc):
    levels, thresh = orc.lloyd_max_tables()
    for b in range(1, 9):
        L = 1 << b
        lv = levels[b - 1, :L]
        assert np.all(np.diff(lv) > 0)
        assert np.array_equal(lv, -lv[::-1])                  # symmetric
        np.testing.assert_array_equal(thresh[b - 1, 1:L], 0.5 * (lv[1:] + lv[:-1]))
    # high-rate asymptote D * 4^b -> sqrt(3) pi / 2
    assert abs(orc.codebook_mse(8) * 4 ** 8 / (np.sqrt(3) * np.pi / 2) - 1) < 0.01


def test_lloyd_max_centroid_by_quadrature(orc):
    """Each 3-bit level is the conditional mean of its cell (scipy quad)."""
    levels, thresh = orc.lloyd_max_tables()
    L = 8
    edges = np.r_[-np.inf, thresh[2, 1:L], np.inf]
    for k in range(L):
        m = scipy.integrate.quad(lambda v: v * scipy.stats.norm.pdf(v), edges[k], edges[k + 1])[0]
        p = scipy.stats.norm.cdf(edges[k + 1]) - scipy.stats.norm.cdf(edges[k])
        assert abs(m / p - levels[2, k]) < 1e-9


def test_lloyd_quant_nearest_level(orc):
    levels, thresh = orc.lloyd_max_tables()
    y = np.linspace(-6, 6, 5001)[:, None]
    for b in (1, 3, 6):
        L = 1 << b
        codes = np.zeros(y.shape, dtype=np.int32)
        orc.lib().orc_quant_lm(np.ascontiguousarray(y), len(y), 1, np.ones(1), 0, 1,
                               np.array([b], dtype=np.uint8), np.ascontiguousarray(thresh), codes)
        near = np.abs(y - levels[b - 1, :L][None, :]).argmin(1)
        assert np.array_equal(codes[:, 0], near)


# ---------------------------------------------------------------- packing
def test_pack_worked_example(orc):
    rows = {r[0]: r[1:] for r in _golden_lines("pack_worked_example.txt")}
    T = int(rows["T"][0])
    bits = np.array([int(v) for v in rows["bits"]], dtype=np.uint8)
    want = np.array([int(v, 16) for v in rows["bytes"]], dtype=np.uint8)
    t = np.arange(T)
    codes = np.stack([t % 4, (t // 2) % 2, np.zeros(T, int)], 1).astype(np.int32)
    codes[32] = [3, 1, 0]
    got = orc.pack(codes, bits)
    assert np.array_equal(got, want)
    assert np.array_equal(orc.unpack(got, T, bits), codes)


def test_pack_roundtrip_random_widths(orc):
    g = np.random.default_rng(7)
    for T in (1, 31, 32, 33, 100, 257):
        bits = g.integers(0, 9, 20).astype(np.uint8)
        codes = (g.integers(0, 256, (T, 20)) & ((1 << bits.astype(int)) - 1)[None, :]).astype(np.int32)
        s = orc.pack(codes, bits)
        assert len(s) % 16 == 0 and len(s) == orc.stream_bytes(T, int(bits.astype(int).sum()))
        assert np.array_equal(orc.unpack(s, T, bits), codes)


# ---------------------------------------------------------------- RWHT
def test_rwht_orthonormal_and_library_hadamard(orc):
    d = 128
    H = orc.hadamard(d)
    assert np.array_equal(H, scipy.linalg.hadamard(d))
    assert np.array_equal(H @ H.T, d * np.eye(d))
    signs = synth.rwht_signs(0, 1, d)[0]
    x = np.random.default_rng(0).standard_normal((9, d))
    y = np.zeros_like(x)
    orc.lib().orc_rwht(x, 9, d, d, signs, y)
    np.testing.assert_allclose(y, x @ (H * signs[None, :]).T / np.sqrt(d), atol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    xb = np.zeros_like(x)
    orc.lib().orc_irwht(y, 9, d, signs, xb)
    np.testing.assert_allclose(xb, x, atol=1e-14)
    e = np.zeros((1, d)); e[0, 5] = 1.0
    ye = np.zeros_like(e)
    orc.lib().orc_rwht(e, 1, d, d, signs, ye)
    np.testing.assert_allclose(ye[0], H[:, 5] * signs[5] / np.sqrt(d), atol=1e-15)


# ---------------------------------------------------------------- attention
def test_attention_vs_library_softmax(orc):
    g = np.random.default_rng(3)
    q, K, V = g.standard_normal(16), g.standard_normal((70, 16)), g.standard_normal((70, 16))
    want = scipy.special.softmax(0.3 * K @ q) @ V
    np.testing.assert_allclose(orc.attention(q, K, V, 0.3), want, rtol=1e-12, atol=1e-14)


def test_attention_one_hot_and_uniform(orc):
    g = np.random.default_rng(4)
    K, V = g.standard_normal((50, 8)), g.standard_normal((50, 8))
    q = 1000.0 * K[17] / np.linalg.norm(K[17]) ** 2
    K2 = K.copy(); K2[17] *= 1.0
    np.testing.assert_allclose(orc.attention(q, K2, V, 1.0), V[17], atol=1e-12)
    Kc = np.tile(K[0], (50, 1))
    np.testing.assert_allclose(orc.attention(g.standard_normal(8), Kc, V, 1.0), V.mean(0), atol=1e-13)


# ---------------------------------------------------------------- end to end
def test_sixteen_bits_near_lossless(orc):
    """Budget 16 bits/value: every channel at 8 bits; the uniform +-3 sigma
    quantizer is near-lossless (relMSE <= 1e-3, cosine >= 0.9995), and
    Lloyd-Max 8-bit reaches about 2.72 * 4^-8 relMSE."""
    x = synth.tiny_gaussian(0, T=256, H=2, d=64).astype(np.float64)
    for quant, lim in ((orc.QUANT_UNIFORM, 1e-3), (orc.QUANT_LLOYD, 1.5 * 2.72 * 4.0 ** -8)):
        plan = orc.make_eigen_plan(x, 16.0, quant)
        assert np.all(plan.bits == 8)
        streams = [e["stream"] for e in orc.encode(plan, x)]
        xh = orc.decode(plan, streams, 256)
        assert orc.relmse(x, xh) <= lim
        assert orc.cosine(x, xh) >= 0.9995


def test_bruteforce_2x16x32_pipeline(orc):
    """All pinned properties on 2 heads x d=16 x 32 tokens: planted-axis
    recovery, budget hit exactly, decode equals per-coordinate nearest
    reconstruction in the latent basis, and 16 bits near-lossless."""
    # planted diagonal covariance -> the eigenbasis is the axes
    g = np.random.default_rng(12)
    lam = np.geomspace(30, 0.1, 16)
    x = g.standard_normal((32, 2, 16)) * np.sqrt(lam)[None, None, :]
    lam_h, Q = orc.calibrate(x)
    for h in range(2):
        G = x[:, h, :].T @ x[:, h, :] / 32
        np.testing.assert_allclose(np.sort(np.linalg.eigvalsh(G))[::-1], lam_h[h], rtol=1e-10)
    Gd = np.diag(np.diag(x[:, 0, :].T @ x[:, 0, :] / 32))
    _, Qd, _ = orc.jacobi_eigh(Gd)
    assert np.array_equal(np.abs(Qd).sum(0), np.ones(16))
    for B in (0.5, 1.0, 2.0, 3.0, 16.0):
        plan = orc.make_eigen_plan(x, B)
        R = orc.total_bits(B, 16)
        assert np.all(plan.bits.astype(int).sum(1) == R)
        for h in range(2):
            enc = orc.encode_head(plan, h, x[:, h, :])
            xh = orc.decode_head(plan, h, enc["stream"], 32)
            # brute force per coordinate: nearest midrise level (clipped)
            y = x[:, h, :] @ plan.basis[h]
            yh = np.zeros_like(y)
            for c in range(16):
                b = int(plan.bits[h, c])
                if b == 0:
                    continue
                s = np.sqrt(plan.eigvals[h, c])
                lv = -3 * s + (np.arange(1 << b) + 0.5) * 6 * s / (1 << b)
                yh[:, c] = lv[np.abs(y[:, c:c + 1] - lv[None, :]).argmin(1)]
            np.testing.assert_allclose(xh, yh @ plan.basis[h].T, atol=1e-9)
        if B == 16.0:
            xs = orc.decode(plan, [orc.encode_head(plan, h, x[:, h, :])["stream"] for h in range(2)], 32)
            assert orc.relmse(x, xs) <= 1e-3


# ---------------------------------------------------------------- RWHT branch of the codec
def _sphere_coordinate_mse(orc, d, b):
    """MSE of the width-b Gaussian Lloyd-Max quantizer on u = sqrt(d) y_c /
    ||y|| for isotropic Gaussian y in d dimensions (a coordinate of a
    uniformly random point on the sphere of radius sqrt(d): density
    proportional to (1 - u^2/d)^((d-3)/2) on |u| < sqrt(d)), by quadrature."""
    levels, thresh = orc.lloyd_max_tables()
    L = 1 << b
    lv, th = levels[b - 1, :L], thresh[b - 1, 1:L]
    r = np.sqrt(d)
    f = lambda u: (1.0 - u * u / d) ** ((d - 3) / 2.0)
    Z = scipy.integrate.quad(f, -r, r, limit=200)[0]
    edges = np.concatenate([[-r], th, [r]])
    return sum(scipy.integrate.quad(lambda u, k=k: (u - lv[k]) ** 2 * f(u), edges[k], edges[k + 1],
                                    limit=200)[0] for k in range(L)) / Z


@pytest.mark.parametrize("seed", [0, 1])
def test_rwht_per_token_sigma_branch(orc, seed):
    """The data-independent variant ("Technisch Overzicht ...", "Experimentele
    Opstelling": randomized WHT, then a fixed Lloyd-Max codebook), with the
    per-token scale sigma = ||x|| / sqrt(d) read for it.  For Gaussian x the
    rotation keeps ||y|| = ||x|| and y/sigma is a coordinate of a random point
    on the sphere of radius sqrt(d), independent of ||x||, so the relative
    reconstruction MSE equals that coordinate's 3-bit quantizer MSE (0.03398
    at d = 128, by quadrature; 0.03455 in the Gaussian limit).  A scale of
    ||x|| instead (or ||x|| / d, or swapped strides) misses it by orders of
    magnitude.  The stored norm is ||x|| rounded to fp32, and the decode
    scales linearly with it."""
    d, T = 128, 4096
    x = np.random.default_rng(100 + seed).standard_normal((T, d))
    plan = orc.make_rwht_plan(synth.rwht_signs(seed, 1, d), 3)
    enc = orc.encode_head(plan, 0, x)
    assert enc["norms"].dtype == np.float32
    assert np.array_equal(enc["norms"], np.linalg.norm(x, axis=1).astype(np.float32))
    np.testing.assert_allclose(enc["sigma"][:, 0], enc["norms"].astype(np.float64) / np.sqrt(d), rtol=0)
    xh = orc.decode_head(plan, 0, enc["stream"], T, enc["norms"])
    want = _sphere_coordinate_mse(orc, d, 3)
    assert abs(want - 0.03398) < 5e-5
    assert abs(orc.relmse(x, xh) - want) <= 0.01 * want, (orc.relmse(x, xh), want)
    xh2 = orc.decode_head(plan, 0, enc["stream"], T, 2 * enc["norms"])
    np.testing.assert_allclose(xh2, 2 * xh, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- decision margin
def test_decision_margin_worked_example(orc):
    """Distances to the nearest decision boundary in units of sigma, against
    tests/golden/decision_margin_worked_example.txt (computed by hand; the
    Lloyd-Max rows use Max's 4-digit thresholds, hence the 1e-4 tolerance)."""
    for r in _golden_lines("decision_margin_worked_example.txt"):
        kind, b, y, want = r[0], int(r[1]), float(r[2]), float(r[3])
        quant = orc.QUANT_UNIFORM if kind == "u" else orc.QUANT_LLOYD
        plan = orc.Plan(orc.BASIS_EIGEN, quant, np.array([[b]], dtype=np.uint8),
                        basis=np.eye(1)[None], eigvals=np.array([[4.0]]))
        enc = orc.encode_head(plan, 0, np.array([[y]]))
        got = orc.decision_margin(plan, 0, enc)[0, 0]
        if np.isinf(want):
            assert np.isinf(got)
        else:
            assert abs(got - want) <= (1e-12 if kind == "u" else 1e-4), (r, got)


# ---------------------------------------------------------------- GQA head map
def test_attn_decode_gqa_head_map(orc):
    """Grouped-query attention: query head j reads kv head j // (Hq / Hkv).
    Every kv head holds a constant value vector (h + 1) * 1 and distinct
    random keys, so each output names the kv head it read: with Hq = 8 and
    Hkv = 4, heads (0..7) read kv (0,0,1,1,2,2,3,3); a j % Hkv map would read
    (0,1,2,3,0,1,2,3)."""
    g = np.random.default_rng(6)
    B, Hq, Hkv, ctx, d = 2, 8, 4, 9, 16
    K = g.standard_normal((B, ctx, Hkv, d))
    V = np.zeros((B, ctx, Hkv, d))
    for h in range(Hkv):
        V[:, :, h, :] = h + 1.0
    q = g.standard_normal((B, Hq, d))
    out = orc.attn_decode(q, K, V, 0.5)
    for b in range(B):
        for j in range(Hq):
            np.testing.assert_allclose(out[b, j], np.full(d, j // 2 + 1.0), rtol=1e-13)
    # and per head: the same as single-query attention over the mapped kv head
    for j in range(Hq):
        np.testing.assert_allclose(out[1, j], orc.attention(q[1, j], K[1, :, j // 2], V[1, :, j // 2], 0.5),
                                   rtol=1e-14)


# ---------------------------------------------------------------- grouped widths, d_eff, Plain-KV
def test_grouped_alloc_worked_example(orc):
    rows = _golden_lines("grouped_alloc_worked_example.txt")
    lam = np.array([float(v) for v in rows[0][1:]])
    for r in rows[1:]:
        g, keep, R = int(r[0]), int(r[1]), int(r[2])
        assert list(orc.alloc_grouped(lam, R, g, keep)) == [int(v) for v in r[3:]], r


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_grouped_alloc_properties_and_identity(orc, seed):
    """Group 1 over all channels is the plain greedy; every group shares one
    width; channels past `keep` get nothing; the total is g * floor(R / g)
    while groups have room; widths never exceed 8."""
    g = np.random.default_rng(seed)
    lam = np.sort(g.gamma(0.7, 3.0, 64))[::-1]
    lam[-5:] = 0.0
    for R in (0, 1, 31, 128, 200, 511, 512):
        assert np.array_equal(orc.alloc_grouped(lam, R, 1, 64), orc.alloc(lam, R))
        for grp in (2, 4, 8, 16):
            for keep in (64, 40, 16):
                b = orc.alloc_grouped(lam, R, grp, keep).astype(int)
                ng = keep // grp
                assert np.all(b[ng * grp:] == 0)
                assert np.all(b[: ng * grp].reshape(ng, grp) == b[: ng * grp: grp][:, None])
                assert b.max() <= 8
                assert b.sum() == grp * min(R // grp, 8 * ng)


def test_grouped_alloc_optimal_vs_dynamic_programming(orc):
    """Greedy on the convex high-rate distortion Lam_G 4^-b is optimal: its
    distortion equals the exhaustive minimum over group widths with at most
    floor(R / g) steps (d = 16, groups of 2 and 4, every budget 0..64)."""
    g = np.random.default_rng(9)
    lam = np.sort(g.gamma(0.5, 2.0, 16))[::-1]
    for grp in (2, 4):
        ng = 16 // grp
        Lam = lam.reshape(ng, grp).sum(1)
        for R in range(0, 65):
            steps = R // grp
            best = {0: 0.0}
            for G in range(ng):          # DP over groups: minimal distortion per step count
                nxt = {}
                for used, dist in best.items():
                    for b in range(0, 9):
                        if used + b > steps:
                            break
                        v = dist + Lam[G] * 4.0 ** -b
                        if used + b not in nxt or v < nxt[used + b]:
                            nxt[used + b] = v
                best = nxt
            b = orc.alloc_grouped(lam, R, grp, 16).astype(int)[::grp]
            greedy = float((Lam * 4.0 ** -b).sum())
            assert greedy <= min(best.values()) * (1 + 1e-12) + 1e-300, (grp, R)


def test_effective_dim_worked_example(orc):
    for r in _golden_lines("effective_dim_worked_example.txt"):
        bar = r.index("|")
        energy, de, dg = float(r[0]), int(r[1]), int(r[2])
        lam = np.array([float(v) for v in r[bar + 1:]])
        assert orc.effective_dim(lam, energy) == (de, dg), r


def test_effective_dim_spiked_spectrum(orc):
    """A planted gap: 6 strong directions over a flat noise floor -- at any
    energy fraction the gap criterion lands on 6, and one spurious large
    eigenvalue on top (a 20x outlier) moves it to 1 only when that gap is the
    widest, which it is by construction here."""
    lam = np.concatenate([np.geomspace(60, 20, 6), np.full(58, 1.0)])
    for energy in (0.7, 0.9, 0.99):
        de, dg = orc.effective_dim(lam, energy)
        assert dg == min(6, de) or (de < 6 and dg <= de)
    lam2 = np.concatenate([[60 * 20.0], lam[1:]])
    assert orc.effective_dim(lam2, 0.99)[1] == 1


def test_plain_calibration_is_the_gram_diagonal(orc):
    """Plain-KV ("Technisch Overzicht ...", "Belangrijkste Bijdragen" 1:
    scalar quantization without rotation): identity basis, channel variances
    = the raw coordinates' second moments (library matmul's diagonal)."""
    x = synth.tiny_gaussian(4, T=300, H=2, d=16).astype(np.float64)
    lam, Q = orc.calibrate_plain(x)
    for h in range(2):
        np.testing.assert_allclose(lam[h], np.diag(x[:, h, :].T @ x[:, h, :]) / 300, rtol=1e-13)
        assert np.array_equal(Q[h], np.eye(16))
    plan = orc.make_grouped_plan(x, 2.0, plain=True)
    enc = orc.encode_head(plan, 1, x[:, 1, :])
    np.testing.assert_allclose(enc["y"], x[:, 1, :], rtol=0, atol=0)


def test_ks_harness_power_and_size(orc):
    """The KS harness (tests/parity.py) on oracle runs alone, on the Tiny
    Gaussian regime: two independent seed sets of the same codec are not
    separated; 2.0 against 1.75 bits/value is.  (On the heavy-tailed spiked
    regime clipping dominates and even 1.0 bits/value is not separated at
    this sample size -- the ablation page's heavy-tail finding.)"""
    from parity import ks_same_distribution
    T, H = 512, 1

    def errs(seeds, B):
        out = []
        for s in seeds:
            x = synth.tiny_gaussian(s, T=T, H=H, d=64).astype(np.float64)
            op = orc.make_eigen_plan(x[:384], B)
            out.append(orc.relmse(x, orc.decode(op, [e["stream"] for e in orc.encode(op, x)], T)))
        return out
    a, b, c = errs(range(100, 124), 2.0), errs(range(200, 224), 2.0), errs(range(100, 124), 1.75)
    assert ks_same_distribution(a, b)[0]
    assert not ks_same_distribution(a, c)[0]


# ---------------------------------------------------------------- append and the recent window
def test_append_worked_example(orc):
    rows = {r[0]: r[1:] for r in _golden_lines("append_worked_example.txt")}
    base = {r[0]: r[1:] for r in _golden_lines("pack_worked_example.txt")}
    stream = np.array([int(b, 16) for b in base["bytes"]], dtype=np.uint8)
    bits = np.array([int(v) for v in rows["bits"]], dtype=np.uint8)
    codes = np.array([int(v) for v in rows["codes"]], dtype=np.int32).reshape(-1, 3)
    orc.pack_into(stream, codes, bits, int(rows["t0"][0]))
    assert list(stream) == [int(b, 16) for b in rows["bytes"]]


def test_append_in_pieces_equals_one_shot(orc):
    """Appending a token sequence in pieces at arbitrary positions (inside a
    group, at its end, across groups and 128-token tiles) gives the bytes of
    the one-shot pack, whatever the stream held at those positions before."""
    g = np.random.default_rng(8)
    bits = g.integers(0, 9, 24).astype(np.uint8)
    T = 700
    codes = (g.integers(0, 256, (T, 24)) & ((1 << bits.astype(int)) - 1)[None, :]).astype(np.int32)
    want = orc.pack(codes, bits)
    stream = g.integers(0, 256, len(want)).astype(np.uint8)      # stale contents
    cuts = [0, 1, 31, 32, 33, 127, 128, 129, 400, 641, T]
    for a, b in zip(cuts[:-1], cuts[1:]):
        orc.pack_into(stream, codes[a:b], bits, a)
    n_bytes = orc.stream_bytes(T, int(bits.astype(int).sum()))
    # bytes holding only tokens >= T (zero in the one-shot pack) keep their stale values
    assert np.array_equal(orc.unpack(stream, T, bits), codes)
    assert np.array_equal(orc.unpack(stream[:n_bytes], T, bits), orc.unpack(want, T, bits))


def test_attention_window_is_concatenation(orc):
    """A bf16 recent window joins the softmax: attention over (history,
    window) equals textbook softmax attention over the concatenated keys and
    values (scipy), and an empty window reduces to attn_decode."""
    g = np.random.default_rng(15)
    B, Hq, Hkv, ctx, W, d = 2, 4, 2, 40, 7, 16
    K, V = g.standard_normal((B, ctx, Hkv, d)), g.standard_normal((B, ctx, Hkv, d))
    Kw, Vw = g.standard_normal((B, W, Hkv, d)), g.standard_normal((B, W, Hkv, d))
    q = g.standard_normal((B, Hq, d))
    got = orc.attn_decode_window(q, K, V, Kw, Vw, 0.7)
    for b in range(B):
        for j in range(Hq):
            h = j // (Hq // Hkv)
            Kc = np.concatenate([K[b, :, h], Kw[b, :, h]])
            Vc = np.concatenate([V[b, :, h], Vw[b, :, h]])
            np.testing.assert_allclose(got[b, j], scipy.special.softmax(0.7 * Kc @ q[b, j]) @ Vc, rtol=1e-12)
    np.testing.assert_allclose(orc.attn_decode_window(q, K, V, Kw[:, :0], Vw[:, :0], 0.7),
                               orc.attn_decode(q, K, V, 0.7), rtol=1e-14)


# ---------------------------------------------------------------- QJL residual sketch
def test_qjl_worked_example(orc):
    for r in _golden_lines("qjl_worked_example.txt"):
        v = [float(a) for a in r]
        S = np.array(v[0:4]).reshape(2, 2)
        res, q = np.array(v[4:6]), np.array(v[6:8])
        bits, norms = orc.qjl_sketch(res[None], S)
        assert list(bits[0]) == [int(v[8]), int(v[9])]
        assert norms[0] == v[10]
        assert abs(orc.qjl_estimate(q, S, bits[0], norms[0]) - v[11]) < 1e-12


def test_qjl_unbiased_and_variance(orc):
    """Over independent Gaussian sketch matrices the estimate of <q, r> is
    unbiased, with variance ((pi/2) |q|^2 |r|^2 - <q, r>^2) / m (the
    moments of <s, q> sign(<s, r>) for Gaussian s)."""
    g = np.random.default_rng(31)
    d, m, n = 16, 32, 6000
    q, r = g.standard_normal(d), g.standard_normal(d)
    est = np.empty(n)
    for i in range(n):
        S = g.standard_normal((m, d))
        bits, norms = orc.qjl_sketch(r[None], S)
        est[i] = orc.qjl_estimate(q, S, bits[0], norms[0])
    true = float(q @ r)
    var = ((np.pi / 2) * (q @ q) * (r @ r) - true ** 2) / m
    assert abs(est.mean() - true) < 4 * np.sqrt(var / n)
    assert abs(est.var() / var - 1) < 0.1


def test_qjl_residual_is_the_reconstruction_error(orc):
    """The sketched residual is the key's reconstruction error: its norm is
    ||x - xhat|| (the rotation is orthonormal), and with m large the
    corrected score <q, xhat> + estimate approaches <q, x>."""
    x = synth.tiny_gaussian(3, T=64, H=1, d=16)[:, 0, :].astype(np.float64)
    plan = orc.make_eigen_plan(x[:, None, :], 1.0)
    enc = orc.encode_head(plan, 0, x)
    xh = orc.decode_head(plan, 0, enc["stream"], 64)
    S = np.random.default_rng(2).standard_normal((20000, 16))
    bits, norms = orc.qjl_encode_head(plan, 0, x, enc["stream"], S)
    np.testing.assert_allclose(norms, np.linalg.norm(x - xh, axis=1), rtol=1e-6)   # the fp32 plan basis
    q = np.random.default_rng(4).standard_normal(16)
    qt = plan.basis[0].T @ q
    corr = np.array([orc.qjl_estimate(qt, S, bits[t], norms[t]) for t in range(64)])
    err_plain = np.abs(xh @ q - x @ q).mean()
    err_qjl = np.abs(xh @ q + corr - x @ q).mean()
    assert err_qjl < 0.1 * err_plain


def test_qjl_attention_uses_the_estimate(orc):
    """The attention's vectorised correction is qjl_estimate token by token,
    and with a zero residual sketch norm it is plain attention."""
    g = np.random.default_rng(33)
    B, Hq, Hkv, ctx, d, m = 1, 2, 1, 12, 8, 8
    K, V = g.standard_normal((B, ctx, Hkv, d)), g.standard_normal((B, ctx, Hkv, d))
    S = g.standard_normal((m, d))
    bits = g.integers(0, 2, (B, Hkv, ctx, m)).astype(np.uint8)
    nrm = g.uniform(0.1, 1.0, (B, Hkv, ctx))
    q = g.standard_normal((B, Hq, d))
    Qb = np.linalg.qr(g.standard_normal((d, d)))[0]
    rot = [lambda v: Qb.T @ v]
    got = orc.attn_decode_qjl(q, K, V, bits, nrm, S, rot, 0.5)
    for j in range(Hq):
        s = np.array([K[0, t, 0] @ q[0, j] + orc.qjl_estimate(Qb.T @ q[0, j], S, bits[0, 0, t], nrm[0, 0, t])
                      for t in range(ctx)])
        np.testing.assert_allclose(got[0, j], scipy.special.softmax(0.5 * s) @ V[0, :, 0], rtol=1e-12)
    np.testing.assert_allclose(orc.attn_decode_qjl(q, K, V, bits, 0 * nrm, S, rot, 0.5),
                               orc.attn_decode(q, K, V, 0.5), rtol=1e-13)
