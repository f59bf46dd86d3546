"""Oracle for spectral transform coding of a KV cache -- TEST INFRASTRUCTURE.

A plain, slow fp64 CPU implementation of what the CUDA library computes,
written from the method's description (page titles and sections are cited at
each routine, here and in ``spectra_oracle.c``).  Only ``tests/``, the smoke
entry point and the benchmark's CPU-baseline leg may import this package; the
library never does, and the two share no code, tables or constants.

The heavy loops are plain C (``spectra_oracle.c``, built with gcc into
``_liboracle.so`` beside it); this module only marshals numpy arrays and
composes those loops in the order the method describes them:

    Gram  ->  eigenbasis (Jacobi)  ->  bit allocation (reverse water-filling)
          ->  project  ->  quantize  ->  pack           (encode)
          ->  unpack  ->  dequantize  ->  reconstruct   (decode)
          ->  softmax attention over the reconstruction

Parity status of every function is pinned by ``tests/test_oracle_*.py``;
none is unpinned.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass, field
from functools import lru_cache

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spectra_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

BASIS_EIGEN = 0
BASIS_RWHT = 1
QUANT_UNIFORM = 0
QUANT_LLOYD = 1


def build(force: bool = False) -> str:
    """Compile the oracle's C loops with gcc (no GPU, no nvcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11",
                               "-D_DEFAULT_SOURCE", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_P = np.ctypeslib.ndpointer
_D = _P(dtype=np.float64, flags="C_CONTIGUOUS")
_I32 = _P(dtype=np.int32, flags="C_CONTIGUOUS")
_U8 = _P(dtype=np.uint8, flags="C_CONTIGUOUS")
_I8 = _P(dtype=np.int8, flags="C_CONTIGUOUS")
_L, _I = C.c_long, C.c_int


@lru_cache(maxsize=1)
def lib() -> C.CDLL:
    h = C.CDLL(build())
    sig = {
        "orc_gram": (None, [_D, _L, _L, _I, _D]),
        "orc_jacobi": (_I, [_D, _I, C.c_double, _I, _D, _D]),
        "orc_alloc": (_L, [_D, _I, _L, _U8]),
        "orc_alloc_grouped": (_L, [_D, _I, _L, _I, _I, _U8]),
        "orc_effective_dim": (None, [_D, _I, C.c_double, C.POINTER(C.c_int), C.POINTER(C.c_int)]),
        "orc_lloyd_max": (_L, [_I, C.c_double, _L, _D, _D]),
        "orc_codebook_mse": (C.c_double, [_I, _D, _D]),
        "orc_project": (None, [_D, _L, _L, _I, _D, _D]),
        "orc_reconstruct": (None, [_D, _L, _I, _D, _D]),
        "orc_rwht": (None, [_D, _L, _L, _I, _I8, _D]),
        "orc_irwht": (None, [_D, _L, _I, _I8, _D]),
        "orc_quant_uniform": (None, [_D, _L, _I, _D, _U8, _I32]),
        "orc_dequant_uniform": (None, [_I32, _L, _I, _D, _U8, _D]),
        "orc_quant_lm": (None, [_D, _L, _I, _D, _L, _L, _U8, _D, _I32]),
        "orc_dequant_lm": (None, [_I32, _L, _I, _D, _L, _L, _U8, _D, _D]),
        "orc_stream_bytes": (_L, [_L, _L]),
        "orc_pack": (None, [_I32, _L, _I, _U8, _U8]),
        "orc_unpack": (None, [_U8, _L, _I, _U8, _I32]),
        "orc_pack_into": (None, [_I32, _L, _I, _U8, _L, _U8]),
        "orc_qjl_sketch": (None, [_D, _L, _I, _D, _I, _U8, _D]),
        "orc_qjl_estimate": (C.c_double, [_D, _I, _D, _I, _U8, C.c_double]),
        "orc_attention": (None, [_D, _D, _D, _L, _I, C.c_double, _D]),
    }
    for name, (res, args) in sig.items():
        f = getattr(h, name)
        f.restype = res
        f.argtypes = args
    return h


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# --------------------------------------------------------------------------
# Calibration: Gram + eigenbasis  ("Sintesi Tecnica: SPECTRA", Metodologia
# items 1 and 3; "La Pipeline di SPECTRA" phase 1)
# --------------------------------------------------------------------------
def gram(x: np.ndarray) -> np.ndarray:
    """G = (1/n) sum_t x_t x_t^T for x[n, d] (uncentred second moment)."""
    x = _f64(x)
    n, d = x.shape
    G = np.zeros((d, d))
    lib().orc_gram(x, n, d, d, G)
    return G


def jacobi_eigh(G: np.ndarray, tol: float = 1e-14, max_sweeps: int = 60):
    """Cyclic Jacobi on a symmetric matrix.  Returns (lam desc, Q, sweeps);
    column c of Q is the eigenvector of lam[c], sign-fixed."""
    G = _f64(G)
    d = G.shape[0]
    lam = np.zeros(d)
    Q = np.zeros((d, d))
    sweeps = lib().orc_jacobi(G, d, tol, max_sweeps, lam, Q)
    if sweeps < 0:
        raise RuntimeError("oracle Jacobi did not converge")
    return lam, Q, sweeps


def calibrate(x_cal: np.ndarray):
    """Per-head Gram + eigenbasis for x_cal[n, H, d].

    Returns (lam[H, d] fp64, Q[H, d, d] fp64)."""
    x_cal = np.asarray(x_cal)
    n, H, d = x_cal.shape
    lams, Qs = np.zeros((H, d)), np.zeros((H, d, d))
    for h in range(H):
        lam, Q, _ = jacobi_eigh(gram(x_cal[:, h, :]))
        lams[h], Qs[h] = lam, Q
    return lams, Qs


# --------------------------------------------------------------------------
# Allocation ("La Pipeline di SPECTRA" phase 2: reverse water-filling;
# Metodologia item 2: zero-bit channels dropped)
# --------------------------------------------------------------------------
def total_bits(avg_bits: float, d: int) -> int:
    """R_tot = min(floor(B*d + 1e-9), 8d): integer budget per vector.
    Reading: widths saturate at 8, so budgets above 8 bits/value give 8d."""
    if not (avg_bits >= 0.0):
        raise ValueError("avg_bits must be >= 0")
    return int(min(np.floor(avg_bits * d + 1e-9), 8 * d))


def alloc(lam, R_tot: int) -> np.ndarray:
    """Greedy integer reverse water-filling on lam (per channel)."""
    lam = _f64(lam)
    bits = np.zeros(lam.shape[0], dtype=np.uint8)
    lib().orc_alloc(lam, lam.shape[0], int(R_tot), bits)
    return bits


def alloc_grouped(lam, R_tot: int, group: int = 1, keep: int | None = None) -> np.ndarray:
    """Grouped reverse water-filling over the first `keep` channels
    ("La Pipeline di SPECTRA" phase 2, "Raggruppamento")."""
    lam = _f64(lam)
    d = lam.shape[0]
    bits = np.zeros(d, dtype=np.uint8)
    lib().orc_alloc_grouped(lam, d, int(R_tot), int(group), int(d if keep is None else keep), bits)
    return bits


def effective_dim(lam, energy: float = 0.95):
    """(d_energy, d_gap) of a descending spectrum ("Technisch Overzicht ...",
    "Regime-Specifieke Prestaties": spectral-gap pruning of d_eff)."""
    lam = _f64(lam)
    de, dg = C.c_int(0), C.c_int(0)
    lib().orc_effective_dim(lam, lam.shape[0], float(energy), C.byref(de), C.byref(dg))
    return de.value, dg.value


# --------------------------------------------------------------------------
# Codebooks
# --------------------------------------------------------------------------
@lru_cache(maxsize=1)
def lloyd_max_tables(tol: float = 1e-13):
    """Gaussian Lloyd-Max levels/thresholds for widths 1..8.

    Returns (levels[8, 256], thresh[8, 256]); row b-1 holds width b,
    levels[b-1, :2^b] ascending, thresh[b-1, k] for k = 1..2^b-1."""
    levels = np.zeros((8, 256))
    thresh = np.zeros((8, 256))
    for b in range(1, 9):
        lv = np.zeros(1 << b)
        th = np.zeros(1 << b)
        it = lib().orc_lloyd_max(b, tol, 50_000_000, lv, th)
        if it < 0:
            raise RuntimeError(f"Lloyd-Max width {b} did not converge")
        levels[b - 1, : 1 << b] = lv
        thresh[b - 1, : 1 << b] = th
        thresh[b - 1, 0] = -np.inf
    return levels, thresh


def codebook_mse(b: int) -> float:
    levels, thresh = lloyd_max_tables()
    L = 1 << b
    return lib().orc_codebook_mse(L, _f64(levels[b - 1, :L]), _f64(thresh[b - 1, :L]))


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix in natural order, built by doubling."""
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


# --------------------------------------------------------------------------
# Plans
# --------------------------------------------------------------------------
@dataclass
class Plan:
    """A per-head codec plan as both sides consume it.

    basis[H, d, d] (column c = channel c) and eigvals[H, d] hold values that
    are exactly representable in fp32 (the plan format), bits[H, d] uint8,
    signs[H, d] int8 (RWHT)."""
    basis_kind: int
    quant: int
    bits: np.ndarray
    basis: np.ndarray | None = None
    eigvals: np.ndarray | None = None
    signs: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def heads(self) -> int:
        return self.bits.shape[0]

    @property
    def d(self) -> int:
        return self.bits.shape[1]

    def rec_bits(self) -> np.ndarray:
        return self.bits.astype(np.int64).sum(axis=1)


def make_eigen_plan(x_cal: np.ndarray, avg_bits: float, quant: int = QUANT_UNIFORM,
                    fixed_bits: int = 0) -> Plan:
    """Calibrate on x_cal[n, H, d], round the plan to fp32, then allocate.

    The allocation runs on the fp32 eigenvalues (the plan's precision), so a
    device allocation given the same plan must agree bit for bit."""
    lam, Q = calibrate(x_cal)
    lam32 = lam.astype(np.float32).astype(np.float64)
    Q32 = Q.astype(np.float32).astype(np.float64)
    H, d = lam.shape
    if fixed_bits:
        bits = np.full((H, d), fixed_bits, dtype=np.uint8)
    else:
        R = total_bits(avg_bits, d)
        bits = np.stack([alloc(lam32[h], R) for h in range(H)])
    return Plan(BASIS_EIGEN, quant, bits, basis=Q32, eigvals=lam32,
                extra={"lam64": lam, "Q64": Q})


def make_grouped_plan(x_cal: np.ndarray, avg_bits: float, group: int = 1, keep=None,
                      quant: int = QUANT_UNIFORM, plain: bool = False) -> Plan:
    """Eigenbasis (or, with `plain`, the identity basis with the raw
    coordinates' second moments -- the ablation page's Plain-KV) rounded to
    fp32, then grouped water-filling over the first keep[h] channels of each
    head (keep: None = all, an int, or one value per head)."""
    if plain:
        lam, Q = calibrate_plain(x_cal)
    else:
        lam, Q = calibrate(x_cal)
    lam32 = lam.astype(np.float32).astype(np.float64)
    Q32 = Q.astype(np.float32).astype(np.float64)
    H, d = lam.shape
    keeps = [d] * H if keep is None else ([int(keep)] * H if np.isscalar(keep) else [int(k) for k in keep])
    R = total_bits(avg_bits, d)
    bits = np.stack([alloc_grouped(lam32[h], R, group, keeps[h]) for h in range(H)])
    return Plan(BASIS_EIGEN, quant, bits, basis=Q32, eigvals=lam32, extra={"lam64": lam, "Q64": Q})


def calibrate_plain(x_cal: np.ndarray):
    """Plain-KV calibration ("Technisch Overzicht ...", "Belangrijkste
    Bijdragen" 1: scalar quantization without rotation): the identity basis,
    the raw coordinates' uncentred second moments (the Gram diagonal) as the
    channel variances.  Returns (lam[H, d], Q[H, d, d] = I)."""
    x_cal = np.asarray(x_cal)
    n, H, d = x_cal.shape
    lams = np.stack([np.diag(gram(x_cal[:, h, :])) for h in range(H)])
    return lams, np.broadcast_to(np.eye(d), (H, d, d)).copy()


def make_rwht_plan(signs: np.ndarray, width: int = 3) -> Plan:
    """Data-independent plan: seeded +-1 signs, fixed Gaussian Lloyd-Max
    width on every channel, no water-filling (the TurboQuant-style variant
    of the ablation page)."""
    signs = np.asarray(signs, dtype=np.int8)
    H, d = signs.shape
    return Plan(BASIS_RWHT, QUANT_LLOYD, np.full((H, d), width, dtype=np.uint8), signs=signs)


# --------------------------------------------------------------------------
# Encode / decode of one head
# --------------------------------------------------------------------------
def stream_bytes(T: int, R: int) -> int:
    return int(lib().orc_stream_bytes(T, R))


def pack(codes: np.ndarray, bits: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    T, d = codes.shape
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.zeros(stream_bytes(T, int(bits.astype(np.int64).sum())), dtype=np.uint8)
    lib().orc_pack(codes, T, d, bits, out)
    return out


def pack_into(stream: np.ndarray, codes: np.ndarray, bits: np.ndarray, t0: int) -> np.ndarray:
    """Write the codes of tokens t0 .. t0+n-1 into `stream` (in place, every
    other bit kept) -- the append-only latent cache ("La Pipeline di
    SPECTRA" phases 2-3).  Returns the stream."""
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    n, d = codes.shape
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    assert stream.dtype == np.uint8 and stream.flags["C_CONTIGUOUS"]
    assert len(stream) >= stream_bytes(t0 + n, int(bits.astype(np.int64).sum()))
    lib().orc_pack_into(codes, n, d, bits, int(t0), stream)
    return stream


def unpack(stream: np.ndarray, T: int, bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    d = bits.shape[0]
    codes = np.zeros((T, d), dtype=np.int32)
    lib().orc_unpack(np.ascontiguousarray(stream, dtype=np.uint8), T, d, bits, codes)
    return codes


def _sig_channel(eigvals_h):
    return np.sqrt(np.maximum(_f64(eigvals_h), 0.0))


def encode_head(plan: Plan, h: int, x: np.ndarray):
    """Encode x[T, d] of head h.  Returns dict with y (pre-quantization
    coordinates), codes[T, d], stream (uint8), norms (RWHT, fp32) and sigma
    (the scale each decision used, per entry)."""
    x = _f64(x)
    T, d = x.shape
    bits = np.ascontiguousarray(plan.bits[h], dtype=np.uint8)
    y = np.zeros((T, d))
    codes = np.zeros((T, d), dtype=np.int32)
    norms = None
    if plan.basis_kind == BASIS_EIGEN:
        lib().orc_project(x, T, d, d, _f64(plan.basis[h]), y)
        lam = _f64(plan.eigvals[h])
        if plan.quant == QUANT_UNIFORM:
            lib().orc_quant_uniform(y, T, d, lam, bits, codes)
        else:
            _, thresh = lloyd_max_tables()
            sig = _sig_channel(lam)
            lib().orc_quant_lm(y, T, d, sig, 0, 1, bits, _f64(thresh), codes)
        sigma = np.broadcast_to(_sig_channel(lam), (T, d))
    else:
        signs = np.ascontiguousarray(plan.signs[h], dtype=np.int8)
        lib().orc_rwht(x, T, d, d, signs, y)
        # Reading: per-vector scale sigma = ||x|| / sqrt(d); the norm is kept
        # in fp32 and both sides scale by the stored value.
        norms = np.sqrt((x * x).sum(axis=1)).astype(np.float32)
        sig = _f64(norms) / np.sqrt(d)
        _, thresh = lloyd_max_tables()
        lib().orc_quant_lm(y, T, d, sig, 1, 0, bits, _f64(thresh), codes)
        sigma = np.broadcast_to(sig[:, None], (T, d))
    stream = pack(codes, bits)
    return {"y": y, "codes": codes, "stream": stream, "norms": norms, "sigma": sigma}


def decode_head(plan: Plan, h: int, stream: np.ndarray, T: int, norms=None) -> np.ndarray:
    """Decode head h's stream back to x_hat[T, d] (fp64)."""
    bits = np.ascontiguousarray(plan.bits[h], dtype=np.uint8)
    d = bits.shape[0]
    codes = unpack(stream, T, bits)
    yh = np.zeros((T, d))
    xh = np.zeros((T, d))
    if plan.basis_kind == BASIS_EIGEN:
        lam = _f64(plan.eigvals[h])
        if plan.quant == QUANT_UNIFORM:
            lib().orc_dequant_uniform(codes, T, d, lam, bits, yh)
        else:
            levels, _ = lloyd_max_tables()
            lib().orc_dequant_lm(codes, T, d, _sig_channel(lam), 0, 1, bits, _f64(levels), yh)
        lib().orc_reconstruct(yh, T, d, _f64(plan.basis[h]), xh)
    else:
        levels, _ = lloyd_max_tables()
        sig = _f64(np.asarray(norms, dtype=np.float32)) / np.sqrt(d)
        lib().orc_dequant_lm(codes, T, d, sig, 1, 0, bits, _f64(levels), yh)
        lib().orc_irwht(yh, T, d, np.ascontiguousarray(plan.signs[h], dtype=np.int8), xh)
    return xh


def decision_margin(plan: Plan, h: int, enc: dict) -> np.ndarray:
    """Distance of each pre-quantization value to its nearest decision
    boundary, in units of sigma (inf for dropped channels).  A code may
    legitimately differ between two correct implementations only where this
    is tiny (the 1e-5-relative boundary band)."""
    y, sig = enc["y"], np.asarray(enc["sigma"])
    bits = plan.bits[h].astype(np.int64)
    T, d = y.shape
    out = np.full((T, d), np.inf)
    _, thresh = lloyd_max_tables()
    for c in range(d):
        b = int(bits[c])
        if b == 0:
            continue
        s = sig[:, c]
        ok = s > 0
        if plan.basis_kind == BASIS_EIGEN and plan.quant == QUANT_UNIFORM:
            delta = 6.0 * s / (1 << b)
            bounds = -3.0 * s[:, None] + np.arange(1, 1 << b)[None, :] * delta[:, None]
        else:
            bounds = thresh[b - 1, 1: 1 << b][None, :] * s[:, None]
        dist = np.abs(y[:, c:c + 1] - bounds).min(axis=1)
        out[ok, c] = dist[ok] / s[ok]
    return out


# --------------------------------------------------------------------------
# Multi-head helpers
# --------------------------------------------------------------------------
def encode(plan: Plan, x: np.ndarray):
    """x[T, H, d] -> list of per-head encode dicts."""
    return [encode_head(plan, h, x[:, h, :]) for h in range(plan.heads)]


def decode(plan: Plan, streams, T: int, norms=None) -> np.ndarray:
    """Per-head streams -> x_hat[T, H, d] (fp64)."""
    out = np.zeros((T, plan.heads, plan.d))
    for h in range(plan.heads):
        out[:, h, :] = decode_head(plan, h, streams[h], T,
                                   None if norms is None else norms[h])
    return out


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one query q[d] over K[ctx, d], V[ctx, d]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    out = np.zeros(q.shape[0])
    lib().orc_attention(q, K, V, K.shape[0], q.shape[0], float(scale), out)
    return out


def dequant_head(plan: Plan, h: int, codes: np.ndarray, norms=None) -> np.ndarray:
    """Latent reconstruction yhat[T, d] of head h from its codes (the decode's
    dequantization step alone)."""
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    T, d = codes.shape
    bits = np.ascontiguousarray(plan.bits[h], dtype=np.uint8)
    yh = np.zeros((T, d))
    levels, _ = lloyd_max_tables()
    if plan.basis_kind == BASIS_EIGEN and plan.quant == QUANT_UNIFORM:
        lib().orc_dequant_uniform(codes, T, d, _f64(plan.eigvals[h]), bits, yh)
    elif plan.basis_kind == BASIS_EIGEN:
        lib().orc_dequant_lm(codes, T, d, _sig_channel(plan.eigvals[h]), 0, 1, bits, _f64(levels), yh)
    else:
        sig = _f64(np.asarray(norms, dtype=np.float32)) / np.sqrt(d)
        lib().orc_dequant_lm(codes, T, d, sig, 1, 0, bits, _f64(levels), yh)
    return yh


def qjl_sketch(r: np.ndarray, S: np.ndarray):
    """1-bit JL sketch of residuals r[T, d] with the Gaussian S[m, d]
    ("Technisch Overzicht ...", TQ-QKV).  Returns (bits[T, m] 0/1, norms[T])."""
    r, S = _f64(r), _f64(S)
    T, d = r.shape
    m = S.shape[0]
    bits = np.zeros((T, m), dtype=np.uint8)
    norms = np.zeros(T)
    lib().orc_qjl_sketch(r, T, d, S, m, bits, norms)
    return bits, norms


def qjl_estimate(q: np.ndarray, S: np.ndarray, bits: np.ndarray, norm: float) -> float:
    S = _f64(S)
    return float(lib().orc_qjl_estimate(_f64(q), S.shape[1], S, S.shape[0],
                                        np.ascontiguousarray(bits, dtype=np.uint8), float(norm)))


def qjl_encode_head(plan: Plan, h: int, x: np.ndarray, stream: np.ndarray, S: np.ndarray, norms=None):
    """Sketch of head h's key residuals: r = y - yhat in the latent basis, y
    the projection of x, yhat the dequantized codes of `stream`.  Returns
    (bits[T, m], residual norms[T])."""
    x = _f64(x)
    T, d = x.shape
    y = np.zeros((T, d))
    if plan.basis_kind == BASIS_EIGEN:
        lib().orc_project(x, T, d, d, _f64(plan.basis[h]), y)
    else:
        lib().orc_rwht(x, T, d, d, np.ascontiguousarray(plan.signs[h], dtype=np.int8), y)
    yh = dequant_head(plan, h, unpack(stream, T, plan.bits[h]), norms)
    return qjl_sketch(y - yh, S)


def attn_decode_qjl(q, Khat, Vhat, kbits, knorm, S, rot, scale: float) -> np.ndarray:
    """Decode-step GQA attention whose key scores carry the QJL correction:
    s_t = scale (<q, khat_t> + qjl_estimate(B_K^T q, bits_t, ||r_t||)).
    q[B, Hq, d]; Khat, Vhat[B, ctx, Hkv, d]; kbits[B, Hkv, ctx, m]; knorm[B,
    Hkv, ctx]; rot[Hkv] maps q to the latent coordinates of kv head h."""
    B, Hq, d = q.shape
    Hkv = Khat.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for j in range(Hq):
            h = j // g
            qt = rot[h](_f64(q[b, j]))
            s = Khat[b, :, h, :] @ _f64(q[b, j])
            # qjl_estimate for every token at once: sqrt(pi/2)/m ||r_t|| sum_j <s_j, qt> z_j(t)
            z = 2.0 * kbits[b, h].astype(np.float64) - 1.0
            s = s + np.sqrt(np.pi / 2) / S.shape[0] * _f64(knorm[b, h]) * (z @ (_f64(S) @ qt))
            s = scale * s
            p = np.exp(s - s.max())
            out[b, j] = (p / p.sum()) @ Vhat[b, :, h, :]
    return out


def attn_decode_window(q, Khat, Vhat, Kwin, Vwin, scale: float) -> np.ndarray:
    """Decode-step GQA attention over a cache that holds a packed history
    (Khat, Vhat [B, ctx, Hkv, d], reconstructed) followed by a recent window
    kept uncompressed (Kwin, Vwin [B, W, Hkv, d]): the softmax runs over the
    concatenation of both ("La Pipeline di SPECTRA" phase 3: reconstructed
    keys and values feed standard attention; the newest tokens are the ones
    not yet appended)."""
    return attn_decode(q, np.concatenate([Khat, Kwin], axis=1), np.concatenate([Vhat, Vwin], axis=1), scale)


def attn_decode(q: np.ndarray, Khat: np.ndarray, Vhat: np.ndarray, scale: float) -> np.ndarray:
    """Decode-step GQA attention in the original basis.

    q[B, Hq, d]; Khat, Vhat[B, ctx, Hkv, d] (reconstructed caches).
    Query head j reads KV head j // (Hq // Hkv).  Returns out[B, Hq, d]."""
    B, Hq, d = q.shape
    Hkv = Khat.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for j in range(Hq):
            kv = j // g
            out[b, j] = attention(q[b, j], Khat[b, :, kv, :], Vhat[b, :, kv, :], scale)
    return out


def relmse(x: np.ndarray, xh: np.ndarray) -> float:
    """Relative MSE ||x - xh||^2 / ||x||^2 (the ablation page's relMSE)."""
    x = _f64(x)
    return float(((x - _f64(xh)) ** 2).sum() / max((x * x).sum(), 1e-300))


def cosine(x: np.ndarray, xh: np.ndarray) -> float:
    """Mean per-vector cosine similarity over the last axis."""
    x, xh = _f64(x), _f64(xh)
    num = (x * xh).sum(-1)
    den = np.sqrt((x * x).sum(-1) * (xh * xh).sum(-1))
    ok = den > 0
    return float((num[ok] / den[ok]).mean())
