"""Spectral transform coding of transformer KV caches on B300 (sm_103a).

Thin Python binding of the C ABI in ``include/spectra.h``: the functions
below carry the same names and only marshal arguments (torch tensors ->
device pointers, the current torch stream -> cudaStream_t).  Every step of
the codec runs in the CUDA library ``libspectra.so`` built in-tree by
``kv_cache_transform_encode_b300.build``; importing this module on a machine
where that library cannot be loaded raises, and there is no CPU fallback.

Method: "Sintesi Tecnica: SPECTRA" (gist.science 2608.07915) -- Gram-matrix
eigenbasis, reverse water-filling of bits, zero-bit channels dropped,
per-token quantize-and-append, on-the-fly reconstruction, attention in the
latent space; "Technisch Overzicht ... KV-Cache Compressie" (gist.science
2607.09683) -- randomized Walsh-Hadamard rotation with a Lloyd-Max codebook.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

SPECTRA_OK = 0
SPECTRA_BF16, SPECTRA_F32 = 0, 1
SPECTRA_BASIS_EIGEN, SPECTRA_BASIS_RWHT = 0, 1
SPECTRA_Q_UNIFORM3S, SPECTRA_Q_LLOYD_GAUSS = 0, 1
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error",
                4: "eigensolve not converged", 5: "bounded wait timed out",
                6: "non-finite input", 7: "stream buffer too small"}

SPECTRA_KERNELS_AUTO, SPECTRA_KERNELS_CUDA_CORE, SPECTRA_KERNELS_TENSOR_CORE = 0, 1, 2

EXPORTS = ("spectra_version", "spectra_set_kernel_family", "spectra_get_kernel_family",
           "spectra_status_string", "spectra_plan_derived_bytes",
           "spectra_stream_bytes", "spectra_calibrate_workspace_bytes", "spectra_calibrate",
           "spectra_alloc_bits", "spectra_alloc_bits_ex", "spectra_effective_dim", "spectra_calibrate_plain",
           "spectra_plan_finalize", "spectra_encode", "spectra_encode_kv", "spectra_append", "spectra_decode",
           "spectra_decode_kv",
           "spectra_attn_workspace_bytes", "spectra_attn_decode", "spectra_attn_decode_window",
           "spectra_qjl_encode", "spectra_attn_decode_qjl", "spectra_selftest_wait", "spectra_attn_decode_noalloc")


class SpectraError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status})")
        self.status = status


class spectra_plan(C.Structure):
    _fields_ = [("heads", C.c_int32), ("head_dim", C.c_int32), ("basis", C.c_int32),
                ("quant", C.c_int32), ("max_rec_bits", C.c_int32), ("reserved", C.c_int32),
                ("basis_mat", C.c_void_p), ("eigvals", C.c_void_p), ("signs", C.c_void_p),
                ("bits", C.c_void_p), ("rec_bits", C.c_void_p), ("derived", C.c_void_p),
                ("status", C.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib() -> C.CDLL:
    """Load libspectra.so (built in-tree); raise if it is missing."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise ImportError(f"libspectra.so is not built ({path}); run "
                              "python -m kv_cache_transform_encode_b300.build")
        h = C.CDLL(path)
        vp, i32, i64, sz, f32, f64 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float, C.c_double
        P = C.POINTER(spectra_plan)
        sig = {
            "spectra_version": (C.c_int, []),
            "spectra_set_kernel_family": (C.c_int, [C.c_int]),
            "spectra_get_kernel_family": (C.c_int, []),
            "spectra_status_string": (C.c_char_p, [C.c_int]),
            "spectra_plan_derived_bytes": (sz, [C.c_int, C.c_int]),
            "spectra_stream_bytes": (sz, [i32, i64]),
            "spectra_calibrate_workspace_bytes": (sz, [C.c_int, C.c_int, i64]),
            "spectra_calibrate": (C.c_int, [P, vp, C.c_int, i64, i64, C.c_int, vp, sz, vp, vp]),
            "spectra_alloc_bits": (C.c_int, [P, f64, C.c_int, vp]),
            "spectra_alloc_bits_ex": (C.c_int, [P, f64, C.c_int, vp, vp]),
            "spectra_effective_dim": (C.c_int, [P, f64, vp, vp, vp]),
            "spectra_calibrate_plain": (C.c_int, [P, vp, C.c_int, i64, i64, vp, sz, vp]),
            "spectra_plan_finalize": (C.c_int, [P, vp]),
            "spectra_encode": (C.c_int, [P, vp, C.c_int, i64, i64, vp, i64, vp, i64, vp]),
            "spectra_encode_kv": (C.c_int, [P, P, vp, vp, C.c_int, i64, i64, vp, vp, i64, vp, vp, i64, vp]),
            "spectra_decode": (C.c_int, [P, vp, i64, vp, i64, i64, vp, C.c_int, i64, vp]),
            "spectra_decode_kv": (C.c_int, [P, P, vp, vp, i64, vp, vp, i64, i64, vp, vp, C.c_int, i64, vp]),
            "spectra_qjl_encode": (C.c_int, [P, vp, vp, C.c_int, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                             vp]),
            "spectra_attn_decode_qjl": (C.c_int, [P, P, vp, C.c_int, C.c_int, C.c_int, vp, vp, i64, vp, vp, i64,
                                                  i64, vp, vp, i64, vp, i64, f32, vp, vp, sz, vp]),
            "spectra_selftest_wait": (C.c_int, [C.c_uint64, vp, vp, vp]),
            "spectra_append": (C.c_int, [P, vp, C.c_int, i64, i64, i64, vp, i64, vp, i64, vp]),
            "spectra_attn_decode_window": (C.c_int, [P, P, vp, C.c_int, C.c_int, C.c_int, vp, vp, i64, vp, vp,
                                                     i64, i64, vp, vp, C.c_int, i64, i64, f32, vp, vp, sz, vp]),
            "spectra_attn_workspace_bytes": (sz, [C.c_int, C.c_int, C.c_int, i64]),
            "spectra_attn_decode": (C.c_int, [P, P, vp, C.c_int, C.c_int, C.c_int, vp, vp, i64, vp, vp,
                                              i64, i64, f32, vp, vp, sz, vp]),
            "spectra_attn_decode_noalloc": (C.c_int, [P, P, vp, C.c_int, C.c_int, C.c_int, vp, vp, i64, vp,
                                                      vp, i64, i64, f32, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _LIB = h
    return _LIB


def _check(st: int, what: str):
    if st != SPECTRA_OK:
        raise SpectraError(st, what)


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPECTRA_BF16
    if t.dtype == torch.float32:
        return SPECTRA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


class Plan:
    """Device buffers of one codec plan (caller-owned, allocated through
    torch) and the matching C struct."""

    def __init__(self, heads: int, head_dim: int, basis: int = SPECTRA_BASIS_EIGEN,
                 quant: int = SPECTRA_Q_UNIFORM3S, device="cuda"):
        self.heads, self.head_dim, self.basis, self.quant = heads, head_dim, basis, quant
        H, d = heads, head_dim
        kw = dict(device=device)
        self.basis_mat = torch.zeros((H, d, d), dtype=torch.float32, **kw)
        self.eigvals = torch.zeros((H, d), dtype=torch.float32, **kw)
        self.signs = torch.ones((H, d), dtype=torch.int8, **kw)
        self.bits = torch.zeros((H, d), dtype=torch.uint8, **kw)
        self.rec_bits = torch.zeros((H,), dtype=torch.int32, **kw)
        nbytes = spectra_plan_derived_bytes(H, d)
        self._derived = torch.zeros((nbytes + 256,), dtype=torch.uint8, **kw)
        off = (-self._derived.data_ptr()) % 256
        self.derived = self._derived[off: off + nbytes]
        self.status = torch.zeros((H,), dtype=torch.int32, **kw)
        self.max_rec_bits = 0

    def c(self) -> spectra_plan:
        return spectra_plan(self.heads, self.head_dim, self.basis, self.quant, self.max_rec_bits, 0,
                            self.basis_mat.data_ptr(), self.eigvals.data_ptr(), self.signs.data_ptr(),
                            self.bits.data_ptr(), self.rec_bits.data_ptr(), self.derived.data_ptr(),
                            self.status.data_ptr())

    def stream_bytes(self, T: int) -> int:
        return spectra_stream_bytes(self.max_rec_bits, T)

    def new_streams(self, T: int, n: int | None = None) -> torch.Tensor:
        """uint8 [n, stream_bytes] (n defaults to heads), zero-filled."""
        n = self.heads if n is None else n
        return torch.zeros((n, max(self.stream_bytes(T), 16)), dtype=torch.uint8,
                           device=self.bits.device)


# ----------------------------------------------------------------- C ABI
def spectra_version() -> int:
    return lib().spectra_version()


def spectra_set_kernel_family(family: int):
    """Process-wide kernel family: SPECTRA_KERNELS_AUTO, _CUDA_CORE or
    _TENSOR_CORE (initially from the SPECTRA_PATH environment variable)."""
    _check(lib().spectra_set_kernel_family(int(family)), "spectra_set_kernel_family")


def spectra_get_kernel_family() -> int:
    return lib().spectra_get_kernel_family()


def spectra_status_string(st: int) -> str:
    return lib().spectra_status_string(st).decode()


def spectra_plan_derived_bytes(heads: int, head_dim: int) -> int:
    return lib().spectra_plan_derived_bytes(heads, head_dim)


def spectra_stream_bytes(rec_bits: int, T: int) -> int:
    return lib().spectra_stream_bytes(rec_bits, T)


def spectra_calibrate_workspace_bytes(heads: int, head_dim: int, n_cal: int) -> int:
    return lib().spectra_calibrate_workspace_bytes(heads, head_dim, n_cal)


def spectra_attn_workspace_bytes(B: int, Hq: int, head_dim: int, ctx: int) -> int:
    return lib().spectra_attn_workspace_bytes(B, Hq, head_dim, ctx)


def spectra_calibrate(plan: Plan, x: torch.Tensor, n_cal: int | None = None, max_sweeps: int = 30,
                      workspace: torch.Tensor | None = None, gram_out: torch.Tensor | None = None,
                      stream=None):
    """x: [T, H, d] bf16/f32 cuda tensor (token stride = x.stride(0))."""
    n_cal = x.shape[0] if n_cal is None else n_cal
    need = spectra_calibrate_workspace_bytes(plan.heads, plan.head_dim, n_cal)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=x.device)
    p = plan.c()
    st = lib().spectra_calibrate(C.byref(p), _ptr(x), _dt(x), n_cal, x.stride(0), max_sweeps,
                                 _ptr(workspace), workspace.numel(), _ptr(gram_out), _stream(stream))
    _check(st, "spectra_calibrate")


def spectra_alloc_bits(plan: Plan, avg_bits: float, fixed_bits: int = 0, stream=None):
    p = plan.c()
    st = lib().spectra_alloc_bits(C.byref(p), float(avg_bits), int(fixed_bits), _stream(stream))
    _check(st, "spectra_alloc_bits")
    plan.max_rec_bits = p.max_rec_bits


def spectra_alloc_bits_ex(plan: Plan, avg_bits: float, group: int = 1, keep: torch.Tensor | None = None,
                          stream=None):
    """Grouped water-filling over the first keep[h] channels (keep: int32
    cuda tensor [heads] or None)."""
    p = plan.c()
    st = lib().spectra_alloc_bits_ex(C.byref(p), float(avg_bits), int(group), _ptr(keep), _stream(stream))
    _check(st, "spectra_alloc_bits_ex")
    plan.max_rec_bits = p.max_rec_bits


def spectra_effective_dim(plan: Plan, energy: float, d_energy: torch.Tensor, d_gap: torch.Tensor, stream=None):
    """d_energy, d_gap: int32 cuda tensors [heads] (outputs)."""
    p = plan.c()
    _check(lib().spectra_effective_dim(C.byref(p), float(energy), _ptr(d_energy), _ptr(d_gap), _stream(stream)),
           "spectra_effective_dim")


def spectra_calibrate_plain(plan: Plan, x: torch.Tensor, n_cal: int | None = None,
                            workspace: torch.Tensor | None = None, stream=None):
    """Identity basis, raw second moments (Plain-KV); x as for spectra_calibrate."""
    n_cal = x.shape[0] if n_cal is None else n_cal
    need = spectra_calibrate_workspace_bytes(plan.heads, plan.head_dim, n_cal)
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=x.device)
    p = plan.c()
    st = lib().spectra_calibrate_plain(C.byref(p), _ptr(x), _dt(x), n_cal, x.stride(0), _ptr(workspace),
                                       workspace.numel(), _stream(stream))
    _check(st, "spectra_calibrate_plain")


def spectra_plan_finalize(plan: Plan, stream=None):
    p = plan.c()
    _check(lib().spectra_plan_finalize(C.byref(p), _stream(stream)), "spectra_plan_finalize")


def spectra_encode(plan: Plan, x: torch.Tensor, codes: torch.Tensor, norms: torch.Tensor | None = None,
                   T: int | None = None, stream=None):
    """x: [T, H, d]; codes: uint8 [H, stride]; norms (RWHT): f32 [H, >=T]."""
    T = x.shape[0] if T is None else T
    p = plan.c()
    st = lib().spectra_encode(C.byref(p), _ptr(x), _dt(x), T, x.stride(0), _ptr(codes),
                              codes.stride(0) if codes.dim() > 1 else 0, _ptr(norms),
                              norms.stride(0) if norms is not None and norms.dim() > 1 else 0,
                              _stream(stream))
    _check(st, "spectra_encode")


def spectra_encode_kv(kplan: Plan, vplan: Plan, k: torch.Tensor, v: torch.Tensor, k_codes: torch.Tensor,
                      v_codes: torch.Tensor, k_norms: torch.Tensor | None = None,
                      v_norms: torch.Tensor | None = None, T: int | None = None, stream=None):
    """k, v: [T, H, d] (same dtype and token stride); k_codes, v_codes: uint8
    [H, stride] (same stride); norms (RWHT): f32 [H, >=T] (same stride)."""
    T = k.shape[0] if T is None else T
    if v.stride(0) != k.stride(0) or v.dtype != k.dtype:
        raise ValueError("spectra_encode_kv: k and v need the same dtype and token stride")
    ss = k_codes.stride(0) if k_codes.dim() > 1 else 0
    if (v_codes.stride(0) if v_codes.dim() > 1 else 0) != ss:
        raise ValueError("spectra_encode_kv: k_codes and v_codes need the same stride")
    ns = k_norms.stride(0) if k_norms is not None and k_norms.dim() > 1 else 0
    if v_norms is not None and v_norms.dim() > 1 and v_norms.stride(0) != ns:
        raise ValueError("spectra_encode_kv: k_norms and v_norms need the same stride")
    kp, vp = kplan.c(), vplan.c()
    st = lib().spectra_encode_kv(C.byref(kp), C.byref(vp), _ptr(k), _ptr(v), _dt(k), T, k.stride(0),
                                 _ptr(k_codes), _ptr(v_codes), ss, _ptr(k_norms), _ptr(v_norms), ns,
                                 _stream(stream))
    _check(st, "spectra_encode_kv")


def spectra_append(plan: Plan, x: torch.Tensor, t0: int, codes: torch.Tensor,
                   norms: torch.Tensor | None = None, stream=None):
    """Append x [n, H, d] at stream positions t0 .. t0+n-1 of codes
    [H, stride] (norms [H, >= t0+n] for RWHT)."""
    p = plan.c()
    st = lib().spectra_append(C.byref(p), _ptr(x), _dt(x), x.shape[0], x.stride(0), int(t0), _ptr(codes),
                              codes.stride(0) if codes.dim() > 1 else 0, _ptr(norms),
                              norms.stride(0) if norms is not None and norms.dim() > 1 else 0, _stream(stream))
    _check(st, "spectra_append")


def spectra_decode(plan: Plan, codes: torch.Tensor, T: int, out: torch.Tensor,
                   norms: torch.Tensor | None = None, stream=None):
    """codes: uint8 [H, stride]; out: [T, H, d] bf16/f32."""
    p = plan.c()
    st = lib().spectra_decode(C.byref(p), _ptr(codes), codes.stride(0) if codes.dim() > 1 else 0,
                              _ptr(norms), norms.stride(0) if norms is not None and norms.dim() > 1 else 0,
                              T, _ptr(out), _dt(out), out.stride(0), _stream(stream))
    _check(st, "spectra_decode")


def spectra_decode_kv(kplan: Plan, vplan: Plan, k_codes: torch.Tensor, v_codes: torch.Tensor, T: int,
                      k_out: torch.Tensor, v_out: torch.Tensor, k_norms: torch.Tensor | None = None,
                      v_norms: torch.Tensor | None = None, stream=None):
    """k_codes, v_codes: uint8 [H, stride] (same stride); k_out, v_out: [T, H, d]
    (same dtype and token stride); norms (RWHT): f32 [H, >=T] (same stride)."""
    ss = k_codes.stride(0) if k_codes.dim() > 1 else 0
    if (v_codes.stride(0) if v_codes.dim() > 1 else 0) != ss:
        raise ValueError("spectra_decode_kv: k_codes and v_codes need the same stride")
    if v_out.stride(0) != k_out.stride(0) or v_out.dtype != k_out.dtype:
        raise ValueError("spectra_decode_kv: k_out and v_out need the same dtype and token stride")
    ns = k_norms.stride(0) if k_norms is not None and k_norms.dim() > 1 else 0
    if v_norms is not None and v_norms.dim() > 1 and v_norms.stride(0) != ns:
        raise ValueError("spectra_decode_kv: k_norms and v_norms need the same stride")
    kp, vp = kplan.c(), vplan.c()
    st = lib().spectra_decode_kv(C.byref(kp), C.byref(vp), _ptr(k_codes), _ptr(v_codes), ss, _ptr(k_norms),
                                 _ptr(v_norms), ns, T, _ptr(k_out), _ptr(v_out), _dt(k_out), k_out.stride(0),
                                 _stream(stream))
    _check(st, "spectra_decode_kv")


def spectra_attn_decode(kplan: Plan, vplan: Plan, q: torch.Tensor, k_codes: torch.Tensor,
                        v_codes: torch.Tensor, ctx: int, softmax_scale: float, out: torch.Tensor,
                        workspace: torch.Tensor | None = None, k_norms: torch.Tensor | None = None,
                        v_norms: torch.Tensor | None = None, stream=None):
    """q: [B, Hq, d]; k_codes/v_codes: uint8 [B*Hkv, stride]; out: f32 [B, Hq, d]."""
    B, Hq, d = q.shape
    if workspace is None:
        workspace = torch.empty((max(spectra_attn_workspace_bytes(B, Hq, d, ctx), 16) + 256,),
                                dtype=torch.uint8, device=q.device)
    off = (-workspace.data_ptr()) % 256
    ws = workspace[off:]
    kp, vp = kplan.c(), vplan.c()
    nstride = k_norms.stride(0) if k_norms is not None else 0
    st = lib().spectra_attn_decode(C.byref(kp), C.byref(vp), _ptr(q), _dt(q), B, Hq, _ptr(k_codes),
                                   _ptr(v_codes), k_codes.stride(0), _ptr(k_norms), _ptr(v_norms),
                                   nstride, ctx, float(softmax_scale), _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _check(st, "spectra_attn_decode")


def spectra_attn_decode_window(kplan: Plan, vplan: Plan, q: torch.Tensor, k_codes: torch.Tensor,
                               v_codes: torch.Tensor, ctx: int, k_win: torch.Tensor, v_win: torch.Tensor,
                               softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor | None = None,
                               k_norms: torch.Tensor | None = None, v_norms: torch.Tensor | None = None,
                               stream=None):
    """Attention over ctx packed tokens followed by the uncompressed window
    k_win / v_win [B, W, Hkv, d] (contiguous rows: token stride Hkv * d)."""
    B, Hq, d = q.shape
    W = k_win.shape[1]
    if workspace is None:
        workspace = torch.empty((max(spectra_attn_workspace_bytes(B, Hq, d, ctx), 16) + 256,),
                                dtype=torch.uint8, device=q.device)
    off = (-workspace.data_ptr()) % 256
    ws = workspace[off:]
    kp, vp = kplan.c(), vplan.c()
    nstride = k_norms.stride(0) if k_norms is not None else 0
    st = lib().spectra_attn_decode_window(C.byref(kp), C.byref(vp), _ptr(q), _dt(q), B, Hq, _ptr(k_codes),
                                          _ptr(v_codes), k_codes.stride(0), _ptr(k_norms), _ptr(v_norms), nstride,
                                          ctx, _ptr(k_win), _ptr(v_win), _dt(k_win), W, k_win.stride(1),
                                          float(softmax_scale), _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "spectra_attn_decode_window")


def spectra_qjl_encode(plan: Plan, sketch: torch.Tensor, x: torch.Tensor, codes: torch.Tensor,
                       qjl_bits: torch.Tensor, qjl_norms: torch.Tensor, norms: torch.Tensor | None = None,
                       stream=None):
    """sketch f32 [d, d]; x [T, H, d]; codes [H, stride]; qjl_bits uint8
    [H, >= spectra_stream_bytes(d, T)]; qjl_norms f32 [H, >= T]."""
    p = plan.c()
    T = x.shape[0]
    st = lib().spectra_qjl_encode(C.byref(p), _ptr(sketch), _ptr(x), _dt(x), T, x.stride(0), _ptr(codes),
                                  codes.stride(0), _ptr(norms), norms.stride(0) if norms is not None else 0,
                                  _ptr(qjl_bits), qjl_bits.stride(0), _ptr(qjl_norms), qjl_norms.stride(0),
                                  _stream(stream))
    _check(st, "spectra_qjl_encode")


def spectra_attn_decode_qjl(kplan: Plan, vplan: Plan, q: torch.Tensor, k_codes: torch.Tensor,
                            v_codes: torch.Tensor, ctx: int, sketch: torch.Tensor, k_qjl_bits: torch.Tensor,
                            k_qjl_norms: torch.Tensor, softmax_scale: float, out: torch.Tensor,
                            workspace: torch.Tensor | None = None, k_norms: torch.Tensor | None = None,
                            v_norms: torch.Tensor | None = None, stream=None):
    B, Hq, d = q.shape
    if workspace is None:
        workspace = torch.empty((max(spectra_attn_workspace_bytes(B, Hq, d, ctx), 16) + 256,),
                                dtype=torch.uint8, device=q.device)
    off = (-workspace.data_ptr()) % 256
    ws = workspace[off:]
    kp, vp = kplan.c(), vplan.c()
    nstride = k_norms.stride(0) if k_norms is not None else 0
    st = lib().spectra_attn_decode_qjl(C.byref(kp), C.byref(vp), _ptr(q), _dt(q), B, Hq, _ptr(k_codes),
                                       _ptr(v_codes), k_codes.stride(0), _ptr(k_norms), _ptr(v_norms), nstride, ctx,
                                       _ptr(sketch), _ptr(k_qjl_bits), k_qjl_bits.stride(0), _ptr(k_qjl_norms),
                                       k_qjl_norms.stride(0), float(softmax_scale), _ptr(out), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(st, "spectra_attn_decode_qjl")


def spectra_selftest_wait(limit_ns: int, status: torch.Tensor, elapsed_ns: torch.Tensor, stream=None):
    """status: int32 cuda [2]; elapsed_ns: int64 cuda [1] (see spectra.h)."""
    _check(lib().spectra_selftest_wait(int(limit_ns), _ptr(status), _ptr(elapsed_ns), _stream(stream)),
           "spectra_selftest_wait")


SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES = 16 << 20


def spectra_attn_decode_noalloc(kplan: Plan, vplan: Plan, q: torch.Tensor, k_codes: torch.Tensor,
                                v_codes: torch.Tensor, ctx: int, softmax_scale: float, out: torch.Tensor,
                                k_norms: torch.Tensor | None = None, v_norms: torch.Tensor | None = None,
                                stream=None):
    """spectra_attn_decode for callers that cannot allocate device memory:
    the split-context scratch comes from a static buffer inside the library
    (SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES), so neither this binding nor the
    library allocates anything.  Calls that overlap on the GPU race on that
    shared buffer; make the first call on a device before any stream
    capture."""
    B, Hq, d = q.shape
    kp, vp = kplan.c(), vplan.c()
    nstride = k_norms.stride(0) if k_norms is not None else 0
    st = lib().spectra_attn_decode_noalloc(C.byref(kp), C.byref(vp), _ptr(q), _dt(q), B, Hq, _ptr(k_codes),
                                           _ptr(v_codes), k_codes.stride(0), _ptr(k_norms), _ptr(v_norms),
                                           nstride, ctx, float(softmax_scale), _ptr(out), _stream(stream))
    _check(st, "spectra_attn_decode_noalloc")
