"""spectra_attn_decode_noalloc: the allocation-free attention entry point.

It exists for callers that cannot allocate device memory when they run a
decode step (code inside an allocator or memory-pool callback, hosts whose
device memory belongs to another framework's pool, deployments that forbid
allocation after start-up): its scratch is a static buffer inside the
library.  Here it is called through the C ABI and must reproduce the
workspace-taking spectra_attn_decode, call after call; requests larger than
its static scratch are refused.

This file is collected last on purpose and builds all of its inputs itself,
so it runs the same alone in a fresh process or after the other tests."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


@pytest.fixture(scope="module")
def spx():
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    return spx


def _inputs(spx, B=2, Hq=8, Hkv=2, ctx=3000, d=128):
    """Device plans calibrated and allocated by the library, and packed K/V
    streams for B batch elements."""
    dev = torch.device("cuda")
    kx = torch.stack([torch.from_numpy(synth.spiked_t(21 + b, ctx, Hkv, d, role=synth.ROLE_K))
                      for b in range(B)]).to(torch.bfloat16).to(dev)
    vx = torch.stack([torch.from_numpy(synth.spiked_t(21 + b, ctx, Hkv, d, role=synth.ROLE_V))
                      for b in range(B)]).to(torch.bfloat16).to(dev)
    kp, vp = spx.Plan(Hkv, d, device=dev), spx.Plan(Hkv, d, device=dev)
    spx.spectra_calibrate(kp, kx[0], n_cal=min(ctx, 2048))
    spx.spectra_calibrate(vp, vx[0], n_cal=min(ctx, 2048))
    spx.spectra_alloc_bits(kp, 2.0)
    spx.spectra_alloc_bits(vp, 2.0)
    sb = kp.stream_bytes(ctx)
    kc = torch.zeros((B * Hkv, sb), dtype=torch.uint8, device=dev)
    vc = torch.zeros((B * Hkv, sb), dtype=torch.uint8, device=dev)
    for b in range(B):
        spx.spectra_encode(kp, kx[b], kc[b * Hkv:(b + 1) * Hkv])
        spx.spectra_encode(vp, vx[b], vc[b * Hkv:(b + 1) * Hkv])
    q = torch.from_numpy(synth.queries(9, B, Hq, d)).to(torch.bfloat16).to(dev)
    return kp, vp, q, kc, vc


def test_noalloc_matches_workspace_entry_point(spx):
    B, Hq, ctx = 2, 8, 3000
    kp, vp, q, kc, vc = _inputs(spx, B=B, Hq=Hq, ctx=ctx)
    ref = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode(kp, vp, q, kc, vc, ctx, 1.0, ref)
    torch.cuda.synchronize()
    want = ref.cpu().numpy().astype(np.float64)
    assert np.isfinite(want).all() and np.abs(want).max() > 0
    for _ in range(2):                           # two calls in a row share the scratch
        out = torch.full((B, Hq, 128), float("nan"), device="cuda")
        spx.spectra_attn_decode_noalloc(kp, vp, q, kc, vc, ctx, 1.0, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(got - want) <= ATTN_TOL * np.linalg.norm(want)


def test_noalloc_refuses_oversized_requests(spx):
    """A well-formed call whose scratch need is beyond the static buffer is
    refused with SPECTRA_ERR_UNSUPPORTED before any launch; malformed calls
    get the same status as from spectra_attn_decode; an empty context needs
    no scratch at any batch size and only zeroes the output."""
    import ctypes as C
    kp, vp, q, kc, vc = _inputs(spx, B=1, Hq=4, ctx=256)
    B, Hq, big_ctx = 64, 64, 1 << 40                   # scratch need far beyond the static buffer
    assert spx.spectra_attn_workspace_bytes(B, Hq, 128, big_ctx) > spx.SPECTRA_ATTN_NOALLOC_SCRATCH_BYTES
    stride = spx.spectra_stream_bytes(max(kp.max_rec_bits, vp.max_rec_bits), big_ctx)
    out = torch.zeros((B, Hq, 128), device="cuda")
    kps, vps = kp.c(), vp.c()

    def call(Hq_, ctx_, stride_):
        return spx.lib().spectra_attn_decode_noalloc(C.byref(kps), C.byref(vps), C.c_void_p(q.data_ptr()), 0,
                                                      B, Hq_, C.c_void_p(kc.data_ptr()),
                                                      C.c_void_p(vc.data_ptr()), stride_, None, None, 0, ctx_,
                                                      1.0, C.c_void_p(out.data_ptr()), None)
    assert call(Hq, big_ctx, stride) == 2              # well formed, too large: unsupported
    assert call(Hq + 1, big_ctx, stride) == 1          # query heads not a multiple of kv heads
    assert call(Hq, big_ctx, 16) == 1                  # streams too short for the context
    out.fill_(3.0)
    assert call(Hq, 0, stride) == 0                    # empty context: zeroes the output
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
