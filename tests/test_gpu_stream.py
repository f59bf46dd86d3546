"""GPU parity of the streaming path ("Sintesi Tecnica: SPECTRA", "La Pipeline
di SPECTRA" phases 2-3: an append-only latent cache, tokens appended one
step at a time): appends at any stream position give the codes of the
one-shot encode (boundary-band rule), and attention over packed history plus
an uncompressed recent window matches the oracle's attention over the
concatenation (2e-3 relative L2)."""
import numpy as np
import pytest
import torch

import synth
from parity import ATTN_TOL, BAND_SIGMA, FLIP_FRAC, bf16, gpu_plan, rel_l2

pytestmark = pytest.mark.gpu

FAMILY = {"tc": 2, "generic": 1}


@pytest.fixture(params=["tc", "generic"])
def path(request):
    import kv_cache_transform_encode_b300 as spx
    prev = spx.spectra_get_kernel_family()
    spx.spectra_set_kernel_family(0 if request.param == "tc" else 1)
    yield request.param
    spx.spectra_set_kernel_family(prev)


@pytest.fixture(scope="module")
def spx():
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    return spx


def _check_stream(orc, oplan, enc, stream, T):
    flips = total = 0
    for h in range(oplan.heads):
        R = int(oplan.rec_bits()[h])
        got = orc.unpack(np.ascontiguousarray(stream[h, : orc.stream_bytes(T, R)]), T, oplan.bits[h])
        diff = (got != enc[h]["codes"]) & (oplan.bits[h] > 0)[None, :]
        if diff.any():
            assert orc.decision_margin(oplan, h, enc[h])[diff].max() <= BAND_SIGMA
        flips += int(diff.sum())
        total += diff.size
    assert flips <= FLIP_FRAC * total, (flips, total)


@pytest.mark.parametrize("kind", ["eigen", "rwht"])
def test_append_in_pieces(spx, orc, path, kind):
    """Pieces starting inside a group, at its last lane, on a 128-token
    boundary and past 4096, into streams full of stale bits: the final
    streams hold the one-shot encode's codes (and the RWHT norms)."""
    T, H = 4500, 3
    x = synth.to_bf16_exact(synth.spiked_t(17, T, H, 128))
    x64 = x.astype(np.float64)
    if kind == "eigen":
        oplan = orc.make_eigen_plan(x64[:1024], 2.0)
    else:
        oplan = orc.make_rwht_plan(synth.rwht_signs(17, H, 128), 3)
    p = gpu_plan(spx, oplan)
    xd = bf16(x).cuda()
    g = torch.Generator(device="cuda").manual_seed(3)
    codes = torch.randint(0, 256, (H, p.stream_bytes(T)), dtype=torch.uint8, device="cuda", generator=g)
    norms = torch.zeros((H, T), device="cuda") if kind == "rwht" else None
    cuts = [0, 1, 31, 32, 127, 128, 129, 4097, T]
    for a, b in zip(cuts[:-1], cuts[1:]):
        spx.spectra_append(p, xd[a:b], a, codes, norms=norms)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() >= 0)
    enc = orc.encode(oplan, x64)
    _check_stream(orc, oplan, enc, codes.cpu().numpy(), T)
    if kind == "rwht":
        np.testing.assert_allclose(norms.cpu().numpy(), np.stack([e["norms"] for e in enc]), rtol=1e-5)


def test_append_one_token_per_step(spx, orc, path):
    """Decode-step appends: one token at a time from position 100 on, on top
    of an encoded prefix; equal to the one-shot encode."""
    T, H, t0 = 170, 2, 100
    x = synth.to_bf16_exact(synth.spiked_t(19, T, H, 128))
    x64 = x.astype(np.float64)
    oplan = orc.make_eigen_plan(x64, 2.0)
    p = gpu_plan(spx, oplan)
    xd = bf16(x).cuda()
    codes = p.new_streams(T)
    spx.spectra_encode(p, xd[:t0], codes)
    for t in range(t0, T):
        spx.spectra_append(p, xd[t:t + 1], t, codes)
    torch.cuda.synchronize()
    _check_stream(orc, oplan, orc.encode(oplan, x64), codes.cpu().numpy(), T)


@pytest.mark.parametrize("ctx,W", [(0, 64), (777, 0), (777, 1), (2500, 300), (5000, 128)])
def test_attn_window(spx, orc, path, ctx, W):
    B, Hq, Hkv = 2, 8, 2
    kx = [synth.to_bf16_exact(synth.spiked_t(23 + b, ctx + W, Hkv, 128, role=synth.ROLE_K)).astype(np.float64)
          for b in range(B)]
    vx = [synth.to_bf16_exact(synth.spiked_t(23 + b, ctx + W, Hkv, 128, role=synth.ROLE_V)).astype(np.float64)
          for b in range(B)]
    cal_k = kx[0][:2048] if ctx + W >= 256 else synth.to_bf16_exact(
        synth.spiked_t(23, 2048, Hkv, 128, role=synth.ROLE_K)).astype(np.float64)
    cal_v = vx[0][:2048] if ctx + W >= 256 else synth.to_bf16_exact(
        synth.spiked_t(23, 2048, Hkv, 128, role=synth.ROLE_V)).astype(np.float64)
    kp, vp = orc.make_eigen_plan(cal_k, 2.0), orc.make_eigen_plan(cal_v, 2.0)
    sb = max(orc.stream_bytes(max(ctx, 1), 1024), 16)
    ks = np.zeros((B * Hkv, sb), dtype=np.uint8)
    vs = np.zeros((B * Hkv, sb), dtype=np.uint8)
    krec = np.zeros((B, ctx, Hkv, 128))
    vrec = np.zeros((B, ctx, Hkv, 128))
    if ctx > 0:
        for b in range(B):
            ek, ev = orc.encode(kp, kx[b][:ctx]), orc.encode(vp, vx[b][:ctx])
            for h in range(Hkv):
                ks[b * Hkv + h, : len(ek[h]["stream"])] = ek[h]["stream"]
                vs[b * Hkv + h, : len(ev[h]["stream"])] = ev[h]["stream"]
            krec[b] = orc.decode(kp, [e["stream"] for e in ek], ctx)
            vrec[b] = orc.decode(vp, [e["stream"] for e in ev], ctx)
    kw = np.stack([kx[b][ctx:] for b in range(B)])          # [B, W, Hkv, d] exact bf16 values
    vw = np.stack([vx[b][ctx:] for b in range(B)])
    q = synth.to_bf16_exact(synth.queries(29, B, Hq, 128))
    want = orc.attn_decode_window(q.astype(np.float64), krec, vrec, kw, vw, 1.0)
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode_window(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(),
                                   torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda(), ctx,
                                   bf16(kw.astype(np.float32)).cuda(), bf16(vw.astype(np.float32)).cuda(), 1.0, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert rel_l2(got, want) <= ATTN_TOL, rel_l2(got, want)
