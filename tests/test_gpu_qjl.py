"""GPU parity of the 1-bit QJL key-residual sketch ("Technisch Overzicht:
Ablatie ...", "Experimentele Opstelling" and "Belangrijkste Bijdragen" 1:
TQ-QKV) against the oracle: sketch bits equal except where <s_j, r> is
within 1e-4 relative of zero (fewer than 1e-3 of the bits), residual norms to
1e-4, and attention with the corrected scores to 2e-3 relative L2."""
import numpy as np
import pytest
import torch

import synth
from parity import ATTN_TOL, bf16, gpu_plan, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def spx():
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    return spx


def _case(orc, kind, T, H, seed):
    x = synth.to_bf16_exact(synth.spiked_t(seed, T, H, 128))
    x64 = x.astype(np.float64)
    if kind == "eigen":
        oplan = orc.make_eigen_plan(x64[: min(T, 1024)], 2.0)
    elif kind == "lloyd":
        oplan = orc.make_eigen_plan(x64[: min(T, 1024)], 1.33, orc.QUANT_LLOYD)
    else:
        oplan = orc.make_rwht_plan(synth.rwht_signs(seed, H, 128), 3)
    S = np.random.default_rng(seed + 100).standard_normal((128, 128))
    return x, x64, oplan, S


@pytest.mark.parametrize("kind", ["eigen", "lloyd", "rwht"])
def test_qjl_encode_matches_oracle(spx, orc, kind):
    T, H = 700, 3
    x, x64, oplan, S = _case(orc, kind, T, H, 41)
    encs = orc.encode(oplan, x64)
    p = gpu_plan(spx, oplan)
    sb = p.stream_bytes(T)
    cd = torch.zeros((H, max(sb, 16)), dtype=torch.uint8)
    for h in range(H):
        cd[h, : len(encs[h]["stream"])] = torch.from_numpy(encs[h]["stream"])
    cd = cd.cuda()
    nd = (torch.from_numpy(np.stack([e["norms"] for e in encs])).cuda() if kind == "rwht" else None)
    qb = torch.zeros((H, spx.spectra_stream_bytes(128, T)), dtype=torch.uint8, device="cuda")
    qn = torch.zeros((H, T), device="cuda")
    spx.spectra_qjl_encode(p, torch.from_numpy(S.astype(np.float32)).cuda(), bf16(x).cuda(), cd, qb, qn, norms=nd)
    torch.cuda.synchronize()
    S32 = S.astype(np.float32).astype(np.float64)
    flips = total = 0
    for h in range(H):
        bits, nrm = orc.qjl_encode_head(oplan, h, x64[:, h, :], encs[h]["stream"], S32, encs[h]["norms"])
        ones = np.ones(128, dtype=np.uint8)
        got = orc.unpack(np.ascontiguousarray(qb[h].cpu().numpy()), T, ones)        # [T, 128] 0/1
        np.testing.assert_allclose(qn[h].cpu().numpy(), nrm, rtol=1e-4)
        diff = got != bits
        if diff.any():
            # the residual the oracle sketched, to find each flip's margin
            y = np.zeros((T, 128))
            if oplan.basis_kind == orc.BASIS_EIGEN:
                y = x64[:, h, :] @ oplan.basis[h]
            else:
                y = x64[:, h, :] @ (orc.hadamard(128) * oplan.signs[h][None, :]).T / np.sqrt(128)
            yh = orc.dequant_head(oplan, h, orc.unpack(encs[h]["stream"], T, oplan.bits[h]), encs[h]["norms"])
            a = (y - yh) @ S32.T
            rel = np.abs(a) / (np.linalg.norm(S32, axis=1)[None, :] * np.maximum(nrm, 1e-30)[:, None])
            assert rel[diff].max() <= 1e-4, rel[diff].max()
        flips += int(diff.sum())
        total += diff.size
    assert flips <= 1e-3 * total, (flips, total)


@pytest.fixture(params=["tc", "generic"])
def path(request):
    """Kernel family: the level-table tensor-core kernel (required) or the
    CUDA-core kernel."""
    import kv_cache_transform_encode_b300 as spx
    prev = spx.spectra_get_kernel_family()
    spx.spectra_set_kernel_family({"tc": 2, "generic": 1}[request.param])
    yield request.param
    spx.spectra_set_kernel_family(prev)


@pytest.mark.parametrize("B,Hq,Hkv,ctx", [(2, 8, 2, 1500), (2, 14, 2, 2048 + 1029)])
def test_attn_qjl_matches_oracle(spx, orc, path, B, Hq, Hkv, ctx):
    S = np.random.default_rng(7).standard_normal((128, 128))
    S32 = S.astype(np.float32).astype(np.float64)
    kx = [synth.to_bf16_exact(synth.spiked_t(51 + b, ctx, Hkv, 128, role=synth.ROLE_K)).astype(np.float64)
          for b in range(B)]
    vx = [synth.to_bf16_exact(synth.spiked_t(51 + b, ctx, Hkv, 128, role=synth.ROLE_V)).astype(np.float64)
          for b in range(B)]
    kp, vp = orc.make_eigen_plan(kx[0][:1024], 2.0), orc.make_eigen_plan(vx[0][:1024], 2.0)
    sb = orc.stream_bytes(ctx, 256)
    ks = np.zeros((B * Hkv, sb), np.uint8)
    vs = np.zeros((B * Hkv, sb), np.uint8)
    qbs = np.zeros((B * Hkv, orc.stream_bytes(ctx, 128)), np.uint8)
    qns = np.zeros((B * Hkv, ctx), np.float32)
    kbits = np.zeros((B, Hkv, ctx, 128), np.uint8)
    knorm = np.zeros((B, Hkv, ctx))
    krec = np.zeros((B, ctx, Hkv, 128))
    vrec = np.zeros((B, ctx, Hkv, 128))
    for b in range(B):
        ek, ev = orc.encode(kp, kx[b]), orc.encode(vp, vx[b])
        for h in range(Hkv):
            ks[b * Hkv + h, : len(ek[h]["stream"])] = ek[h]["stream"]
            vs[b * Hkv + h, : len(ev[h]["stream"])] = ev[h]["stream"]
            bits, nrm = orc.qjl_encode_head(kp, h, kx[b][:, h, :], ek[h]["stream"], S32)
            kbits[b, h], knorm[b, h] = bits, nrm.astype(np.float32)
            qbs[b * Hkv + h] = orc.pack(bits.astype(np.int32), np.ones(128, np.uint8))
            qns[b * Hkv + h] = nrm
        krec[b] = orc.decode(kp, [e["stream"] for e in ek], ctx)
        vrec[b] = orc.decode(vp, [e["stream"] for e in ev], ctx)
    q = synth.to_bf16_exact(synth.queries(53, B, Hq, 128))
    rot = [lambda v, h=h: kp.basis[h].T @ v for h in range(Hkv)]
    want = orc.attn_decode_qjl(q.astype(np.float64), krec, vrec, kbits, knorm, S32, rot, 1.0)
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode_qjl(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(), torch.from_numpy(ks).cuda(),
                                torch.from_numpy(vs).cuda(), ctx, torch.from_numpy(S.astype(np.float32)).cuda(),
                                torch.from_numpy(qbs).cuda(), torch.from_numpy(qns).cuda(), 1.0, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert rel_l2(got, want) <= ATTN_TOL, rel_l2(got, want)
    # the correction changes the result (it is not silently skipped)
    plain = orc.attn_decode(q.astype(np.float64), krec, vrec, 1.0)
    assert rel_l2(plain, want) > 10 * ATTN_TOL


def test_attn_qjl_rwht_matches_oracle(spx, orc, path):
    """TQ-KV with the QJL key sketch: RWHT + 3-bit Lloyd-Max plans (per-token
    norms on both sides) and the sketch correction in the same scores, over
    three context splits with a ragged last group."""
    B, Hq, Hkv, ctx, d = 2, 8, 2, 2048 + 77, 128
    S = np.random.default_rng(9).standard_normal((d, d))
    S32 = S.astype(np.float32).astype(np.float64)
    kx = [synth.to_bf16_exact(synth.spiked_t(61 + b, ctx, Hkv, d, role=synth.ROLE_K)).astype(np.float64)
          for b in range(B)]
    vx = [synth.to_bf16_exact(synth.spiked_t(61 + b, ctx, Hkv, d, role=synth.ROLE_V)).astype(np.float64)
          for b in range(B)]
    kp = orc.make_rwht_plan(synth.rwht_signs(63, Hkv, d), 3)
    vp = orc.make_rwht_plan(synth.rwht_signs(64, Hkv, d), 3)
    sb = orc.stream_bytes(ctx, 3 * d)
    ks = np.zeros((B * Hkv, sb), np.uint8)
    vs = np.zeros((B * Hkv, sb), np.uint8)
    kn = np.zeros((B * Hkv, ctx), np.float32)
    vn = np.zeros((B * Hkv, ctx), np.float32)
    qbs = np.zeros((B * Hkv, orc.stream_bytes(ctx, d)), np.uint8)
    qns = np.zeros((B * Hkv, ctx), np.float32)
    kbits = np.zeros((B, Hkv, ctx, d), np.uint8)
    knorm = np.zeros((B, Hkv, ctx))
    krec = np.zeros((B, ctx, Hkv, d))
    vrec = np.zeros((B, ctx, Hkv, d))
    for b in range(B):
        ek, ev = orc.encode(kp, kx[b]), orc.encode(vp, vx[b])
        for h in range(Hkv):
            i = b * Hkv + h
            ks[i, : len(ek[h]["stream"])] = ek[h]["stream"]
            vs[i, : len(ev[h]["stream"])] = ev[h]["stream"]
            kn[i], vn[i] = ek[h]["norms"], ev[h]["norms"]
            bits, nrm = orc.qjl_encode_head(kp, h, kx[b][:, h, :], ek[h]["stream"], S32, norms=ek[h]["norms"])
            kbits[b, h], knorm[b, h] = bits, nrm.astype(np.float32)
            qbs[i] = orc.pack(bits.astype(np.int32), np.ones(d, np.uint8))
            qns[i] = nrm
        krec[b] = orc.decode(kp, [e["stream"] for e in ek], ctx, [e["norms"] for e in ek])
        vrec[b] = orc.decode(vp, [e["stream"] for e in ev], ctx, [e["norms"] for e in ev])
    q = synth.to_bf16_exact(synth.queries(67, B, Hq, d))

    def rot(v, h):
        y = np.zeros((1, d))
        orc.lib().orc_rwht(np.ascontiguousarray(v[None, :], dtype=np.float64), 1, d, d,
                           np.ascontiguousarray(kp.signs[h], dtype=np.int8), y)
        return y[0]
    want = orc.attn_decode_qjl(q.astype(np.float64), krec, vrec, kbits, knorm, S32,
                               [lambda v, h=h: rot(v, h) for h in range(Hkv)], 1.0)
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.zeros((B, Hq, d), device="cuda")
    spx.spectra_attn_decode_qjl(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(), torch.from_numpy(ks).cuda(),
                                torch.from_numpy(vs).cuda(), ctx, torch.from_numpy(S.astype(np.float32)).cuda(),
                                torch.from_numpy(qbs).cuda(), torch.from_numpy(qns).cuda(), 1.0, out,
                                k_norms=torch.from_numpy(kn).cuda(), v_norms=torch.from_numpy(vn).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert rel_l2(got, want) <= ATTN_TOL, rel_l2(got, want)
    plain = orc.attn_decode(q.astype(np.float64), krec, vrec, 1.0)
    assert rel_l2(plain, want) > 10 * ATTN_TOL
