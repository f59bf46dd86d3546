"""GPU parity of the packed-cache decode-step attention against the oracle's
fp64 attention over the same reconstructed cache (identical plans, streams
and queries on both sides).  Shapes span several context splits, 64-token
tiles and a ragged tail, with grouped-query heads."""
import numpy as np
import pytest
import torch

import synth
from parity import ATTN_TOL, gpu_plan, rel_l2

pytestmark = pytest.mark.gpu

FAMILY = {"tc": 2, "generic": 1}


@pytest.fixture(params=["tc", "generic"])
def path(request):
    """Kernel family: the tensor-core kernels (required: bit-plane for
    uniform eigenbasis plans with <= 4 query heads per kv head, level-table
    otherwise) or the CUDA-core kernels."""
    import kv_cache_transform_encode_b300 as spx
    prev = spx.spectra_get_kernel_family()
    spx.spectra_set_kernel_family(FAMILY[request.param])
    yield request.param
    spx.spectra_set_kernel_family(prev)


@pytest.fixture(scope="module")
def spx():
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    return spx


def _setup(orc, B, Hkv, ctx, d=128, kind="eigen", B_bits=2.0, quant=0, seed=11):
    """Oracle plans from batch element 0's first tokens; per-batch caches."""
    kx = [synth.to_bf16_exact(synth.spiked_t(seed + b, ctx, Hkv, d, role=synth.ROLE_K)).astype(np.float64)
          for b in range(B)]
    vx = [synth.to_bf16_exact(synth.spiked_t(seed + b, ctx, Hkv, d, role=synth.ROLE_V)).astype(np.float64)
          for b in range(B)]
    if kind == "eigen":
        kp = orc.make_eigen_plan(kx[0][: min(ctx, 2048)], B_bits, quant)
        vp = orc.make_eigen_plan(vx[0][: min(ctx, 2048)], B_bits, quant)
    else:
        kp = orc.make_rwht_plan(synth.rwht_signs(seed, Hkv, d), 3)
        vp = orc.make_rwht_plan(synth.rwht_signs(seed + 1, Hkv, d), 3)
    return kx, vx, kp, vp


def _streams(orc, plan, xs, ctx):
    """Oracle-encoded streams [B*Hkv] (+ norms) and reconstructions."""
    encs = [orc.encode(plan, x) for x in xs]
    rec = np.stack([orc.decode(plan, [e["stream"] for e in en], ctx,
                               [e["norms"] for e in en] if plan.basis_kind == orc.BASIS_RWHT else None)
                    for en in encs])                      # [B, ctx, Hkv, d]
    flat = [e for en in encs for e in en]
    sb = max(len(e["stream"]) for e in flat)
    st = np.zeros((len(flat), max(sb, 16)), dtype=np.uint8)
    for i, e in enumerate(flat):
        st[i, : len(e["stream"])] = e["stream"]
    norms = (np.stack([e["norms"] for e in flat]) if plan.basis_kind == orc.BASIS_RWHT else None)
    return st, norms, rec


def _run(spx, orc, B, Hq, Hkv, ctx, kind="eigen", quant=0, B_bits=2.0, scale=1.0, q=None):
    kx, vx, kp, vp = _setup(orc, B, Hkv, ctx, kind=kind, quant=quant, B_bits=B_bits)
    ks, kn, krec = _streams(orc, kp, kx, ctx)
    vs, vn, vrec = _streams(orc, vp, vx, ctx)
    if q is None:
        q = synth.to_bf16_exact(synth.queries(5, B, Hq, 128))
    want = orc.attn_decode(q.astype(np.float64), krec, vrec, scale)
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    stride = max(ks.shape[1], vs.shape[1])
    kd = torch.zeros((ks.shape[0], stride), dtype=torch.uint8)
    vd = torch.zeros((vs.shape[0], stride), dtype=torch.uint8)
    kd[:, : ks.shape[1]] = torch.from_numpy(ks)
    vd[:, : vs.shape[1]] = torch.from_numpy(vs)
    out = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(), kd.cuda(), vd.cuda(),
                            ctx, scale, out,
                            k_norms=None if kn is None else torch.from_numpy(kn).cuda(),
                            v_norms=None if vn is None else torch.from_numpy(vn).cuda())
    torch.cuda.synchronize()
    return out.cpu().numpy(), want


@pytest.mark.parametrize("ctx", [1, 100, 2048, 4500])
def test_attn_uniform_gqa(spx, orc, path, ctx):
    got, want = _run(spx, orc, B=2, Hq=8, Hkv=2, ctx=ctx)
    assert rel_l2(got, want) <= ATTN_TOL, rel_l2(got, want)


def test_attn_lloyd(spx, orc, path):
    got, want = _run(spx, orc, B=1, Hq=4, Hkv=1, ctx=3000, quant=1, B_bits=1.33)
    assert rel_l2(got, want) <= ATTN_TOL


@pytest.mark.parametrize("B_bits", [4.0, 1.33, 8.0])
def test_attn_uniform_budgets(spx, orc, path, B_bits):
    """Other budgets, including 8-bit channels (codes up to 255)."""
    got, want = _run(spx, orc, B=1, Hq=4, Hkv=1, ctx=1500, quant=0, B_bits=B_bits)
    assert rel_l2(got, want) <= ATTN_TOL


@pytest.mark.parametrize("G", [1, 2])
def test_attn_small_groups(spx, orc, path, G):
    """Fewer query heads per kv head than the tensor-core tile holds."""
    got, want = _run(spx, orc, B=2, Hq=2 * G, Hkv=2, ctx=700)
    assert rel_l2(got, want) <= ATTN_TOL


def test_attn_rwht(spx, orc, path):
    got, want = _run(spx, orc, B=2, Hq=4, Hkv=2, ctx=1200, kind="rwht")
    assert rel_l2(got, want) <= ATTN_TOL


def test_attn_peaky_scores(spx, orc, path):
    """Sharper softmax (scale 4 on N(0,1/d) queries): still within tolerance."""
    got, want = _run(spx, orc, B=1, Hq=8, Hkv=2, ctx=2500, scale=4.0)
    assert rel_l2(got, want) <= ATTN_TOL


@pytest.fixture
def tc_only():
    import kv_cache_transform_encode_b300 as spx
    prev = spx.spectra_get_kernel_family()
    spx.spectra_set_kernel_family(FAMILY["tc"])
    yield
    spx.spectra_set_kernel_family(prev)


def test_attn_full_layer_sampled(spx, orc, tc_only):
    """The benchmark's attention launch (1 x 32 query heads over 8 kv heads,
    32768 tokens at 2.0 bits/value) on the tensor-core kernels; the oracle's
    fp64 attention checked on the query heads of kv heads 0 and 5."""
    B, Hq, Hkv, ctx = 1, 32, 8, 32768
    kx = [synth.to_bf16_exact(synth.spiked_t(31, ctx, Hkv, 128, role=synth.ROLE_K)).astype(np.float64)]
    vx = [synth.to_bf16_exact(synth.spiked_t(31, ctx, Hkv, 128, role=synth.ROLE_V)).astype(np.float64)]
    kp = orc.make_eigen_plan(kx[0][:2048], 2.0)
    vp = orc.make_eigen_plan(vx[0][:2048], 2.0)
    kenc, venc = orc.encode(kp, kx[0]), orc.encode(vp, vx[0])
    stride = max(max(len(e["stream"]) for e in kenc), max(len(e["stream"]) for e in venc))
    kd = torch.zeros((Hkv, stride), dtype=torch.uint8)
    vd = torch.zeros((Hkv, stride), dtype=torch.uint8)
    for h in range(Hkv):
        kd[h, : len(kenc[h]["stream"])] = torch.from_numpy(kenc[h]["stream"])
        vd[h, : len(venc[h]["stream"])] = torch.from_numpy(venc[h]["stream"])
    q = synth.to_bf16_exact(synth.queries(9, B, Hq, 128))
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(), kd.cuda(), vd.cuda(),
                            ctx, 1.0, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    G = Hq // Hkv
    for h in (0, 5):
        kr = orc.decode_head(kp, h, kenc[h]["stream"], ctx)
        vr = orc.decode_head(vp, h, venc[h]["stream"], ctx)
        for j in range(G):
            want = orc.attention(q[0, h * G + j].astype(np.float64), kr, vr, 1.0)
            assert rel_l2(got[0, h * G + j], want) <= ATTN_TOL, (h, j)


def test_attn_empty_context(spx, orc):
    kx, vx, kp, vp = _setup(orc, 1, 2, 64)
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.full((1, 4, 128), 7.0, device="cuda")
    codes = torch.zeros((2, 16), dtype=torch.uint8, device="cuda")
    spx.spectra_attn_decode(gk, gv, torch.zeros((1, 4, 128), device="cuda"), codes, codes, 0, 1.0, out)
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0


def _single_head_cache(seed, ctx, role):
    return synth.to_bf16_exact(synth.spiked_t(seed, ctx, 1, 128, role=role))[:, 0, :].astype(np.float64)


def _batched_case(spx, orc, B, Hq, Hkv, ctx, checked, seed=71, B_bits=2.0, quant=0):
    """Plans per kv head from their own first 2048 tokens; the streams of the
    (batch, kv head) pairs in `checked` hold oracle-encoded synthetic caches,
    every other stream seeded random code words (every bit pattern is a valid
    code, so the kernels do the full work everywhere).  Returns the device
    output and, for each checked pair, the oracle's reconstruction."""
    cal_k = np.stack([_single_head_cache(seed * 100 + h, 2048, synth.ROLE_K) for h in range(Hkv)], 1)
    cal_v = np.stack([_single_head_cache(seed * 100 + h, 2048, synth.ROLE_V) for h in range(Hkv)], 1)
    kp = orc.make_eigen_plan(cal_k, B_bits, quant)
    vp = orc.make_eigen_plan(cal_v, B_bits, quant)
    sb = max(orc.stream_bytes(ctx, int(kp.rec_bits().max())), orc.stream_bytes(ctx, int(vp.rec_bits().max())), 16)
    g = np.random.default_rng(seed)
    ks = g.integers(0, 256, (B * Hkv, sb), dtype=np.uint8)
    vs = g.integers(0, 256, (B * Hkv, sb), dtype=np.uint8)
    rec = {}
    for (b, h) in checked:
        xk = _single_head_cache(seed * 1000 + 17 * b + h, ctx, synth.ROLE_K)
        xv = _single_head_cache(seed * 1000 + 17 * b + h, ctx, synth.ROLE_V)
        ek, ev = orc.encode_head(kp, h, xk), orc.encode_head(vp, h, xv)
        ks[b * Hkv + h] = 0
        vs[b * Hkv + h] = 0
        ks[b * Hkv + h, : len(ek["stream"])] = ek["stream"]
        vs[b * Hkv + h, : len(ev["stream"])] = ev["stream"]
        rec[(b, h)] = (orc.decode_head(kp, h, ek["stream"], ctx), orc.decode_head(vp, h, ev["stream"], ctx))
    # tails of random streams past the last token are never read; the
    # oracle-encoded ones are zero-padded like the library's
    q = synth.to_bf16_exact(synth.queries(seed, B, Hq, 128))
    gk, gv = gpu_plan(spx, kp), gpu_plan(spx, vp)
    out = torch.zeros((B, Hq, 128), device="cuda")
    spx.spectra_attn_decode(gk, gv, torch.from_numpy(q).to(torch.bfloat16).cuda(), torch.from_numpy(ks).cuda(),
                            torch.from_numpy(vs).cuda(), ctx, 1.0, out)
    torch.cuda.synchronize()
    return out.cpu().numpy(), q, rec


def _check_batched(orc, got, q, rec, Hq, Hkv):
    G = Hq // Hkv
    for (b, h), (kr, vr) in rec.items():
        for j in range(G):
            want = orc.attention(q[b, h * G + j].astype(np.float64), kr, vr, 1.0)
            err = rel_l2(got[b, h * G + j], want)
            assert err <= ATTN_TOL, ((b, h, j), err)


def test_attn_batched_many_splits(spx, orc, path):
    """Batch 8 x 32 query heads over 8 kv heads (256 (batch, query head)
    pairs, the long-split branch), 8192 + 37 tokens: five context splits
    with a ragged last one, merged per query head; checked on the query heads
    of four (batch, kv head) pairs."""
    B, Hq, Hkv, ctx = 8, 32, 8, 8192 + 37
    checked = [(0, 0), (3, 5), (7, 7), (5, 2)]
    got, q, rec = _batched_case(spx, orc, B, Hq, Hkv, ctx, checked)
    _check_batched(orc, got, q, rec, Hq, Hkv)


def test_attn_compressed_attention_workload_sampled(spx, orc):
    """The compressed-attention workload the benchmark times, at full size:
    batch 16, 32 query heads over 8 kv heads, 65536-token context at 2.0
    bits/value, on the default kernel family; the oracle's fp64 attention
    over its own reconstruction checked on three (batch, kv head) pairs
    (12 query heads), the other streams random code words."""
    B, Hq, Hkv, ctx = 16, 32, 8, 65536
    checked = [(0, 0), (15, 5), (7, 3)]
    got, q, rec = _batched_case(spx, orc, B, Hq, Hkv, ctx, checked, seed=73)
    _check_batched(orc, got, q, rec, Hq, Hkv)
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("kind,quant,G", [("eigen", 1, 4), ("rwht", 1, 4), ("eigen", 1, 8), ("rwht", 1, 7),
                                          ("eigen", 0, 8), ("eigen", 0, 5)])
def test_attn_plans_multi_split(spx, orc, path, kind, quant, G):
    """Lloyd-Max and RWHT plans, and uniform plans with more than four query
    heads per kv head (the level-table tensor-core kernel, or the CUDA-core
    one), over several context splits with a ragged last group."""
    got, want = _run(spx, orc, B=2, Hq=2 * G, Hkv=2, ctx=5000 + 29, kind=kind, quant=quant, B_bits=2.0)
    assert rel_l2(got, want) <= ATTN_TOL, rel_l2(got, want)


def test_attn_lloyd_batched_many_splits(spx, orc, path):
    """Lloyd-Max plans at 2.0 bits/value on the long-split branch: batch 8 x
    32 query heads over 8 kv heads, 8192 + 37 tokens, checked on four
    (batch, kv head) pairs."""
    B, Hq, Hkv, ctx = 8, 32, 8, 8192 + 37
    checked = [(0, 0), (3, 5), (7, 7), (5, 2)]
    got, q, rec = _batched_case(spx, orc, B, Hq, Hkv, ctx, checked, seed=79, quant=1)
    _check_batched(orc, got, q, rec, Hq, Hkv)
