"""GPU parity of calibrate / alloc / encode / decode against the oracle.

Each stage sees identical inputs: the oracle's plan is copied to the device
for encode and decode, the oracle's fp32 eigenvalues feed the device
allocation, the oracle's streams feed the device decode.  Sizes span several
32-token groups and 128-token tiles with a ragged tail."""
import numpy as np
import pytest
import torch

import synth
from parity import (ATTN_TOL, BAND_SIGMA, FLIP_FRAC, REC_TOL, bf16, compare_codes, gpu_plan,
                    rel_l2)

pytestmark = pytest.mark.gpu

FAMILY = {"tc": 2, "generic": 1}


@pytest.fixture(params=["tc", "generic"])
def path(request):
    """Kernel family for bf16 head_dim-128 encode/decode: the tensor-core
    kernels (required: a call they do not cover fails) or the CUDA-core
    kernels."""
    import kv_cache_transform_encode_b300 as spx
    prev = spx.spectra_get_kernel_family()
    spx.spectra_set_kernel_family(FAMILY[request.param])
    yield request.param
    spx.spectra_set_kernel_family(prev)


@pytest.fixture(scope="module")
def spx():
    import kv_cache_transform_encode_b300 as spx
    spx.lib()
    assert torch.cuda.is_available()
    return spx


# ---------------------------------------------------------------- inputs
def tiny_case():
    x = synth.tiny_gaussian(0, T=256, H=2, d=64)            # fp32
    return x, torch.from_numpy(x).cuda(), x.astype(np.float64)


def llama_case(T=1000, H=8, seed=1, role=synth.ROLE_K):
    x = synth.to_bf16_exact(synth.spiked_t(seed, T, H, 128, role=role))
    return x, bf16(x).cuda(), x.astype(np.float64)


# ---------------------------------------------------------------- calibrate
@pytest.mark.parametrize("case", ["tiny", "llama"])
def test_calibrate_matches_oracle(spx, orc, path, case):
    """Gram (tcgen05 for the bf16 d = 128 cache on the tensor-core family,
    CUDA cores otherwise) and Jacobi eigenbasis against the oracle."""
    if case == "tiny":
        x, xd, x64 = tiny_case()
        n = 128
    else:
        x, xd, x64 = llama_case(T=2048)
        n = 2048
    H, d = x.shape[1], x.shape[2]
    p = spx.Plan(H, d)
    gram = torch.zeros((H, d, d), device="cuda")
    spx.spectra_calibrate(p, xd, n_cal=n, gram_out=gram)
    torch.cuda.synchronize()
    st = p.status.cpu().numpy()
    assert np.all(st >= 0), st
    lam_g, Q_g, G_g = p.eigvals.cpu().double().numpy(), p.basis_mat.cpu().double().numpy(), gram.cpu().double().numpy()
    for h in range(H):
        G = orc.gram(x64[:n, h, :])
        assert rel_l2(G_g[h], G) < 1e-5
        lam, Q, _ = orc.jacobi_eigh(G)
        g2 = np.linalg.norm(G, 2)
        # spectral norms: the fp32 round-off floor of a d=128 Jacobi is ~1e-5
        # in Frobenius norm, ~2e-6 in the 2-norm
        assert np.max(np.abs(lam_g[h] - lam)) <= 1e-5 * lam[0]
        assert np.linalg.norm(G @ Q_g[h] - Q_g[h] * lam_g[h][None, :], 2) <= 1e-5 * g2
        assert np.linalg.norm(Q_g[h].T @ Q_g[h] - np.eye(d), 2) <= 1e-5
        gap = np.minimum(np.abs(np.diff(np.r_[np.inf, lam])), np.abs(np.diff(np.r_[lam, -np.inf])))
        for c in np.nonzero(gap > 1e-3 * lam[0])[0]:
            np.testing.assert_allclose(Q_g[h][:, c], Q[:, c], atol=1e-3)   # same sign rule


def test_calibrate_nonfinite_status(spx):
    x = torch.zeros((64, 2, 64), device="cuda")
    x[5, 1, 3] = float("nan")
    p = spx.Plan(2, 64)
    spx.spectra_calibrate(p, x)
    torch.cuda.synchronize()
    st = p.status.cpu().numpy()
    assert st[0] >= 0 and st[1] == -6


# ---------------------------------------------------------------- alloc
def _alloc_gpu(spx, lam32, B, fixed=0):
    H, d = lam32.shape
    p = spx.Plan(H, d)
    p.eigvals.copy_(torch.from_numpy(lam32.astype(np.float32)))
    spx.spectra_alloc_bits(p, B, fixed)
    return p.bits.cpu().numpy(), p.rec_bits.cpu().numpy(), p.max_rec_bits


@pytest.mark.parametrize("B", [0.0, 0.5, 1.33, 2.0, 4.0, 7.5, 8.0, 16.0])
def test_alloc_bit_exact(spx, orc, B):
    x, _, x64 = llama_case(T=2048)
    lam, _ = orc.calibrate(x64)
    lam32 = lam.astype(np.float32)
    bits, rec, R = _alloc_gpu(spx, lam32, B)
    Rt = orc.total_bits(B, 128)
    assert R == Rt
    for h in range(lam32.shape[0]):
        want = orc.alloc(lam32[h].astype(np.float64), Rt)
        assert np.array_equal(bits[h], want), h
        assert rec[h] == Rt


def test_alloc_ties_and_zeros(spx, orc):
    """Ties across channels (equal eigenvalues, 4x multiples), zero and
    negative eigenvalues: the device selection reproduces the greedy order."""
    g = np.random.default_rng(0)
    rows = [np.repeat([4.0, 1.0, 0.25], [40, 40, 48]),
            np.r_[np.full(64, 2.0), np.zeros(32), -np.ones(32)],
            g.choice([16.0, 4.0, 1.0, 0.0], 128),
            np.zeros(128)]
    lam32 = np.stack(rows).astype(np.float32)
    for B in (0.3, 1.0, 2.5, 6.0, 8.0):
        bits, _, _ = _alloc_gpu(spx, lam32, B)
        for h in range(len(rows)):
            assert np.array_equal(bits[h], orc.alloc(lam32[h].astype(np.float64), orc.total_bits(B, 128))), (B, h)


def test_alloc_fixed_bits(spx):
    bits, rec, R = _alloc_gpu(spx, np.ones((3, 64), np.float32), 0.0, fixed=3)
    assert np.all(bits == 3) and np.all(rec == 192) and R == 192


# ---------------------------------------------------------------- encode/decode
def _roundtrip(spx, orc, oplan, x, xd, T, out_dtype=torch.float32):
    H, d = oplan.bits.shape
    p = gpu_plan(spx, oplan)
    codes = p.new_streams(T)
    norms = torch.zeros((H, T), device="cuda") if oplan.basis_kind == orc.BASIS_RWHT else None
    spx.spectra_encode(p, xd, codes, norms=norms)
    out = torch.zeros((T, H, d), device="cuda", dtype=out_dtype)
    spx.spectra_decode(p, codes, T, out, norms=norms)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() >= 0)
    return p, codes.cpu().numpy(), (norms.cpu().numpy() if norms is not None else None), out


def _check_codec(spx, orc, oplan, x64, xd, T):
    H = oplan.bits.shape[0]
    p, codes, norms, out = _roundtrip(spx, orc, oplan, x64, xd, T)
    flips = total = 0
    encs = orc.encode(oplan, x64)
    for h in range(H):
        f, n = compare_codes(orc, oplan, h, encs[h], codes[h], T)
        flips, total = flips + f, total + n
        if oplan.basis_kind == orc.BASIS_RWHT:
            np.testing.assert_allclose(norms[h], encs[h]["norms"], rtol=1e-5)
    assert flips <= FLIP_FRAC * max(total, 1), (flips, total)
    # decode parity on the ORACLE's streams
    streams = [e["stream"] for e in encs]
    sb = p.stream_bytes(T)
    cd = torch.zeros((H, max(sb, 16)), dtype=torch.uint8)
    for h in range(H):
        cd[h, :len(streams[h])] = torch.from_numpy(streams[h])
    cd = cd.cuda()
    nd = torch.from_numpy(np.stack([e["norms"] for e in encs])).cuda() if oplan.basis_kind == orc.BASIS_RWHT else None
    xh = orc.decode(oplan, streams, T, None if nd is None else [e["norms"] for e in encs])
    for dt in (torch.float32, torch.bfloat16):
        out = torch.zeros((T, H, x64.shape[2]), device="cuda", dtype=dt)
        spx.spectra_decode(p, cd, T, out, norms=nd)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        want = xh if dt == torch.float32 else synth.to_bf16_exact(xh.astype(np.float32))
        assert rel_l2(got, want) <= REC_TOL, (dt, rel_l2(got, want))
    return flips, total


def test_codec_tiny_fp32_d64(spx, orc):
    x, xd, x64 = tiny_case()
    oplan = orc.make_eigen_plan(x64[:128], 2.0)
    assert int(oplan.rec_bits()[0]) == 128
    _check_codec(spx, orc, oplan, x64, xd, 256)


@pytest.mark.parametrize("B,quant", [(2.0, 0), (4.0, 1), (2.0, 1), (1.33, 1), (16.0, 0)])
def test_codec_llama_bf16(spx, orc, path, B, quant):
    x, xd, x64 = llama_case(T=1000)
    oplan = orc.make_eigen_plan(x64[:512], B, quant)
    _check_codec(spx, orc, oplan, x64, xd, 1000)


def test_codec_rwht_lloyd3(spx, orc, path):
    x, xd, x64 = llama_case(T=700, H=6, seed=3)
    oplan = orc.make_rwht_plan(synth.rwht_signs(3, 6, 128), 3)
    _check_codec(spx, orc, oplan, x64, xd, 700)


def test_codec_zero_bit_channels(spx, orc, path):
    """0.5 bits/value on a steep spectrum: dropped channels take no bits and
    decode to exactly their zero latent coordinate."""
    x, xd, x64 = llama_case(T=300, H=2)
    oplan = orc.make_eigen_plan(x64, 0.5)
    assert (oplan.bits == 0).any()
    _check_codec(spx, orc, oplan, x64, xd, 300)


@pytest.mark.parametrize("T", [1, 31, 32, 33, 127, 129, 255, 257, 1000])
def test_codec_ragged_lengths(spx, orc, path, T):
    x, xd, x64 = llama_case(T=T, H=2, seed=5)
    x2, _, x642 = llama_case(T=256, H=2, seed=5)
    oplan = orc.make_eigen_plan(x642, 2.0)
    _check_codec(spx, orc, oplan, x64, xd, T)


@pytest.mark.parametrize("kind", ["uniform", "lloyd", "rwht", "mixed"])
def test_encode_decode_kv_matches_oracle(spx, orc, path, kind):
    """spectra_encode_kv / spectra_decode_kv (K and V of a layer in one call; one launch on the
    tensor-core family when both plans share basis and quantizer, two
    otherwise -- "mixed" pairs a uniform K plan with a Lloyd-Max V plan):
    each half's codes against the oracle under the band rule, and byte for
    byte against two spectra_encode calls."""
    T, H = 1000, 3
    xk, kd, k64 = llama_case(T=T, H=H, seed=11, role=synth.ROLE_K)
    xv, vd, v64 = llama_case(T=T, H=H, seed=11, role=synth.ROLE_V)
    if kind == "rwht":
        kpl = orc.make_rwht_plan(synth.rwht_signs(11, H, 128), 3)
        vpl = orc.make_rwht_plan(synth.rwht_signs(12, H, 128), 3)
    else:
        kpl = orc.make_eigen_plan(k64[:512], 2.0, 1 if kind == "lloyd" else 0)
        vpl = orc.make_eigen_plan(v64[:512], 1.33, 0 if kind == "uniform" else 1)
    kp, vp = gpu_plan(spx, kpl), gpu_plan(spx, vpl)
    sb = max(kp.stream_bytes(T), vp.stream_bytes(T), 16)
    kc, vc, kc1, vc1 = (torch.zeros((H, sb), dtype=torch.uint8, device="cuda") for _ in range(4))
    rw = kind == "rwht"
    kn, vn, kn1, vn1 = ((torch.zeros((H, T), device="cuda") if rw else None) for _ in range(4))
    spx.spectra_encode_kv(kp, vp, kd, vd, kc, vc, k_norms=kn, v_norms=vn)
    spx.spectra_encode(kp, kd, kc1, norms=kn1)
    spx.spectra_encode(vp, vd, vc1, norms=vn1)
    torch.cuda.synchronize()
    assert torch.equal(kc, kc1) and torch.equal(vc, vc1)
    if rw:
        assert torch.equal(kn, kn1) and torch.equal(vn, vn1)
    # decode_kv of the same streams: equal to two spectra_decode calls, and to
    # the oracle's reconstruction within the decode bar
    for dt in (torch.float32, torch.bfloat16):
        ko, vo, ko1, vo1 = (torch.zeros((T, H, 128), device="cuda", dtype=dt) for _ in range(4))
        spx.spectra_decode_kv(kp, vp, kc, vc, T, ko, vo, k_norms=kn, v_norms=vn)
        spx.spectra_decode(kp, kc, T, ko1, norms=kn)
        spx.spectra_decode(vp, vc, T, vo1, norms=vn)
        torch.cuda.synchronize()
        assert torch.equal(ko, ko1) and torch.equal(vo, vo1)
    for opl, out, codes, nrm in ((kpl, ko, kc, kn), (vpl, vo, vc, vn)):
        streams = [codes[h].cpu().numpy() for h in range(H)]
        want = orc.decode(opl, streams, T, None if nrm is None else [nrm[h].cpu().numpy() for h in range(H)])
        assert rel_l2(out.float().cpu().numpy(), bf16(want).float().numpy()) <= REC_TOL
    for opl, x64, codes, nrm in ((kpl, k64, kc, kn), (vpl, v64, vc, vn)):
        encs = orc.encode(opl, x64)
        flips = total = 0
        for h in range(H):
            f, n = compare_codes(orc, opl, h, encs[h], codes[h].cpu().numpy(), T)
            flips, total = flips + f, total + n
            if rw:
                np.testing.assert_allclose(nrm[h].cpu().numpy(), encs[h]["norms"], rtol=1e-5)
        assert flips <= FLIP_FRAC * max(total, 1), (flips, total)


def test_codec_empty(spx, orc, path):
    x, xd, x64 = llama_case(T=64, H=2)
    oplan = orc.make_eigen_plan(x64, 2.0)
    p = gpu_plan(spx, oplan)
    codes = p.new_streams(64)
    spx.spectra_encode(p, xd[:0], codes, T=0)
    out = torch.zeros((0, 2, 128), device="cuda")
    spx.spectra_decode(p, codes, 0, out)
    torch.cuda.synchronize()
    assert codes.sum().item() == 0


def test_end_to_end_device_plan(spx, orc, path):
    """Whole path on the device (calibrate -> alloc -> encode -> decode) vs
    the oracle's whole path: allocations agree and reconstruction errors
    match.  A differing width may only come from a near-tie in the greedy
    order; it is reported, not hidden."""
    x, xd, x64 = llama_case(T=4096, H=8, seed=7)
    oplan = orc.make_eigen_plan(x64[:2048], 2.0)
    p = spx.Plan(8, 128)
    spx.spectra_calibrate(p, xd, n_cal=2048)
    spx.spectra_alloc_bits(p, 2.0)
    codes = p.new_streams(4096)
    spx.spectra_encode(p, xd, codes)
    out = torch.zeros((4096, 8, 128), device="cuda")
    spx.spectra_decode(p, codes, 4096, out)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() >= 0)
    bits = p.bits.cpu().numpy()
    lam_g = p.eigvals.cpu().numpy().astype(np.float64)
    R = orc.total_bits(2.0, 128)
    for h in range(8):
        # bit-exact on the device's own eigenvalues ...
        assert np.array_equal(bits[h], orc.alloc(lam_g[h], R)), h
        # ... and every width that differs from the oracle's end-to-end plan
        # sits at a near-tie of the greedy order: the one-bit step one side
        # took and the other did not has a key lam_c 4^-j within the two
        # sides' eigenvalue difference of the cut between taken and untaken
        # keys (reported in the message)
        lam_o = oplan.eigvals[h]
        keys = np.sort(np.concatenate([np.maximum(lam_o, 0) * 4.0 ** -j for j in range(8)]))[::-1]
        cut = np.sqrt(keys[R - 1] * keys[R])
        for c in np.nonzero(bits[h] != oplan.bits[h])[0]:
            j = int(min(bits[h, c], oplan.bits[h, c]))
            margin = abs(np.log(lam_o[c] * 4.0 ** -j / cut))
            # channels whose last taken or first untaken key sits near the cut
            lo = np.maximum(lam_o, 1e-30) * 4.0 ** -oplan.bits[h].astype(float)
            near = (np.abs(np.log(4 * lo / cut)) < 0.05) | (np.abs(np.log(lo / cut)) < 0.05)
            lam_err = np.max(np.abs(np.log(np.maximum(lam_g[h][near | (np.arange(128) == c)], 1e-30)
                                           / np.maximum(lam_o[near | (np.arange(128) == c)], 1e-30))))
            assert margin <= 2 * lam_err + 1e-6, (h, c, bits[h, c], oplan.bits[h, c], margin, lam_err)
            print(f"head {h} channel {c}: width {bits[h, c]} vs {oplan.bits[h, c]}, "
                  f"relative distance to the greedy cut {margin:.2e} (eigenvalue difference {lam_err:.2e})")
    xo = orc.decode(oplan, [e["stream"] for e in orc.encode(oplan, x64)], 4096)
    e_gpu, e_orc = orc.relmse(x64, out.cpu().numpy()), orc.relmse(x64, xo)
    assert abs(e_gpu - e_orc) <= 0.05 * e_orc, (e_gpu, e_orc)


def test_codec_multi_head_tiles(spx, orc, path):
    """More (head, tile) work items than SMs: persistent CTAs walk ranges
    that cross head boundaries and reload the head's operand image."""
    x, xd, x64 = llama_case(T=5000, H=8, seed=11)
    oplan = orc.make_eigen_plan(x64[:1024], 2.0)
    _check_codec(spx, orc, oplan, x64, xd, 5000)


def test_codec_full_size_sampled(spx, orc, path):
    """Llama-shaped layer at full size (32768 tokens x 8 heads, 2.0
    bits/value), the launch the benchmark times: codes of 2048 sampled tokens
    per head against the oracle's encode of those tokens (band rule), and the
    decode of the device's own codes against the oracle's decode of the same
    codes on those tokens."""
    T, H = 32768, 8
    x = synth.to_bf16_exact(synth.spiked_t(21, T, H, 128))
    x64 = x.astype(np.float64)
    oplan = orc.make_eigen_plan(x64[:2048], 2.0)
    p = gpu_plan(spx, oplan)
    xd = bf16(x).cuda()
    codes = p.new_streams(T)
    spx.spectra_encode(p, xd, codes)
    out = torch.zeros((T, H, 128), device="cuda", dtype=torch.bfloat16)
    spx.spectra_decode(p, codes, T, out)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() >= 0)
    g = np.random.default_rng(5)
    idx = np.sort(g.choice(T, size=2048, replace=False))
    idx[:2] = [0, T - 1]
    cc = codes.cpu().numpy()
    outn = out.float().cpu().numpy()
    flips = total = 0
    for h in range(H):
        R = int(oplan.rec_bits()[h])
        got = orc.unpack(np.ascontiguousarray(cc[h, : orc.stream_bytes(T, R)]), T, oplan.bits[h])[idx]
        enc = orc.encode_head(oplan, h, x64[idx, h, :])
        diff = got != enc["codes"]
        if diff.any():
            assert orc.decision_margin(oplan, h, enc)[diff].max() <= BAND_SIGMA
        flips += int(diff.sum())
        total += diff.size
        # decode of the device's codes for the sampled tokens
        sub = orc.pack(got, oplan.bits[h])
        xh = orc.decode_head(oplan, h, sub, len(idx))
        want = synth.to_bf16_exact(xh.astype(np.float32))
        assert rel_l2(outn[idx, h, :], want) <= REC_TOL
    assert flips <= FLIP_FRAC * total, (flips, total)


# ---------------------------------------------------------------- device status words
@pytest.mark.parametrize("case", ["tiny", "llama"])
def test_calibrate_not_converged_status(spx, case):
    """One Jacobi sweep cannot converge on these spectra: every head reports
    -SPECTRA_ERR_NOT_CONVERGED through plan.status (no trap, no hang), and the
    next call with the default sweep budget converges on the same plan."""
    if case == "tiny":
        _, xd, _ = tiny_case()
        n = 128
    else:
        _, xd, _ = llama_case(T=2048)
        n = 2048
    H, d = xd.shape[1], xd.shape[2]
    p = spx.Plan(H, d)
    spx.spectra_calibrate(p, xd, n_cal=n, max_sweeps=1)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() == -4), p.status.cpu().numpy()
    spx.spectra_calibrate(p, xd, n_cal=n)
    torch.cuda.synchronize()
    assert np.all(p.status.cpu().numpy() > 0)


def test_buffer_status(spx, orc, path):
    """A head whose record is longer than plan.max_rec_bits (the bound the
    streams were sized by) is refused on the device: plan_finalize and the
    encode report -SPECTRA_ERR_BUFFER for it and write none of its codes; the
    other head is encoded and decoded normally."""
    T = 300
    x, xd, x64 = llama_case(T=T, H=2)
    oplan = orc.make_eigen_plan(x64, 2.0)
    oplan.bits[1] = np.minimum(oplan.bits[1], 1)
    R1 = int(oplan.rec_bits()[1])
    assert R1 < int(oplan.rec_bits()[0])
    p = gpu_plan(spx, oplan)
    p.max_rec_bits = R1
    spx.spectra_plan_finalize(p)
    torch.cuda.synchronize()
    st = p.status.cpu().numpy()
    assert st[0] == -7 and st[1] >= 0, st
    codes = p.new_streams(T)
    spx.spectra_encode(p, xd, codes)
    out = torch.full((T, 2, 128), 5.0, device="cuda")
    spx.spectra_decode(p, codes, T, out)
    torch.cuda.synchronize()
    st = p.status.cpu().numpy()
    assert st[0] == -7 and st[1] >= 0, st
    cc = codes.cpu().numpy()
    assert not cc[0].any()
    enc = orc.encode_head(oplan, 1, x64[:, 1, :])
    compare_codes(orc, oplan, 1, enc, cc[1], T)
    want = orc.decode_head(oplan, 1, enc["stream"], T)
    assert rel_l2(out[:, 1, :].cpu().numpy(), want) <= 5 * REC_TOL


def test_bounded_wait_gives_up_and_context_survives(spx, orc):
    """The library's bounded waits on a barrier that nothing arrives on: every
    waiter gives up with SPECTRA_ERR_TIMEOUT after the limit (the single-thread
    spin and a suspending warp, through the shared abort flag), the kernel
    returns, and the context keeps working (an ordinary encode/decode after
    it is still exact against the oracle)."""
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    for limit in (2_000, 200_000):
        spx.spectra_selftest_wait(limit, st, el)
        torch.cuda.synchronize()
        assert st[0].item() == -5 and st[1].item() == 33, st.tolist()
        assert limit // 2 <= el.item() < limit + 5_000_000, (limit, el.item())
    x, xd, x64 = llama_case(T=300, H=2, seed=2)
    _check_codec(spx, orc, orc.make_eigen_plan(x64, 2.0), x64, xd, 300)
