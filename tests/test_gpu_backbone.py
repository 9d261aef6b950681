"""Drafter backbone (N1) through the C ABI against oracle/backbone.py.

Tolerances.  The kernels compute in fp32 and the oracle in fp64; both round to bf16 at
the same points.  A bf16 result can then differ by one ulp where the two values lie on
either side of a rounding boundary: the fp32 errors are ~1e-7 relative (sums of at most
a few thousand terms; the rotary angle is reduced in fp64), so such flips hit well under
0.5% of the elements.  Kernel tests (and the per-call checks of a layer, each on the GPU's own inputs):
norms and SiLU within 1 ulp with at most 0.5% off by one; sums of mixed-sign terms
(GEMMs, the rotation, attention) within one ulp plus the recursive-summation bound
n * 2^-24 * sum|terms|.  Chained (the oracle's whole layer stack from the same
weights): a flip of a bf16 activation perturbs every output of the next GEMM by about
2^-8 * sqrt(flip share) of its size, so the flip share grows from ~0.1% toward one half
over four or five GEMMs and h ends about one ulp (2^-8 relative) rms away; h is checked
to rms error <= 2^-7 rms(h) and max error <= 2^-4 rms(h).  Exact: the fp32 residual after an add, the
value heads written to the cache, cache slots outside the written range.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import bf16_ulp_diff, dev, dev_bf16, host, host_bf16_bits
from oracle import backbone as bb

pytestmark = pytest.mark.gpu


def _bits(x):
    """float64 values of bf16 numbers -> their bit patterns."""
    return syn.to_bf16_bits(np.asarray(x, dtype=np.float32))


def _vals(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def _close_ulp(got_bits, ref_vals, share=0.005):
    d = bf16_ulp_diff(np.asarray(got_bits).reshape(-1), _bits(ref_vals).reshape(-1))
    assert d.max() <= 1, "max ulp difference %d" % d.max()
    assert (d > 0).mean() <= share, "%.4f of the elements differ by one ulp" % (d > 0).mean()


def _close_sum(got_bits, ref_vals, mag, nterms):
    """A bf16 rounding of an fp32 sum of terms of mixed sign: within one bf16 ulp of the
    exact value plus the recursive-summation bound nterms * 2^-24 * sum|terms| (mag), and
    at most 1% of the elements more than one ulp away."""
    got = _vals(got_bits).reshape(-1)
    ref = np.asarray(ref_vals, dtype=np.float64).reshape(-1)
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    bound = ulp + nterms * 2.0 ** -24 * np.asarray(mag, dtype=np.float64).reshape(-1)
    assert np.all(np.abs(got - ref) <= bound), "max excess %.3e" % (np.abs(got - ref) - bound).max()
    d = bf16_ulp_diff(np.asarray(got_bits).reshape(-1), _bits(ref).reshape(-1))
    assert (d > 1).mean() < 0.01, "%.4f of the elements more than one ulp away" % (d > 1).mean()


def _layer_dev(L):
    return ds.BackboneLayer(L["nq"], L["nkv"], *[dev_bf16(L[k]) for k in
                                                  ("w_in", "w_post", "w_qn", "w_kn", "w_qkv", "w_o", "w_gu", "w_d")])


def _layer_ref(L):
    out = {k: (_vals(v) if isinstance(v, np.ndarray) else v) for k, v in L.items()}
    out["hd"] = 128
    return out


@pytest.mark.parametrize("M,N,K,out_bf16", [(8, 7168, 5120, True), (112, 300, 256, True),
                                            (7, 2048, 5120, False), (24, 5120, 17408, True)])
def test_linear_matches_oracle(M, N, K, out_bf16):
    x = syn.normal_bf16(300 + M, (M, K))
    w = syn.normal_bf16(301 + N, (N, K), (1.0 / K) ** 0.5)
    ref = _vals(x) @ _vals(w).T
    out = ds.linear(dev_bf16(x), dev_bf16(w), out_bf16=out_bf16)
    if out_bf16:
        _close_sum(host_bf16_bits(out), ref, np.abs(_vals(x)) @ np.abs(_vals(w)).T, K)
    else:
        bound = 1e-5 * (np.abs(_vals(x)) @ np.abs(_vals(w)).T) + 1e-30
        assert np.all(np.abs(host(out).astype(np.float64) - ref) <= bound)


def test_norm_kernels_match_oracle():
    H, V, rows, grp = 5120, 1000, 24, 8
    table = syn.normal_bf16(310, (V, H))
    tok = np.arange(rows, dtype=np.int32) * 37 % V
    w = syn.to_bf16_bits(1.0 + syn.normal_f32(311, (H,), 0.1))
    x, n = ds.embed_rmsnorm(dev_bf16(table), dev(tok), dev_bf16(w))
    xe = _vals(table)[tok]
    np.testing.assert_array_equal(host(x), xe.astype(np.float32))
    _close_ulp(host_bf16_bits(n), bb.rmsnorm(xe, _vals(w)))
    # residual add, the final norm leaving out the first row of each group of 8
    delta = syn.normal_bf16(312, (rows, H), 0.3)
    out = ds.add_rmsnorm(x, dev_bf16(delta), dev_bf16(w), group=grp)
    xs = (xe.astype(np.float32) + _vals(delta).astype(np.float32)).astype(np.float64)
    np.testing.assert_array_equal(host(x), xs.astype(np.float32))
    keep = np.arange(rows) % grp != 0
    _close_ulp(host_bf16_bits(out), bb.rmsnorm(xs[keep], _vals(w)))
    # a plain norm of bf16 rows
    inp = syn.normal_bf16(313, (rows, H), 2.0)
    _close_ulp(host_bf16_bits(ds.rmsnorm_bf16(dev_bf16(inp), dev_bf16(w))), bb.rmsnorm(_vals(inp), _vals(w)))


def test_embed_bad_token_is_recorded_and_clamped():
    H, V = 256, 50
    table = syn.normal_bf16(315, (V, H))
    w = syn.to_bf16_bits(np.ones(H, np.float32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x, _ = ds.embed_rmsnorm(dev_bf16(table), dev(np.array([3, -1, V], np.int32)), dev_bf16(w), status=st)
    assert int(st.item()) == -7   # DSPARK_ERR_BAD_TOKEN
    np.testing.assert_array_equal(host(x), _vals(table)[[3, 0, V - 1]].astype(np.float32))


def _pair_mag(y):
    """|y_d| + |y_{d+64}| of each rotary pair, at both of its dims (the terms of the
    rotated value)."""
    m = np.abs(y[..., :64]) + np.abs(y[..., 64:])
    return np.concatenate([m, m], axis=-1)


@pytest.mark.parametrize("nq,nkv,B,rows_per_req,pos0,cache_len", [(40, 8, 3, 8, 1024, 1040),
                                                                  (0, 8, 2, 7, 1017, 1040),
                                                                  (2, 1, 4, 5, 0, 9)])
def test_qk_norm_rope_matches_oracle(nq, nkv, B, rows_per_req, pos0, cache_len):
    rows = B * rows_per_req
    qkv = syn.normal_bf16(320 + nq, (rows, (nq + 2 * nkv) * 128), 0.7)
    wq = syn.to_bf16_bits(1.0 + syn.normal_f32(321, (128,), 0.1))
    wk = syn.to_bf16_bits(1.0 + syn.normal_f32(322, (128,), 0.1))
    sentinel = syn.normal_bf16(323, (B, cache_len, nkv, 128))
    kc, vc = dev_bf16(sentinel), dev_bf16(sentinel)
    q = ds.qk_norm_rope(dev_bf16(qkv), nq, nkv, dev_bf16(wq) if nq else None, dev_bf16(wk), 1e6, kc, vc,
                        rows_per_req, pos0)
    x = _vals(qkv)
    pos = pos0 + np.arange(rows) % rows_per_req
    kin = x[:, nq * 128:(nq + nkv) * 128].reshape(rows, nkv, 128)
    kref = bb.qk_norm_rope(kin, _vals(wk), pos)
    kgot, vgot = host_bf16_bits(kc), host_bf16_bits(vc)
    slots = np.arange(pos0, pos0 + rows_per_req)
    _close_sum(kgot[:, slots].reshape(rows, nkv, 128), kref, _pair_mag(bb.rmsnorm(kin, _vals(wk))), 16)
    np.testing.assert_array_equal(vgot[:, slots].reshape(rows, nkv * 128),
                                  qkv[:, (nq + nkv) * 128:])
    other = np.setdiff1d(np.arange(cache_len), slots)
    np.testing.assert_array_equal(kgot[:, other], sentinel[:, other])
    np.testing.assert_array_equal(vgot[:, other], sentinel[:, other])
    if nq:
        qin = x[:, :nq * 128].reshape(rows, nq, 128)
        qref = bb.qk_norm_rope(qin, _vals(wq), pos)
        _close_sum(host_bf16_bits(q), qref, _pair_mag(bb.rmsnorm(qin, _vals(wq))), 16)


@pytest.mark.parametrize("B,nr,nq,nkv,cache_len,nkeys", [(2, 8, 40, 8, 1040, 1032), (3, 8, 2, 1, 80, 70),
                                                         (1, 1, 40, 8, 64, 64), (2, 6, 8, 1, 200, 5)])
def test_attention_matches_oracle(B, nr, nq, nkv, cache_len, nkeys):
    q = syn.normal_bf16(330 + nkeys, (B, nr, nq, 128))
    kc = syn.normal_bf16(331 + nkeys, (B, cache_len, nkv, 128))
    vc = syn.normal_bf16(332 + nkeys, (B, cache_len, nkv, 128))
    out = host_bf16_bits(ds.attention(dev_bf16(q), dev_bf16(kc), dev_bf16(vc), nkeys))
    for b in range(B):
        ref = bb.attention(_vals(q[b]), _vals(kc[b, :nkeys]), _vals(vc[b, :nkeys]))
        mag = bb.attention(_vals(q[b]), _vals(kc[b, :nkeys]), np.abs(_vals(vc[b, :nkeys])))
        # terms: the nkeys products p.v, plus the scores' own fp32 error (128-term dot
        # products of unit-scale q and k) carried into every p
        _close_sum(out[b], ref, mag, nkeys + 2048)


def test_silu_mul_matches_oracle():
    M, I = 8, 17408
    gu = syn.normal_bf16(340, (M, 2 * I), 2.0)
    g, u = _vals(gu[:, :I]), _vals(gu[:, I:])
    _close_ulp(host_bf16_bits(ds.silu_mul(dev_bf16(gu))), bb.silu(g) * u)


def _backbone_case(H, nq, nkv, I, L, V, B, C, k, seed, stagewise=False):
    layers, wf = syn.backbone_weights(H, nq, nkv, I, L, seed=seed)
    E = syn.normal_bf16(seed + 100, (V, H), (1.0 / H) ** 0.5 * 8)
    ctx = syn.normal_bf16(seed + 101, (B, C, H))
    prev = (np.arange(B) * 7919 + 11) % (V - 1)
    toks = np.concatenate([prev[:, None], np.full((B, k), V - 1)], axis=1).astype(np.int32)
    nr = k + 1
    # GPU: the context's keys/values into the caches, then the block
    lay_d = [_layer_dev(l) for l in layers]
    kcs = [torch.zeros((B, C + nr, nkv, 128), dtype=torch.bfloat16, device="cuda") for _ in layers]
    vcs = [torch.zeros_like(t) for t in kcs]
    wsp = ds.Workspaces()
    ds.backbone_context(dev_bf16(ctx.reshape(B * C, H)), lay_d, kcs, vcs, 0, workspaces=wsp)
    h = ds.backbone_block(dev(toks), dev_bf16(E), lay_d, dev_bf16(wf), kcs, vcs, C, workspaces=wsp)
    hb = host_bf16_bits(h)
    ref_layers = [_layer_ref(l) for l in layers]
    Ev = _vals(E)
    if stagewise:
        _stagewise(lay_d[0], ref_layers[0], E, wf, ctx, toks, kcs[0], vcs[0], hb, C, nr, wsp)
    got = _vals(hb).reshape(B, k, H)
    for b in range(B):
        ref = bb.backbone(toks[b], _vals(ctx[b]), ref_layers, _vals(wf), Ev)
        err = got[b] - ref
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.sqrt(np.mean(err ** 2)) <= rms * 2.0 ** -7, (b, np.sqrt(np.mean(err ** 2)) / rms)
        assert np.abs(err).max() <= rms * 2.0 ** -4, (b, np.abs(err).max() / rms)


def _stagewise(ly, lr, E, wf, ctx, toks, kc, vc, h_bits, C, nr, wsp):
    """Re-runs one layer call by call and checks every call against the oracle on the
    GPU's own inputs (the tight check), and that the composite calls gave the same bits."""
    B, _, H = ctx.shape
    nq, nkv = lr["nq"], lr["nkv"]
    I = lr["w_d"].shape[1]
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    cx = dev_bf16(ctx.reshape(B * C, H))
    nrm = ds.rmsnorm_bf16(cx, ly.w_in)
    _close_ulp(host_bf16_bits(nrm), bb.rmsnorm(_vals(ctx.reshape(B * C, H)), lr["w_in"]))
    kv = ds.linear(nrm, ly.w_kv, workspaces=wsp, kind="t_kv")
    nv = _vals(host_bf16_bits(nrm))
    wkv = lr["w_qkv"][nq * 128:]
    _close_sum(host_bf16_bits(kv), nv @ wkv.T, np.abs(nv) @ np.abs(wkv).T, H)
    ds.qk_norm_rope(kv, 0, nkv, None, ly.w_kn, 1e6, kc2, vc2, C, 0)
    kvv = _vals(host_bf16_bits(kv))
    kin = kvv[:, :nkv * 128].reshape(B * C, nkv, 128)
    _close_sum(host_bf16_bits(kc2)[:, :C].reshape(B * C, nkv, 128),
               bb.qk_norm_rope(kin, lr["w_kn"], np.tile(np.arange(C), B)), _pair_mag(bb.rmsnorm(kin, lr["w_kn"])), 16)
    x, n = ds.embed_rmsnorm(dev_bf16(E), dev(toks.reshape(-1)), ly.w_in)
    xv = _vals(E)[toks.reshape(-1)]
    _close_ulp(host_bf16_bits(n), bb.rmsnorm(xv, lr["w_in"]))
    qkv = ds.linear(n, ly.w_qkv, workspaces=wsp, kind="t_qkv")
    nv = _vals(host_bf16_bits(n))
    _close_sum(host_bf16_bits(qkv), nv @ lr["w_qkv"].T, np.abs(nv) @ np.abs(lr["w_qkv"]).T, H)
    q = ds.qk_norm_rope(qkv, nq, nkv, ly.w_qn, ly.w_kn, 1e6, kc2, vc2, nr, C)
    np.testing.assert_array_equal(host_bf16_bits(kc2), host_bf16_bits(kc))   # the composite's cache
    np.testing.assert_array_equal(host_bf16_bits(vc2), host_bf16_bits(vc))
    o = ds.attention(q.view(B, nr, nq, 128), kc2, vc2, C + nr, workspaces=wsp)
    qg, Kg, Vg = _vals(host_bf16_bits(q)).reshape(B, nr, nq, 128), _vals(host_bf16_bits(kc2)), _vals(host_bf16_bits(vc2))
    ob = host_bf16_bits(o)
    for b in range(B):
        _close_sum(ob[b], bb.attention(qg[b], Kg[b], Vg[b]), bb.attention(qg[b], Kg[b], np.abs(Vg[b])),
                   C + nr + 2048)
    d = ds.linear(o.view(B * nr, nq * 128), ly.w_o, workspaces=wsp, kind="t_o")
    ov = _vals(ob).reshape(B * nr, nq * 128)
    _close_sum(host_bf16_bits(d), ov @ lr["w_o"].T, np.abs(ov) @ np.abs(lr["w_o"]).T, nq * 128)
    x0 = host(x)
    n2 = ds.add_rmsnorm(x, d, ly.w_post)
    x1 = (x0 + _vals(host_bf16_bits(d)).astype(np.float32)).astype(np.float32)
    np.testing.assert_array_equal(host(x), x1)
    _close_ulp(host_bf16_bits(n2), bb.rmsnorm(x1.astype(np.float64), lr["w_post"]))
    gu = ds.linear(n2, ly.w_gu, workspaces=wsp, kind="t_gu")
    n2v = _vals(host_bf16_bits(n2))
    _close_sum(host_bf16_bits(gu), n2v @ lr["w_gu"].T, np.abs(n2v) @ np.abs(lr["w_gu"]).T, H)
    act = ds.silu_mul(gu)
    guv = _vals(host_bf16_bits(gu))
    _close_ulp(host_bf16_bits(act), bb.silu(guv[:, :I]) * guv[:, I:])
    d2 = ds.linear(act, ly.w_d, workspaces=wsp, kind="t_d")
    av = _vals(host_bf16_bits(act))
    _close_sum(host_bf16_bits(d2), av @ lr["w_d"].T, np.abs(av) @ np.abs(lr["w_d"]).T, I)
    x2 = (host(x) + _vals(host_bf16_bits(d2)).astype(np.float32)).astype(np.float32)
    h2 = ds.add_rmsnorm(x, d2, dev_bf16(wf), group=nr)
    keep = np.arange(B * nr) % nr != 0
    _close_ulp(host_bf16_bits(h2), bb.rmsnorm(x2.astype(np.float64)[keep], _vals(wf)))
    np.testing.assert_array_equal(host_bf16_bits(h2), h_bits)              # the composite's h


def test_backbone_two_layers_small_matches_oracle():
    _backbone_case(H=256, nq=2, nkv=1, I=512, L=2, V=1000, B=3, C=37, k=7, seed=400)


def test_backbone_one_layer_small_stagewise():
    _backbone_case(H=256, nq=2, nkv=1, I=512, L=1, V=1000, B=2, C=70, k=4, seed=450, stagewise=True)


def test_backbone_27b_layer_matches_oracle():
    g = syn.BACKBONE_GEOMETRY[5120]
    _backbone_case(H=5120, nq=g["nq"], nkv=g["nkv"], I=g["I"], L=1, V=4096, B=1, C=1024, k=7, seed=500,
                   stagewise=True)


def test_backbone_new_context_rows_in_the_block_gemm_equal_separate_calls():
    """backbone_block(ctx=...) takes the new context rows' keys and values out of the
    block's QKV GEMM; the caches and h equal those of backbone_context for the same rows
    followed by backbone_block (each GEMM output element is the same fp32 sum)."""
    H, nq, nkv, I, L, V, B, C, k, n = 256, 2, 1, 512, 2, 500, 2, 30, 4, 4
    layers, wf = syn.backbone_weights(H, nq, nkv, I, L, seed=600)
    lay_d = [_layer_dev(l) for l in layers]
    E = dev_bf16(syn.normal_bf16(601, (V, H), 0.5))
    ctx = syn.normal_bf16(602, (B, C, H))
    toks = dev(np.concatenate([np.array([[3], [9]]), np.full((B, k), V - 1)], axis=1).astype(np.int32))
    outs = []
    for fused in (False, True):
        kcs = [torch.zeros((B, C + k + 1, nkv, 128), dtype=torch.bfloat16, device="cuda") for _ in layers]
        vcs = [torch.zeros_like(t) for t in kcs]
        wsp = ds.Workspaces()
        if fused:
            ds.backbone_context(dev_bf16(ctx[:, :C - n].reshape(-1, H)), lay_d, kcs, vcs, 0, workspaces=wsp)
            h = ds.backbone_block(toks, E, lay_d, dev_bf16(wf), kcs, vcs, C, workspaces=wsp,
                                  ctx=dev_bf16(np.ascontiguousarray(ctx[:, C - n:]).reshape(-1, H)), ctx_pos0=C - n)
        else:
            ds.backbone_context(dev_bf16(ctx.reshape(-1, H)), lay_d, kcs, vcs, 0, workspaces=wsp)
            h = ds.backbone_block(toks, E, lay_d, dev_bf16(wf), kcs, vcs, C, workspaces=wsp)
        outs.append(([host_bf16_bits(t) for t in kcs + vcs], host_bf16_bits(h)))
    for a, b in zip(outs[0][0], outs[1][0]):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_backbone_27b_batch4_matches_oracle():
    """27B layer geometry at batch 4 (the QKV GEMM over 32 block rows, the attention
    over 4 x 8 key/value heads x 5 slices of a 264-key cache)."""
    g = syn.BACKBONE_GEOMETRY[5120]
    _backbone_case(H=5120, nq=g["nq"], nkv=g["nkv"], I=g["I"], L=1, V=4096, B=4, C=256, k=7, seed=520)


def test_backbone_flash_geometry_matches_oracle():
    g = syn.BACKBONE_GEOMETRY[2560]
    _backbone_case(H=2560, nq=g["nq"], nkv=g["nkv"], I=g["I"], L=2, V=2048, B=2, C=130, k=7, seed=540)


def test_fused_norm_and_rope_launches_equal_separate_calls():
    """dspark_block_context_rmsnorm and dspark_qk_norm_rope_block_context (the block rows
    and the new context rows in one launch) give the bits of the separate calls: the
    embedding-gather or residual-add norm of the block rows and the plain norm of the
    context rows; the block rows' q/k norm + rotary and the context rows' k one."""
    H, V, B, nr, n, nq, nkv, C = 256, 300, 2, 5, 3, 4, 2, 20
    E = dev_bf16(syn.normal_bf16(700, (V, H), 0.5))
    w = dev_bf16(syn.normal_bf16(701, (H,), 0.3))
    toks = dev(np.array([[1, 299, 5, 7, 9], [0, 2, 4, 6, 8]], dtype=np.int32)).reshape(-1)
    ctx = dev_bf16(syn.normal_bf16(702, (B * n, H)))
    delta = dev_bf16(syn.normal_bf16(703, (B * nr, H)))
    x1, n1 = ds.embed_rmsnorm(E, toks, w)
    c1 = ds.rmsnorm_bf16(ctx, w)
    x2 = torch.empty((B * nr, H), dtype=torch.float32, device="cuda")
    out2 = torch.empty((B * (nr + n), H), dtype=torch.bfloat16, device="cuda")
    ds.block_context_rmsnorm(x2, w, out2, ctx=ctx, table=E, tokens=toks)
    np.testing.assert_array_equal(host(x1), host(x2))
    np.testing.assert_array_equal(host_bf16_bits(n1), host_bf16_bits(out2[:B * nr]))
    np.testing.assert_array_equal(host_bf16_bits(c1), host_bf16_bits(out2[B * nr:]))
    x3, x4 = x1.clone(), x1.clone()
    n3 = ds.add_rmsnorm(x3, delta, w)
    out4 = torch.empty_like(out2)
    ds.block_context_rmsnorm(x4, w, out4, ctx=ctx, delta=delta)
    np.testing.assert_array_equal(host(x3), host(x4))
    np.testing.assert_array_equal(host_bf16_bits(n3), host_bf16_bits(out4[:B * nr]))
    np.testing.assert_array_equal(host_bf16_bits(c1), host_bf16_bits(out4[B * nr:]))

    width = (nq + 2 * nkv) * 128
    qkv = dev_bf16(syn.normal_bf16(704, (B * (nr + n), width)))
    wq = dev_bf16(syn.normal_bf16(705, (128,), 0.5))
    wk = dev_bf16(syn.normal_bf16(706, (128,), 0.5))
    caches = [torch.zeros((B, C + nr, nkv, 128), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    q1 = ds.qk_norm_rope(qkv[:B * nr], nq, nkv, wq, wk, 1e6, caches[0], caches[1], nr, C)
    ds.qk_norm_rope(qkv[B * nr:, nq * 128:], 0, nkv, None, wk, 1e6, caches[0], caches[1], n, C - n)
    q2 = ds.qk_norm_rope_block_context(qkv[:B * nr], nq, nkv, wq, wk, 1e6, caches[2], caches[3], nr, C,
                                       qkv[B * nr:, nq * 128:], n, C - n)
    np.testing.assert_array_equal(host_bf16_bits(q1), host_bf16_bits(q2))
    np.testing.assert_array_equal(host_bf16_bits(caches[0]), host_bf16_bits(caches[2]))
    np.testing.assert_array_equal(host_bf16_bits(caches[1]), host_bf16_bits(caches[3]))
    assert host_bf16_bits(caches[2])[:, C - n:C + nr].any()


def test_backbone_block_records_a_bad_token_and_clamps_it():
    """A block token outside [0, V) reaches the native block pass's status word
    (DSPARK_ERR_BAD_TOKEN) and is clamped like the separate embedding call clamps it:
    the block's output equals the pass over the clamped tokens."""
    H, nq, nkv, I, V, B, C, k = 256, 2, 1, 512, 300, 1, 20, 3
    layers, wf = syn.backbone_weights(H, nq, nkv, I, 1, seed=710)
    lay_d = [_layer_dev(l) for l in layers]
    E = dev_bf16(syn.normal_bf16(711, (V, H), 0.5))
    ctx = dev_bf16(syn.normal_bf16(712, (B * C, H)))
    outs = []
    for toks_np in ([[V + 5, V - 1, V - 1, V - 1]], [[V - 1, V - 1, V - 1, V - 1]]):
        kc = torch.zeros((B, C + k + 1, nkv, 128), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        wsp = ds.Workspaces()
        ds.backbone_context(ctx, lay_d, [kc], [vc], 0, workspaces=wsp)
        h = ds.backbone_block(dev(np.array(toks_np, np.int32)), E, lay_d, dev_bf16(wf), [kc], [vc], C,
                              workspaces=wsp)
        torch.cuda.synchronize()
        outs.append((host_bf16_bits(h), ds.workspace_status(wsp._bufs[("backbone", 0)])))
    assert outs[0][1] == -7 and outs[1][1] == 0
    np.testing.assert_array_equal(outs[0][0], outs[1][0])


def _block_by_calls(tokens, E, layers, wf, kcs, vcs, C, ctx, ctx_pos0, wsp):
    """The block pass composed from the separate calls (each GEMM fixing up its own tiles)."""
    B, nr = tokens.shape
    H = E.shape[1]
    Bb, nc = B * nr, ctx.shape[0]
    xin = torch.empty((Bb + nc, H), dtype=torch.bfloat16, device="cuda")
    x = torch.empty((Bb, H), dtype=torch.float32, device="cuda")
    d2 = None
    for li, ly in enumerate(layers):
        if li == 0:
            ds.block_context_rmsnorm(x, ly.w_in, xin, ctx=ctx, table=E, tokens=tokens.reshape(-1))
        else:
            ds.block_context_rmsnorm(x, ly.w_in, xin, ctx=ctx, delta=d2)
        qkv = ds.linear(xin, ly.w_qkv, workspaces=wsp, kind="q%d" % li)
        q = ds.qk_norm_rope_block_context(qkv[:Bb], ly.nq, ly.nkv, ly.w_qn, ly.w_kn, ly.theta, kcs[li], vcs[li], nr,
                                          C, qkv[Bb:, ly.nq * 128:], nc // B, ctx_pos0)
        o = ds.attention(q.view(B, nr, ly.nq, 128), kcs[li], vcs[li], C + nr, workspaces=wsp)
        d = ds.linear(o.view(Bb, ly.nq * 128), ly.w_o, workspaces=wsp, kind="o%d" % li)
        n2 = ds.add_rmsnorm(x, d, ly.w_post)
        gu = ds.linear(n2, ly.w_gu, workspaces=wsp, kind="g%d" % li)
        d2 = ds.linear(ds.silu_mul(gu), ly.w_d, workspaces=wsp, kind="d%d" % li)
    return ds.add_rmsnorm(x, d2, wf, group=nr)


@pytest.mark.parametrize("B,H,nq,nkv,I,L", [(36, 1024, 8, 2, 2048, 2), (16, 5120, 40, 8, 17408, 1)])
def test_backbone_block_pass_equals_the_separate_calls(B, H, nq, nkv, I, L):
    """The native block pass (projections' split tiles added by the reading kernels) gives
    the bits of the separate calls: at 36 requests (288 block rows: two activation-row
    tiles per output, the 2048-wide projections split over several CTAs) with two
    layers, and at the 27B layer geometry with 16 requests (240 rows in the QKV GEMM).
    Both with new context rows in the QKV GEMM."""
    k, V, C, n = 7, 512, 40, 3
    nr = k + 1
    layers, wf = syn.backbone_weights(H, nq, nkv, I, L, seed=720 + B)
    lay_d = [_layer_dev(l) for l in layers]
    E = dev_bf16(syn.normal_bf16(721, (V, H), 0.5))
    old = dev_bf16(syn.normal_bf16(722, (B * (C - n), H)))
    new = dev_bf16(syn.normal_bf16(723, (B * n, H)))
    toks = dev(np.concatenate([(np.arange(B)[:, None] * 37) % V, np.full((B, k), V - 1)], axis=1).astype(np.int32))
    outs = []
    for native in (True, False):
        kcs = [torch.zeros((B, C + nr, nkv, 128), dtype=torch.bfloat16, device="cuda") for _ in layers]
        vcs = [torch.zeros_like(t) for t in kcs]
        wsp = ds.Workspaces()
        ds.backbone_context(old, lay_d, kcs, vcs, 0, workspaces=wsp)
        if native:
            h = ds.backbone_block(toks, E, lay_d, dev_bf16(wf), kcs, vcs, C, workspaces=wsp, ctx=new, ctx_pos0=C - n)
        else:
            h = _block_by_calls(toks, E, lay_d, dev_bf16(wf), kcs, vcs, C, new, C - n, wsp)
        torch.cuda.synchronize()
        outs.append((host_bf16_bits(h), [host_bf16_bits(t) for t in kcs + vcs]))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    for a, b in zip(outs[0][1], outs[1][1]):
        np.testing.assert_array_equal(a, b)
    assert np.isfinite(syn.bf16_bits_to_f32(outs[0][0])).all()
