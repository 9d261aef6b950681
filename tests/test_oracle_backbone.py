"""Pins of the drafter-backbone oracle (oracle/backbone.py) to closed forms and
invariants that a dropped term, a wrong sign, a wrong head mapping or a misplaced
slice would break."""
import numpy as np
import pytest

from oracle import backbone as bb


def _layer(rng, H, nq, nkv, hd, I, zero_out=False):
    def w(*shape, std=0.05):
        return bb.bf16_round(rng.normal(0.0, std, shape))
    L = {"nq": nq, "nkv": nkv, "hd": hd,
         "w_in": w(H, std=1.0) + 1.0, "w_post": w(H, std=1.0) + 1.0,
         "w_qn": w(hd, std=0.2) + 1.0, "w_kn": w(hd, std=0.2) + 1.0,
         "w_qkv": w((nq + 2 * nkv) * hd, H), "w_o": w(H, nq * hd),
         "w_gu": w(2 * I, H), "w_d": w(H, I)}
    if zero_out:
        L["w_o"] = np.zeros_like(L["w_o"])
        L["w_d"] = np.zeros_like(L["w_d"])
    return L


def test_rmsnorm_closed_forms():
    w = np.array([1.0, 2.0, -0.5, 3.0])
    c = 0.75
    got = bb.rmsnorm(np.full(4, c), w)
    np.testing.assert_allclose(got, c / np.sqrt(c * c + bb.EPS) * w, rtol=1e-15)
    x = np.array([1.0, -1.0, 1.0, -1.0])             # mean square exactly 1
    np.testing.assert_allclose(bb.rmsnorm(x, w), x * w / np.sqrt(1.0 + bb.EPS), rtol=1e-15)
    big = np.array([3e3, -4e3, 1e3, 2e3])             # scale invariant while eps is negligible
    np.testing.assert_allclose(bb.rmsnorm(big, w), bb.rmsnorm(big * 10.0, w), rtol=1e-12)


def test_rope_closed_forms_and_relative_positions():
    # hd = 2: one pair at frequency theta^0 = 1 -> a rotation by pos radians
    x = np.array([[[1.0, 0.0]]])
    for p in (0, 1, 5):
        np.testing.assert_allclose(bb.rope(x, np.array([p]))[0, 0], [np.cos(p), np.sin(p)], atol=1e-15)
    rng = np.random.default_rng(3)
    q = rng.normal(size=(1, 3, 128))
    k = rng.normal(size=(1, 3, 128))
    np.testing.assert_allclose(bb.rope(q, np.array([0])), q, rtol=0, atol=0)    # position 0
    # the pair (d, d + 64) keeps its norm
    r = bb.rope(q, np.array([37]))
    np.testing.assert_allclose(r[..., :64] ** 2 + r[..., 64:] ** 2, q[..., :64] ** 2 + q[..., 64:] ** 2,
                               rtol=1e-12)
    # q . k depends on the position difference only
    d1 = np.sum(bb.rope(q, np.array([10])) * bb.rope(k, np.array([3])), axis=-1)
    d2 = np.sum(bb.rope(q, np.array([1010])) * bb.rope(k, np.array([1003])), axis=-1)
    np.testing.assert_allclose(d1, d2, rtol=1e-9)
    # the second half rotates forward: at a quarter turn of frequency 1, x2' = x1
    x = np.zeros((1, 1, 4)); x[0, 0, 0] = 1.0
    y = bb.rope(x, np.array([np.pi / 2]))
    np.testing.assert_allclose(y[0, 0], [0.0, 0.0, 1.0, 0.0], atol=1e-15)


def test_silu_closed_forms():
    np.testing.assert_allclose(bb.silu(np.array([0.0, 1.0, 40.0, -40.0])),
                               [0.0, 1.0 / (1.0 + np.exp(-1.0)), 40.0, -40.0 * np.exp(-40.0)],
                               rtol=1e-12, atol=1e-30)


def test_attention_equal_keys_dominant_key_and_head_groups():
    rng = np.random.default_rng(5)
    rows, nq, nkv, hd, nk = 3, 4, 2, 8, 6
    q = rng.normal(size=(rows, nq, hd))
    V = rng.normal(size=(nk, nkv, hd))
    # equal keys: uniform weights -> the mean of the values
    K = np.repeat(rng.normal(size=(1, nkv, hd)), nk, axis=0)
    out = bb.attention(q, K, V)
    for j in range(nq):
        np.testing.assert_allclose(out[:, j], np.broadcast_to(V[:, j // 2].mean(axis=0), (rows, hd)),
                                   rtol=1e-12)
    # values all equal: the weights sum to one whatever the keys
    K = rng.normal(size=(nk, nkv, hd))
    Vc = np.broadcast_to(rng.normal(size=(1, nkv, hd)), (nk, nkv, hd))
    np.testing.assert_allclose(bb.attention(q, K, Vc), np.broadcast_to(Vc[0][[0, 0, 1, 1]], (rows, nq, hd)),
                               rtol=1e-12)
    # one key aligned with the queries and large: its value wins
    K = np.zeros((nk, nkv, hd)); K[4] = 1e3
    qq = np.ones((rows, nq, hd))
    out = bb.attention(qq, K, V)
    for j in range(nq):
        np.testing.assert_allclose(out[:, j], np.broadcast_to(V[4, j // 2], (rows, hd)), rtol=1e-12)
    # head groups: query head j reads kv head j // (nq / nkv), as one-head attention does
    K = rng.normal(size=(nk, nkv, hd))
    out = bb.attention(q, K, V)
    for j in range(nq):
        s = q[:, j] @ K[:, j // 2].T / np.sqrt(hd)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref = (p / p.sum(axis=1, keepdims=True)) @ V[:, j // 2]
        np.testing.assert_allclose(out[:, j], ref, rtol=1e-12)


def test_layer_with_zero_output_projections_is_the_identity():
    rng = np.random.default_rng(7)
    H, nq, nkv, hd, I, C = 256, 2, 1, 128, 64, 5
    L = _layer(rng, H, nq, nkv, hd, I, zero_out=True)
    x = bb.bf16_round(rng.normal(size=(4, H)))
    Kc, Vc = bb.context_kv(bb.bf16_round(rng.normal(size=(C, H))), L, np.arange(C))
    y, _, _ = bb.decoder_layer(x, L, Kc, Vc, C)
    np.testing.assert_array_equal(y, x)


def test_block_keys_match_context_keys_of_the_same_rows():
    """The block's keys and values (decoder_layer) and the context path (context_kv)
    slice the same rows of [Wq; Wk; Wv] and rotate at the same positions."""
    rng = np.random.default_rng(11)
    H, nq, nkv, hd, I = 256, 2, 1, 128, 64
    L = _layer(rng, H, nq, nkv, hd, I)
    rows = bb.bf16_round(rng.normal(size=(3, H)))
    C = 7
    _, k_blk, v_blk = bb.decoder_layer(rows, L, np.zeros((0, nkv, hd)), np.zeros((0, nkv, hd)), C)
    K, Vv = bb.context_kv(rows, L, C + np.arange(3))
    np.testing.assert_array_equal(k_blk, K)
    np.testing.assert_array_equal(v_blk, Vv)


def test_backbone_with_zero_output_projections_normalises_the_mask_embedding():
    rng = np.random.default_rng(13)
    H, nq, nkv, hd, I, V, C, k = 256, 2, 1, 128, 64, 50, 6, 4
    layers = [_layer(rng, H, nq, nkv, hd, I, zero_out=True) for _ in range(2)]
    E = bb.bf16_round(rng.normal(size=(V, H)))
    wf = bb.bf16_round(rng.normal(size=H))
    ctx = bb.bf16_round(rng.normal(size=(C, H)))
    toks = np.array([7] + [V - 1] * k)
    h = bb.backbone(toks, ctx, layers, wf, E)
    ref = bb.bf16_round(bb.rmsnorm(E[V - 1], wf))
    np.testing.assert_array_equal(h, np.broadcast_to(ref, (k, H)))


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 1 and 1 + 2^-7: ties to the even 1
    np.testing.assert_array_equal(bb.bf16_round(np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8])),
                                  [1.0, 1.0 + 2.0 ** -6])
