"""Pins of the CPU oracle against things other than itself: library routines,
hand-enumerated cases, closed forms and distributional identities.

No GPU needed.  Each test names what fixes the expected value.
"""
import ctypes
import ctypes.util
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn

# --------------------------------------------------------------------------- bf16


def test_bf16_rounding_matches_torch_cast():
    """bf16 round-to-nearest-even of the oracle == torch's fp32->bf16 cast (a library
    routine), on random values and on hand-picked ties."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 10.0,
        rng.standard_normal(500).astype(np.float32) * 1e-38,   # subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 3.0e38, -3.0e38, np.inf, -np.inf], np.float32),
        # exact ties: low 16 bits == 0x8000, even and odd kept lsb
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80FFFF, 0x3F807FFF],
                 dtype=np.uint32).view(np.float32),
    ])
    ours = oracle.f32_to_bf16(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = oracle.bf16_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16)
                                  .float().numpy())


# --------------------------------------------------------------------------- GEMMs


def test_fc_project_matches_numpy_float64_matmul():
    """fc = bf16( concat(taps) . W^T ): against numpy's float64 matmul of the explicitly
    concatenated taps (a library routine).  Non-square, distinct taps, so a dropped tap,
    a tap-order mistake or a transposed weight fails."""
    M, H, T = 3, 64, 5
    taps = [syn.normal_bf16(100 + j, (M, H)) for j in range(T)]
    fc_w = syn.normal_bf16(200, (H, T * H), (1.0 / (T * H)) ** 0.5)
    h, h32 = oracle.fc_project(taps, fc_w, return_f32=True)
    x = np.concatenate([syn.bf16_bits_to_f32(t) for t in taps], axis=1).astype(np.float64)
    w = syn.bf16_bits_to_f32(fc_w).astype(np.float64)
    ref32 = (x @ w.T).astype(np.float32)
    # both are the fp32 rounding of an fp64 sum; the sums differ only in order
    np.testing.assert_allclose(h32, ref32, rtol=2e-7, atol=1e-30)
    ref_h = syn.to_bf16_bits(ref32)
    same = h32 == ref32
    assert same.mean() > 0.95
    np.testing.assert_array_equal(h[same], ref_h[same])
    # taps in another order give another result
    h_perm = oracle.fc_project(taps[::-1], fc_w)
    assert (h_perm != h).mean() > 0.5


def test_lm_head_matches_numpy_float64_matmul():
    M, H, V = 4, 64, 37
    h = syn.normal_bf16(300, (M, H))
    lm = syn.normal_bf16(301, (V, H), (1.0 / H) ** 0.5)
    out = oracle.lm_head(h, lm)
    ref = (syn.bf16_bits_to_f32(h).astype(np.float64) @ syn.bf16_bits_to_f32(lm).astype(np.float64).T)
    np.testing.assert_allclose(out, ref.astype(np.float32), rtol=2e-7, atol=1e-30)
    assert out.shape == (M, V)


def test_gemm_integer_inputs_are_exact():
    """Small integers: every partial sum is exact, so the oracle must equal the exact
    integer product bit for bit."""
    M, H, V, T = 5, 128, 29, 5
    taps = [syn.integer_valued_bf16(400 + j, (M, H)) for j in range(T)]
    fc_w = syn.integer_valued_bf16(410, (H, T * H), -2, 3)
    x = np.concatenate([syn.bf16_bits_to_f32(t) for t in taps], axis=1).astype(np.int64)
    w = syn.bf16_bits_to_f32(fc_w).astype(np.int64)
    exact = x @ w.T
    h, h32 = oracle.fc_project(taps, fc_w, return_f32=True)
    np.testing.assert_array_equal(h32, exact.astype(np.float32))
    lm = syn.integer_valued_bf16(411, (V, H), -2, 3)
    hh = syn.integer_valued_bf16(412, (M, H))
    ex2 = syn.bf16_bits_to_f32(hh).astype(np.int64) @ syn.bf16_bits_to_f32(lm).astype(np.int64).T
    np.testing.assert_array_equal(oracle.lm_head(hh, lm), ex2.astype(np.float32))


# --------------------------------------------------------------------------- Markov chain


def _load_golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["markov_chain_v8.json", "markov_fma_order.json"])
def test_markov_chain_hand_enumerated(golden_dir, name):
    g = _load_golden(golden_dir, name)
    w1 = syn.to_bf16_bits(np.array(g["w1"], np.float32))
    w2 = syn.to_bf16_bits(np.array(g["w2"], np.float32))
    logits = np.array(g["logits"], np.float32)
    out = oracle.greedy_sample(logits, w1, w2, np.array(g["prev"], np.int32))
    np.testing.assert_array_equal(out["draft_tokens"], np.array(g["expect_draft_tokens"]))
    np.testing.assert_array_equal(out["z"], np.array(g["expect_z"], np.float32))
    if "expect_q_max" in g:
        np.testing.assert_array_equal(out["q_max"], np.array(g["expect_q_max"], np.float64))
    # q_sumexp: closed form from the enumerated z
    z = np.array(g["expect_z"], np.float64)
    ref_s = np.exp(z - z.max(axis=-1, keepdims=True)).sum(axis=-1)
    np.testing.assert_allclose(out["q_sumexp"], ref_s, rtol=1e-14)


def test_markov_lowrank_equals_full_bigram_table():
    """Invariant: the low-rank bias W2 . W1[prev] equals a lookup into the full V x V
    bigram table W1 W2^T built independently (exact integer matmul), and the chain feeds
    each position's biased argmax to the next."""
    B, k, V, r = 3, 5, 64, 4
    w1f = np.random.default_rng(1).integers(-3, 4, size=(V, r)).astype(np.float32)
    w2f = np.random.default_rng(2).integers(-3, 4, size=(V, r)).astype(np.float32)
    table = (w1f.astype(np.int64) @ w2f.astype(np.int64).T).astype(np.float64)  # [prev, v]
    logits = np.random.default_rng(3).integers(-20, 21, size=(B, k, V)).astype(np.float32)
    prev = np.array([0, 17, 63], np.int32)
    out = oracle.greedy_sample(logits, syn.to_bf16_bits(w1f), syn.to_bf16_bits(w2f), prev)
    for b in range(B):
        p = prev[b]
        for i in range(k):
            z = logits[b, i].astype(np.float64) + table[p]
            d = int(np.argmax(z))  # numpy argmax: first occurrence of the max
            assert out["draft_tokens"][b, i] == d
            np.testing.assert_array_equal(out["z"][b, i], z.astype(np.float32))
            p = d


def test_argmax_ties_lowest_index_and_signed_zero():
    logits = np.array([[[-1.0, -0.0, -2.0, 0.0, -0.5]]], np.float32)
    out = oracle.greedy_sample(logits, None, None, np.array([0], np.int32))
    assert out["draft_tokens"][0, 0] == 1
    logits = np.array([[[3.0, 7.0, 7.0, 1.0, 7.0]]], np.float32)
    out = oracle.greedy_sample(logits, None, None, np.array([0], np.int32))
    assert out["draft_tokens"][0, 0] == 1
    assert out["top2_gap"][0, 0] == 0.0


def test_greedy_sample_rejects_bad_prev_token():
    logits = np.zeros((1, 1, 4), np.float32)
    w = syn.to_bf16_bits(np.ones((4, 2), np.float32))
    with pytest.raises(oracle.OracleError):
        oracle.greedy_sample(logits, w, w, np.array([4], np.int32))


# --------------------------------------------------------------------------- confidence


def test_confidence_closed_form_and_truncation():
    """tau = 0.5: sigmoid(z) >= 0.5 <=> z >= 0.  Hand case: integer h and w."""
    B, k, H = 2, 3, 4
    w = syn.to_bf16_bits(np.array([1, -1, 2, 0], np.float32))
    h = syn.to_bf16_bits(np.array([
        [1, 1, 1, 1],    # b0 p0: 1-1+2 = 2   keep
        [0, 3, 1, 0],    # b0 p1: -3+2 = -1   stop -> len 1
        [5, 0, 0, 0],    # b0 p2: 5 (after the stop: still dropped)
        [0, 1, 0, 0],    # b1 p0: -1 stop -> len 0
        [1, 0, 0, 0],
        [1, 0, 0, 0],
    ], np.float32))
    drafts = np.arange(B * k, dtype=np.int32).reshape(B, k) + 10
    out = oracle.confidence(h, B, k, w, 0.0, 0.5, drafts)
    np.testing.assert_array_equal(out["zc"], [[2, -1, 5], [-1, 1, 1]])
    np.testing.assert_array_equal(out["draft_len"], [1, 0])
    np.testing.assert_array_equal(out["draft_tokens"], [[10, -1, -1], [-1, -1, -1]])
    np.testing.assert_allclose(out["conf"], 1.0 / (1.0 + np.exp(-out["zc"])), rtol=1e-15)
    # the bias term shifts every logit; tau != 0.5 uses logit(tau)
    out = oracle.confidence(h, B, k, w, 1.5, 0.5, drafts)
    np.testing.assert_array_equal(out["draft_len"], [3, 3])
    tau = 1.0 / (1.0 + math.exp(-1.75))   # logit(tau) = 1.75: only zc >= 1.75 passes
    out = oracle.confidence(h, B, k, w, 0.0, tau, drafts)
    np.testing.assert_array_equal(out["draft_len"], [1, 0])
    assert oracle.confidence(h, B, k, w, 0.0, 0.0, drafts)["draft_len"].tolist() == [3, 3]
    assert oracle.confidence(h, B, k, w, 0.0, 1.0, drafts)["draft_len"].tolist() == [0, 0]


# --------------------------------------------------------------------------- Philox


def _curand():
    for name in ("libcurand.so", "libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def test_philox_matches_curand_host_generator():
    """Philox4x32-10 (Salmon et al., SC'11) against cuRAND's host-side PHILOX4_32_10
    generator, a library routine.  That generator uses the 64-bit seed as the key (low
    word, high word) and emits 4-word block n from counter (n // 65536, 0, n % 65536, 0),
    so blocks past 65535 exercise counter word 0 and the others word 2."""
    cr = _curand()
    if cr is None:
        pytest.skip("libcurand not available")
    blocks = (0, 1, 777, 65535, 65536, 65537, 3 * 65536 + 5)
    n = 4 * (max(blocks) + 1)
    for seed in (0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF):
        gen = ctypes.c_void_p()
        assert cr.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
        try:
            assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            out = np.zeros(n, np.uint32)
            assert cr.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        finally:
            cr.curandDestroyGenerator(gen)
        key = (seed & 0xFFFFFFFF, seed >> 32)
        for blk in blocks:
            ctr = (blk // 65536, 0, blk % 65536, 0)
            assert oracle.philox4x32_10(ctr, key) == out[4 * blk:4 * blk + 4].tolist(), (seed, blk)


def test_philox_counter_words_all_matter_and_uniforms_exact():
    key = (0x1234, 0x5678)
    base = oracle.philox4x32_10((1, 2, 3, 4), key)
    for i in range(4):
        c = [1, 2, 3, 4]
        c[i] += 1
        assert oracle.philox4x32_10(c, key) != base
    ua, us = oracle.verify_uniforms(0xABCDEF0123456789, 5, 3, 11)
    w = oracle.philox4x32_10((5, 3, 11, 0), (0x23456789, 0xABCDEF01))
    assert ua == (w[0] >> 8) / 2.0 ** 24 and us == (w[1] >> 8) / 2.0 ** 24
    # uniformity of the accept words over many counters (chi-square, 16 bins)
    from scipy.stats import chisquare
    u = np.array([oracle.verify_uniforms(0, rq, 0, 0)[0] for rq in range(20000)])
    counts = np.histogram(u, bins=16, range=(0, 1))[0]
    assert chisquare(counts).pvalue > 1e-3


# --------------------------------------------------------------------------- verify


def _softmax64(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def test_greedy_verify_closed_forms():
    B, k, V = 4, 5, 50
    tgt = syn.uniform_logits(11, (B, k + 1, V), 2.0)
    t = tgt.argmax(axis=-1).astype(np.int32)   # numpy: lowest index on ties
    drafts = t[:, :k].copy()
    drafts[1, 2] = (drafts[1, 2] + 1) % V      # first mismatch at 2
    drafts[2, :] = (t[2, :k] + 1) % V          # all wrong
    dl = np.array([k, k, k, 3], np.int32)       # request 3: only 3 drafts
    out = oracle.verify(0, tgt, drafts, dl)
    np.testing.assert_array_equal(out["accepted_len"], [k, 2, 0, 3])
    np.testing.assert_array_equal(out["next_token"], [t[0, k], t[1, 2], t[2, 0], t[3, 3]])
    # ties in the target resolve to the lowest index
    tgt2 = np.zeros((1, 2, 6), np.float32)
    tgt2[0, 0, [2, 4]] = 1.0
    tgt2[0, 1, [1, 5]] = 3.0
    out = oracle.verify(0, tgt2, np.array([[2]], np.int32))
    assert out["accepted_len"][0] == 1 and out["next_token"][0] == 1
    out = oracle.verify(0, tgt2, np.array([[4]], np.int32))
    assert out["accepted_len"][0] == 0 and out["next_token"][0] == 2


def _chi2_pvalue(counts, probs):
    from scipy.stats import chisquare
    n = counts.sum()
    return chisquare(counts, probs * n).pvalue


def test_rejection_sampling_output_distribution_is_target():
    """The rejection-sampling identity: with x ~ q, accept w.p. min(1, p/q), else draw from
    norm(max(0, p - q)), the emitted token is distributed as p.  10^6 requests on V = 8,
    chi-square p-value > 1e-3; P(accept) = sum_v min(p, q) within 4 sigma."""
    N, V = 1_000_000, 8
    zl = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.0, 0.7, 0.1], np.float32)
    tl = np.array([0.3, 1.1, -0.2, 1.0, 0.5, -2.0, 0.0, 0.9], np.float32)
    p = _softmax64(tl)
    q = _softmax64(zl)
    x = np.random.default_rng(123).choice(V, size=N, p=q).astype(np.int32)
    target = np.broadcast_to(np.stack([tl, tl])[None], (N, 2, V)).copy()
    z = np.broadcast_to(zl[None, None], (N, 1, V)).copy()
    out = oracle.verify(1, target, x[:, None], None, z, seed=0xC0FFEE, step=3)
    acc = out["accepted_len"] == 1
    first = np.where(acc, x, out["next_token"])
    counts = np.bincount(first, minlength=V)
    assert _chi2_pvalue(counts, p) > 1e-3
    pa = np.minimum(p, q).sum()
    assert abs(acc.mean() - pa) < 4 * math.sqrt(pa * (1 - pa) / N)
    # the bonus token of fully accepted requests follows p of row 1 (= p here)
    assert _chi2_pvalue(np.bincount(out["next_token"][acc], minlength=V), p) > 1e-3


def test_rejection_sampling_one_hot_draft():
    """Deterministic (argmax) draft, q one-hot at d: accept w.p. p(d), otherwise draw from p
    with d removed; the emitted token is again distributed as p."""
    N, V = 400_000, 8
    tl = np.array([0.3, 1.1, -0.2, 1.0, 0.5, -2.0, 0.0, 0.9], np.float32)
    p = _softmax64(tl)
    d = 3
    target = np.broadcast_to(np.stack([tl, tl])[None], (N, 2, V)).copy()
    drafts = np.full((N, 1), d, np.int32)
    out = oracle.verify(1, target, drafts, None, None, seed=99, step=0)
    acc = out["accepted_len"] == 1
    assert abs(acc.mean() - p[d]) < 4 * math.sqrt(p[d] * (1 - p[d]) / N)
    first = np.where(acc, d, out["next_token"])
    assert _chi2_pvalue(np.bincount(first, minlength=V), p) > 1e-3
    assert not np.any(out["next_token"][~acc] == d)


def test_rejection_sampling_two_positions_joint():
    """k = 2 with independent rows: among requests that accept position 0, the pair
    (x_0, second emitted token) follows [min(p0,q0)/sum] x p1 (63-dof chi-square);
    acceptance of position 1 given position 0 is sum min(p1, q1)."""
    N, V = 1_000_000, 8
    t0 = np.array([0.3, 1.1, -0.2, 1.0, 0.5, -2.0, 0.0, 0.9], np.float32)
    t1 = np.array([-1.0, 0.0, 1.5, 0.2, 0.2, 0.8, -0.4, 0.0], np.float32)
    z0 = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.0, 0.7, 0.1], np.float32)
    z1 = np.array([0.0, 0.5, 1.0, -1.0, 0.3, 1.2, 0.0, -0.3], np.float32)
    p0, p1, q0, q1 = (_softmax64(a) for a in (t0, t1, z0, z1))
    rng = np.random.default_rng(5)
    x = np.stack([rng.choice(V, size=N, p=q0), rng.choice(V, size=N, p=q1)], axis=1).astype(np.int32)
    target = np.broadcast_to(np.stack([t0, t1, t1])[None], (N, 3, V)).copy()
    z = np.broadcast_to(np.stack([z0, z1])[None], (N, 2, V)).copy()
    out = oracle.verify(1, target, x, None, z, seed=7, step=1)
    a = out["accepted_len"]
    sel = a >= 1
    second = np.where(a[sel] == 2, x[sel, 1], out["next_token"][sel])
    m0 = np.minimum(p0, q0)
    joint = np.outer(m0 / m0.sum(), p1).reshape(-1)
    counts = np.bincount(x[sel, 0] * V + second, minlength=V * V)
    assert _chi2_pvalue(counts, joint) > 1e-3
    pa1 = np.minimum(p1, q1).sum()
    n1 = sel.sum()
    assert abs((a[sel] == 2).mean() - pa1) < 4 * math.sqrt(pa1 * (1 - pa1) / n1)


def test_verify_draft_len_zero_takes_bonus_from_row_zero():
    V = 16
    tgt = syn.uniform_logits(21, (2, 4, V), 1.0)
    drafts = np.full((2, 3), -1, np.int32)
    out = oracle.verify(0, tgt, drafts, np.array([0, 0], np.int32))
    np.testing.assert_array_equal(out["accepted_len"], [0, 0])
    np.testing.assert_array_equal(out["next_token"], tgt[:, 0].argmax(axis=-1))
    out = oracle.verify(1, tgt, drafts, np.array([0, 0], np.int32), None, seed=1)
    np.testing.assert_array_equal(out["accepted_len"], [0, 0])
    np.testing.assert_array_equal(out["sample_row"], [0, 0])


def _gumbel(seed, req, row, step, V):
    """Gumbel noise of the documented draw counters, from the Philox pinned above."""
    g = np.empty(V)
    for v in range(V):
        w = oracle.philox4x32_10((req, row, step, 1 + v // 4), (seed & 0xFFFFFFFF, seed >> 32))
        u = (2 * (w[v % 4] >> 9) + 1) / 2.0 ** 24
        g[v] = -math.log(-math.log(u))
    return g


def test_verify_draws_are_gumbel_argmax():
    """Draws: next = argmax_v log w_v + G_v with G from the documented Philox counters
    (numpy recomputation); accept iff u < p(d)/q(d) with q one-hot at the argmax draft."""
    V = 12
    tgt = syn.uniform_logits(31, (64, 2, V), 1.5)
    d = tgt[:, 0].argmax(axis=-1).astype(np.int32)[:, None]
    out = oracle.verify(0, tgt, d)
    assert np.all(out["accepted_len"] == 1)
    outp = oracle.verify(1, tgt, d, None, None, seed=42, step=9)
    for b in range(64):
        ua, _ = oracle.verify_uniforms(42, b, 0, 9)
        p0 = _softmax64(tgt[b, 0])
        if ua < p0[d[b, 0]]:
            assert outp["accepted_len"][b] == 1
            key = np.log(_softmax64(tgt[b, 1])) + _gumbel(42, b, 1, 9, V)
        else:
            assert outp["accepted_len"][b] == 0
            lw = np.log(p0)
            lw[d[b, 0]] = -np.inf
            key = lw + _gumbel(42, b, 0, 9, V)
        assert outp["next_token"][b] == int(np.argmax(key))


def test_gumbel_draw_distribution_large_vocab():
    """Bonus draws from p over V = 37 (several Philox blocks per row, a ragged last block):
    chi-square against p over 200k requests."""
    N, V = 200_000, 37
    tl = syn.uniform_logits(77, (V,), 1.0)
    p = _softmax64(tl)
    target = np.broadcast_to(np.stack([tl, tl])[None], (N, 2, V)).copy()
    drafts = np.full((N, 1), -1, np.int32)
    out = oracle.verify(1, target, drafts, np.zeros(N, np.int32), None, seed=3, step=4)
    assert np.all(out["accepted_len"] == 0) and np.all(out["sample_row"] == 0)
    assert _chi2_pvalue(np.bincount(out["next_token"], minlength=V), p) > 1e-3
    assert np.nanmin(out["sample_margin"]) > -1.0


# --------------------------------------------------------------------------- FP8 (E4M3)


def test_e4m3_codes_match_torch_float8_cast():
    """E4M3 rounding (ties to even) against torch's float8_e4m3fn cast (a library routine)
    over the whole finite range, every code's decode, and saturation beyond 448 (torch
    maps overflow to NaN; the oracle saturates, as cvt.satfinite does)."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.standard_normal(20000) * 1e-2,
                        rng.standard_normal(5000) * 3e-3,
                        # exact ties between neighbouring codes
                        (np.arange(1, 40) + 0.5) * 2.0 ** -9, 1.0 + (np.arange(8) + 0.5) / 8.0,
                        [0.0, -0.0, 448.0, -448.0, 2.0 ** -6, 2.0 ** -9]]).astype(np.float32)
    ours = oracle.f32_to_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inr = np.abs(x) <= 448
    np.testing.assert_array_equal(ours[inr], ref[inr])
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_to_f32(codes)
    tdec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(tdec))
    np.testing.assert_array_equal(dec[~np.isnan(dec)], tdec[~np.isnan(tdec)])
    assert oracle.f32_to_e4m3(np.array([464.0, 1e6, -5000.0], np.float32)).tolist() == [0x7E, 0x7E, 0xFE]


def test_fp8_row_quantisation_closed_form():
    """scale = amax / 448; the row maximum maps to code 0x7E (448); all-zero rows use
    scale 1; codes are the E4M3 rounding of x / scale."""
    x = np.array([[1.0, -2.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0], [3.0, 3.0, -3.0, 1e-3]], np.float32)
    codes, scales = oracle.quantize_fp8_rows(syn.to_bf16_bits(x))
    xb = syn.bf16_bits_to_f32(syn.to_bf16_bits(x))
    np.testing.assert_array_equal(scales, [np.float32(2.0) / np.float32(448.0), 1.0,
                                           np.float32(3.0) / np.float32(448.0)])
    assert codes[0, 1] == 0xFE and codes[2, 0] == 0x7E and codes[2, 2] == 0xFE
    np.testing.assert_array_equal(codes[1], 0)
    for r in range(3):
        np.testing.assert_array_equal(codes[r], oracle.f32_to_e4m3(xb[r] / scales[r]))


def test_fp8_gemm_matches_numpy_on_decoded_operands():
    """The FP8 GEMM is the fp64 dot product of the decoded codes times both scales:
    numpy float64 matmul of torch-decoded operands (library routines)."""
    M, N, K = 5, 33, 256
    a = np.random.default_rng(1).integers(0, 256, (M, K), dtype=np.uint8)
    w = np.random.default_rng(2).integers(0, 256, (N, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0
    w[(w & 0x7F) == 0x7F] = 0
    sa = np.random.default_rng(3).uniform(0.5, 2, M).astype(np.float32)
    sw = np.random.default_rng(4).uniform(0.5, 2, N).astype(np.float32)
    dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    ref = (dec(a) @ dec(w).T) * sa[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
    np.testing.assert_allclose(oracle.gemm_fp8(a, sa, w, sw), ref.astype(np.float32), rtol=2e-7, atol=1e-30)


def test_bf16_array_rounding_matches_torch():
    x = np.random.default_rng(9).standard_normal(5000).astype(np.float32) * 7
    np.testing.assert_array_equal(oracle.f32_to_bf16_array(x), syn.to_bf16_bits(x))


# ----------------------------------------------------------------------------- row statistics

def test_row_stats_matches_library_definitions():
    """max, first argmax and the fp64 sum of exp(x - max) of each row equal numpy's on
    rows with ties, -0/+0, -inf entries, an all -inf row and large values (no overflow:
    the max is subtracted before the exponential)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 257)).astype(np.float32)
    x[0, [5, 200]] = 9.0                       # tie -> index 5
    x[1, :] = -np.inf
    x[2, 10] = -0.0
    x[2, 11] = 0.0
    x[2, :10] = -5.0
    x[2, 12:] = -5.0                           # -0 == +0: the first of the two wins
    x[3, ::3] = -np.inf
    x[4] *= 1000.0                              # exp(x) alone would overflow
    x[5, 256] = 50.0                            # the max in the last entry
    got = oracle.row_stats(x)
    xd = x.astype(np.float64)
    for r in range(x.shape[0]):
        m = xd[r].max()
        assert got["max"][r] == m
        assert got["argmax"][r] == int(np.argmax(xd[r]))
        ref = 0.0 if m == -np.inf else float(np.exp(xd[r] - m).sum())
        assert got["sumexp"][r] == pytest.approx(ref, rel=1e-14, abs=0.0)
    assert got["argmax"][0] == 5 and got["argmax"][2] == 10 and got["argmax"][1] == 0
    assert got["sumexp"][1] == 0.0 and got["max"][1] == -np.inf


# ----------------------------------------------------------------------------- draw margins

def _gumbel32(seed, req, row, step, V):
    """The same noise evaluated in binary32 (numpy float32 logarithms)."""
    g = np.empty(V, np.float32)
    for v in range(V):
        w = oracle.philox4x32_10((req, row, step, 1 + v // 4), (seed & 0xFFFFFFFF, seed >> 32))
        u = np.float32((2 * (w[v % 4] >> 9) + 1) * 2.0 ** -24)
        g[v] = -np.log(-np.log(u))
    return g


def _float32_draw(t, z, row, seed, b, step, kind):
    """Binary32 evaluation of a draw's keys with numpy float32 (normalisers rounded to
    fp32; residual log(p - q) as (t - cp) + log1p(-exp((z - cq) - (t - cp))); noise
    -log(-log U)) -> the argmax."""
    V = t.shape[-1]
    tr = t[b, row]
    fin = tr[np.isfinite(tr)].astype(np.float64)
    cp = np.float32(fin.max() + math.log(np.exp(fin - fin.max()).sum()))
    g = _gumbel32(seed, b, row, step, V)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        if kind == "residual":
            zr = z[b, row]
            cq = np.float32(float(zr.max()) + math.log(float(np.exp(zr.astype(np.float64) - zr.max()).sum())))
            av = (tr - cp).astype(np.float32)
            bv = (zr - cq).astype(np.float32)
            kr = np.where(av > bv, av + np.log1p(-np.exp(bv - av)) + g, -np.inf)
        else:
            kr = tr + g
    return int(np.argmax(kr.astype(np.float32)))


def test_draw_margin_bounds_a_binary32_evaluation():
    """Where the oracle reports a positive draw margin, an independent binary32 evaluation
    of the draw keys picks the oracle's token.  Two families: random rows (residual draws
    after a rejection, and bonus draws), and bonus draws built so that the top two keys
    lie 1e-7 .. 1e-3 apart, which puts many margins just above zero; a margin formula
    that under-counted the binary32 error would let the two sides disagree there."""
    seed, step = 77, 5
    # family 1: random rows, residual draws (q = softmax of z, draft = argmax z)
    N, V = 400, 24
    rng = np.random.default_rng(9)
    t = (rng.standard_normal((N, 2, V)) * 0.05).astype(np.float32)
    z = (t[:, :1] + rng.standard_normal((N, 1, V)).astype(np.float32) * 0.05).astype(np.float32)
    d = z[:, 0].argmax(axis=-1).astype(np.int32)[:, None]
    out = oracle.verify(1, t, d, None, z, seed=seed, step=step)
    checked = 0
    for b in range(N):
        if out["sample_margin"][b] > 0:
            row = out["sample_row"][b]
            kind = "residual" if row == 0 else "bonus"
            assert _float32_draw(t, z, row, seed, b, step, kind) == out["next_token"][b]
            checked += 1
    assert checked > N // 2
    # family 2: built close pairs at the bonus row (the draft has p = 1, so it is accepted)
    deltas = np.logspace(-7, -3, 200)
    M, V2, a, c = len(deltas), 8, 1, 6
    tb = np.full((M, 2, V2), -np.inf, np.float32)
    tb[:, 0, 3] = 0.0                                   # p(3) = 1 at row 0
    for b, dl in enumerate(deltas):
        g = _gumbel(seed, b, 1, step, V2)
        tb[b, 1, a] = 0.0
        tb[b, 1, c] = np.float32(g[a] - g[c] + (dl if b % 2 else -dl))
    outb = oracle.verify(1, tb, np.full((M, 1), 3, np.int32), None, None, seed=seed, step=step)
    assert np.all(outb["accepted_len"] == 1) and np.all(outb["sample_row"] == 1)
    pos = 0
    for b in range(M):
        if outb["sample_margin"][b] > 0:
            assert _float32_draw(tb, None, 1, seed, b, step, "bonus") == outb["next_token"][b], b
            pos += 1
    neg = int((outb["sample_margin"] < 0).sum())
    assert pos > 50 and neg > 20                         # both sides of the bound exercised
    # the bound sits between 1e-6 and 1e-4 for keys of this size
    assert np.all(outb["sample_margin"][deltas > 1e-4] > 0)
    assert np.all(outb["sample_margin"][deltas < 1e-6] < 0)


def test_draw_margin_is_negative_on_a_built_near_tie():
    """Two candidates whose keys log p + G differ by about one fp32 ulp: the oracle must
    flag the draw (negative margin), since binary32 evaluations may order them either way."""
    seed, step, V = 5, 3, 8
    a, c = 2, 6                              # the two candidates; every other weight is zero
    g = _gumbel(seed, 0, 0, step, V)
    t = np.full((1, 2, V), -np.inf, np.float32)
    t[0, 0, a] = 0.0
    t[0, 0, c] = np.float32(g[a] - g[c])     # t_c + G_c = t_a + G_a up to fp32 rounding
    t[0, 1] = 0.0
    drafts = np.array([[0]], np.int32)       # p(0) = 0: rejected; residual = p without 0
    out = oracle.verify(1, t, drafts, None, None, seed=seed, step=step)
    assert out["accepted_len"][0] == 0 and out["sample_row"][0] == 0
    assert out["next_token"][0] in (a, c)
    assert out["sample_margin"][0] < 0


# ----------------------------------------------------------------------------- confidence with the Markov context

def test_confidence_markov_hand_case():
    """H = 2, r = 2, V = 4, integer weights, worked by hand.
    h rows (1, 2), (0, 1), (2, -1); conf_w = (1, -1 | 2, 1); markov_w1 rows
    (0, 0), (1, 0), (0, 1), (-1, 1); bonus token 1; drafts (2, 3, 0).
      position 0: h.w = 1 - 2 = -1, context 1 -> e = (1, 0) -> 2;  zc = 1
      position 1: h.w = 0 - 1 = -1, context 2 -> e = (0, 1) -> 1;  zc = 0
      position 2: h.w = 2 + 1 =  3, context 3 -> e = (-1, 1) -> -1; zc = 2
    Per position at tau = 0.5 (keep iff zc >= 0): all three kept.
    Cumulative at tau = 0.5: sigmoid(1) = 0.731 kept; 0.731 * sigmoid(0) = 0.366 < 0.5 ->
    draft_len 1.  At tau = 0.3: 0.366 kept; 0.366 * sigmoid(2) = 0.322 kept -> 3."""
    bf = syn.to_bf16_bits
    h = bf(np.array([[1, 2], [0, 1], [2, -1]], np.float32))
    w = bf(np.array([1, -1, 2, 1], np.float32))
    w1 = bf(np.array([[0, 0], [1, 0], [0, 1], [-1, 1]], np.float32))
    prev = np.array([1], np.int32)
    drafts = np.array([[2, 3, 0]], np.int32)
    per = oracle.confidence_markov(h, 1, 3, w, 0.0, 0.5, drafts, False, w1, prev)
    assert per["zc"][0].tolist() == [1.0, 0.0, 2.0]
    assert per["draft_len"][0] == 3 and per["draft_tokens"][0].tolist() == [2, 3, 0]
    cum = oracle.confidence_markov(h, 1, 3, w, 0.0, 0.5, drafts, True, w1, prev)
    assert cum["draft_len"][0] == 1 and cum["draft_tokens"][0].tolist() == [2, -1, -1]
    cum3 = oracle.confidence_markov(h, 1, 3, w, 0.0, 0.3, drafts, True, w1, prev)
    assert cum3["draft_len"][0] == 3
    # a bias shifts every position: b = -1.5 fails position 0 under either rule
    low = oracle.confidence_markov(h, 1, 3, w, -1.5, 0.5, drafts, False, w1, prev)
    assert low["draft_len"][0] == 0 and low["draft_tokens"][0].tolist() == [-1, -1, -1]


def test_confidence_markov_reduces_to_the_plain_head_and_product_rule():
    """Without markov_w1 the head is the plain one (same zc and draft lengths); the
    cumulative rule cuts where numpy's running product of sigmoids first drops below tau."""
    B, k, H = 6, 7, 64
    h = syn.normal_bf16(81, (B * k, H))
    w = syn.normal_bf16(82, (H,), (4.0 / H) ** 0.5)
    drafts = np.tile(np.arange(k, dtype=np.int32), (B, 1))
    plain = oracle.confidence(h, B, k, w, 0.1, 0.5, drafts)
    mk = oracle.confidence_markov(h, B, k, w, 0.1, 0.5, drafts, False)
    np.testing.assert_array_equal(mk["zc"], plain["zc"])
    np.testing.assert_array_equal(mk["draft_len"], plain["draft_len"])
    for tau in (0.05, 0.2, 0.5, 0.8):
        cum = oracle.confidence_markov(h, B, k, w, 0.1, tau, drafts, True)
        prod = np.cumprod(1.0 / (1.0 + np.exp(-mk["zc"])), axis=1)
        want = np.array([int(np.argmax(row < tau)) if (row < tau).any() else k for row in prod])
        np.testing.assert_array_equal(cum["draft_len"], want)
    assert (oracle.confidence_markov(h, B, k, w, 0.1, 0.0, drafts, True)["draft_len"] == k).all()
    assert (oracle.confidence_markov(h, B, k, w, 0.1, 1.0, drafts, True)["draft_len"] == 0).all()
