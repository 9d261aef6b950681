"""GPU path (through the C ABI) against the CPU oracle, element by element.

Tolerances (from the arithmetic):
  * LM head / fc accumulate in fp32 on the tensor cores, the oracle in fp64:
    fp32 logits within rtol 2e-3 / atol 2e-3; the bf16 fc output within one bf16
    ulp plus the recursive-summation bound K * 2^-24 * sum|a w| (near-zero sums can
    differ by a few ulps of a tiny value), and off by more than one ulp on under 1%.
  * Markov chain on identical fp32 logits: the bias is a fixed sequential fp32 fma
    chain on both sides, so z and the draft tokens are bit-exact; the softmax sum of
    q (fp32 partial sums vs fp64) within rtol 1e-5.
  * Verify on identical inputs: greedy decisions bit-exact; probabilistic decisions
    bit-exact except where the oracle's |u - p/q| < 1e-5 or its Gumbel-max draw has a
    gap to the runner-up below its binary32 error bound (counted, then excluded).
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import bf16_ulp_diff, dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu

LOGIT_RTOL = 2e-3
LOGIT_ATOL = 2e-3
DECISION_EPS = 1e-5


def _assert_logits_close(gpu, ref):
    err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    bound = LOGIT_ATOL + LOGIT_RTOL * np.abs(ref.astype(np.float64))
    assert np.all(err <= bound), "max err %.3e" % err.max()
    return float(err.max())


def _assert_fc_close(got_bits, ref_bits, taps, fc_w):
    """h is a bf16 rounding of an fp32 sum of K = T*H products.  Any fp32 summation
    order is within K * 2^-24 * sum|a_k w_k| of the exact sum (recursive-summation bound),
    and the final bf16 rounding of either side adds at most one bf16 ulp."""
    x = np.concatenate([syn.bf16_bits_to_f32(t) for t in taps], axis=1).astype(np.float64)
    w = syn.bf16_bits_to_f32(fc_w).astype(np.float64)
    K = x.shape[1]
    mag = np.abs(x) @ np.abs(w).T
    got = syn.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = syn.bf16_bits_to_f32(ref_bits).astype(np.float64)
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    bound = ulp + K * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound), "max excess %.3e" % (np.abs(got - ref) - bound).max()
    d = bf16_ulp_diff(got_bits, ref_bits)
    assert (d > 1).mean() < 0.01 and (d > 0).mean() < 0.05


# ----------------------------------------------------------------------------- GEMMs

@pytest.mark.parametrize("M,H,V", [(1, 256, 4096), (7, 256, 4096), (33, 512, 1000),
                                   (112, 256, 4097), (300, 128, 777), (7, 1024, 20000)])
def test_lm_head_matches_oracle(M, H, V):
    h = syn.normal_bf16(10 + M, (M, H))
    w = syn.normal_bf16(20 + V, (V, H), (1.0 / H) ** 0.5)
    ref = oracle.lm_head(h, w)
    got = host(ds.lm_head(dev_bf16(h), dev_bf16(w)))
    torch.cuda.synchronize()
    _assert_logits_close(got, ref)


def test_lm_head_integer_inputs_bit_exact_and_deterministic():
    M, H, V = 21, 512, 3000
    h = syn.integer_valued_bf16(5, (M, H))
    w = syn.integer_valued_bf16(6, (V, H), -2, 3)
    ref = oracle.lm_head(h, w)
    hd, wd = dev_bf16(h), dev_bf16(w)
    a = host(ds.lm_head(hd, wd))
    b = host(ds.lm_head(hd, wd))
    np.testing.assert_array_equal(a, ref)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("M,H,T", [(1, 256, 5), (7, 256, 5), (28, 512, 5), (130, 128, 3),
                                   (7, 1024, 5), (513, 256, 5)])
def test_fc_project_matches_oracle(M, H, T):
    taps = [syn.normal_bf16(100 * M + j, (M, H)) for j in range(T)]
    fc_w = syn.normal_bf16(7 + H, (H, T * H), (1.0 / (T * H)) ** 0.5)
    ref = oracle.fc_project(taps, fc_w)
    got = host_bf16_bits(ds.fc_project([dev_bf16(t) for t in taps], dev_bf16(fc_w)))
    _assert_fc_close(got, ref, taps, fc_w)


def test_fc_project_strided_taps_and_integer_exact():
    """Taps as column slices of one wider buffer (row stride > H); integer inputs make
    every order of summation exact, so the result is bit-exact."""
    M, H, T = 9, 256, 5
    full = syn.integer_valued_bf16(8, (M, T * H + 64))
    taps_host = [np.ascontiguousarray(full[:, j * H:(j + 1) * H]) for j in range(T)]
    fc_w = syn.integer_valued_bf16(9, (H, T * H), -1, 2)
    ref = oracle.fc_project(taps_host, fc_w)
    fd = dev_bf16(full)
    taps = [fd[:, j * H:(j + 1) * H] for j in range(T)]
    got = host_bf16_bits(ds.fc_project(taps, dev_bf16(fc_w)))
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------------------- Markov chain

@pytest.mark.parametrize("M,H,T,V", [(7, 256, 5, 4096), (28, 512, 5, 20000), (130, 128, 3, 3001),
                                     (300, 256, 2, 1000), (1, 64, 1, 7)])
def test_fc_lm_head_one_launch_matches_oracle(M, H, T, V):
    """fc and LM head in one cooperative launch: h within the fc bound of the oracle,
    logits within the logit tolerance of the oracle's LM head on the GPU's h."""
    taps = [syn.normal_bf16(700 + 10 * j + M, (M, H)) for j in range(T)]
    fc_w = syn.normal_bf16(800 + H, (H, T * H), (1.0 / (T * H)) ** 0.5)
    lm_w = syn.normal_bf16(900 + V, (V, H), (1.0 / H) ** 0.5)
    h, logits = ds.fc_lm_head([dev_bf16(t) for t in taps], dev_bf16(fc_w), dev_bf16(lm_w))
    torch.cuda.synchronize()
    hb = host_bf16_bits(h)
    _assert_fc_close(hb, oracle.fc_project(taps, fc_w), taps, fc_w)
    _assert_logits_close(host(logits), oracle.lm_head(hb, lm_w))


def test_fc_lm_head_one_launch_equals_two_calls_and_repeats():
    """With one CTA per SM in both forms the single launch gives the two calls' bits,
    and repeated launches (counter reset by the last CTA) give the same bits."""
    M, H, T, V = 7, 1024, 5, 40000
    taps = [dev_bf16(syn.normal_bf16(710 + j, (M, H))) for j in range(T)]
    fc_w = dev_bf16(syn.normal_bf16(811, (H, T * H), (1.0 / (T * H)) ** 0.5))
    lm_w = dev_bf16(syn.normal_bf16(912, (V, H), (1.0 / H) ** 0.5))
    h2 = ds.fc_project(taps, fc_w)
    l2 = ds.lm_head(h2, lm_w)
    wsp = ds.Workspaces()
    for _ in range(3):
        h1, l1 = ds.fc_lm_head(taps, fc_w, lm_w, workspaces=wsp)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host_bf16_bits(h1), host_bf16_bits(h2))
        np.testing.assert_array_equal(host(l1), host(l2))


@pytest.mark.parametrize("B,k,V,r", [(1, 7, 4096, 16), (3, 4, 5001, 16), (16, 7, 20000, 64),
                                     (9, 2, 513, 128), (2, 1, 1, 8), (1, 7, 40000, 128),
                                     (12, 5, 30011, 128)])
def test_greedy_sample_bit_exact(B, k, V, r):
    logits = syn.uniform_logits(31 + V, (B, k, V), 1.5)
    w1 = syn.normal_bf16(32, (V, r))
    w2 = syn.normal_bf16(33, (V, r), (1.0 / r) ** 0.5)
    prev = (np.arange(B, dtype=np.int64) * 7919 % V).astype(np.int32)
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    lg = dev(logits)
    d, qs = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev))
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
    np.testing.assert_array_equal(host(lg), ref["z"])
    q = host(qs)
    np.testing.assert_array_equal(q[..., 0], ref["q_max"].astype(np.float32))
    np.testing.assert_allclose(q[..., 1], ref["q_sumexp"], rtol=1e-5)


# (13, 7, 20011, 64): a second 8-request group of 5 (an odd request pair, staged logits)
@pytest.mark.parametrize("B,k,V,r", [(1, 7, 4096, 16), (3, 4, 5001, 16), (16, 7, 20000, 64),
                                     (9, 16, 3001, 32), (1, 7, 20000, 0), (20, 3, 20000, 128),
                                     (13, 7, 20011, 64)])
def test_greedy_sample_without_q_stats_bit_exact(B, k, V, r):
    """Without a q_stats buffer the chain reduces only the argmax keys (another kernel
    variant): z and the draft tokens stay bit-exact, and draft_len is not touched."""
    logits = syn.uniform_logits(41 + V, (B, k, V), 1.5)
    if r:
        w1 = syn.normal_bf16(42, (V, r))
        w2 = syn.normal_bf16(43, (V, r), (1.0 / r) ** 0.5)
    else:
        w1 = w2 = None
    prev = (np.arange(B, dtype=np.int64) * 7919 % V).astype(np.int32)
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    lg = dev(logits)
    d, qs = ds.greedy_sample(lg, dev_bf16(w1) if r else None, dev_bf16(w2) if r else None,
                             dev(prev), want_q_stats=False)
    assert qs is None
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
    np.testing.assert_array_equal(host(lg), ref["z"])


# Batches above 8 requests (r <= 64) run the two-halves chain: request groups of 8
# alternate between two halves of the CTA on the FMA pipe.  Cases: a group slot left
# empty in one half (24, 40 requests), a partial group with an odd request pair (17,
# 33), V = 38913, where the last two of 152 CTAs (260-row slices) own no rows, and
# r = 128 (markov_w2 read through L2 instead of shared memory).
@pytest.mark.parametrize("B,k,V,r,stats", [(17, 3, 38913, 16, True), (24, 4, 20000, 64, False),
                                           (40, 3, 38913, 32, False), (33, 2, 4099, 64, True),
                                           (1, 3, 38913, 16, True), (16, 2, 38913, 64, False),
                                           (24, 3, 20000, 128, True), (17, 2, 38913, 128, False)])
def test_greedy_sample_two_halves_kernel(B, k, V, r, stats, monkeypatch):
    logits = syn.uniform_logits(51 + V + B, (B, k, V), 1.5)
    w1 = syn.normal_bf16(52, (V, r))
    w2 = syn.normal_bf16(53, (V, r), (1.0 / r) ** 0.5)
    prev = (np.arange(B, dtype=np.int64) * 7919 % V).astype(np.int32)
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("DSPARK_CHAIN_SPLIT", flag)
        lg = dev(logits)
        d, qs = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev), want_q_stats=stats)
        outs.append((host(d), host(lg), None if qs is None else host(qs)))
    for d, z, q in outs:
        np.testing.assert_array_equal(d, ref["draft_tokens"])
        np.testing.assert_array_equal(z, ref["z"])
        if stats:
            np.testing.assert_array_equal(q[..., 0], ref["q_max"].astype(np.float32))
            np.testing.assert_allclose(q[..., 1], ref["q_sumexp"], rtol=1e-5)
    if stats:
        np.testing.assert_array_equal(outs[0][2], outs[1][2])


def test_greedy_sample_per_position_kernels_agree(monkeypatch):
    """The per-position kernels (used when a cooperative launch is not possible) give
    the same bits as the persistent kernel and the oracle."""
    B, k, V, r = 5, 7, 30000, 64
    logits = syn.uniform_logits(35, (B, k, V), 1.5)
    w1 = syn.normal_bf16(36, (V, r))
    w2 = syn.normal_bf16(37, (V, r), (1.0 / r) ** 0.5)
    prev = np.array([0, 1, 29999, 12345, 777], np.int32)
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    outs = []
    for flag in ("0", "1"):
        monkeypatch.setenv("DSPARK_CHAIN_PER_POSITION", flag)
        lg = dev(logits)
        d, qs = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev))
        outs.append((host(d), host(lg), host(qs)))
    for d, z, q in outs:
        np.testing.assert_array_equal(d, ref["draft_tokens"])
        np.testing.assert_array_equal(z, ref["z"])
        np.testing.assert_allclose(q[..., 1], ref["q_sumexp"], rtol=1e-5)


def test_greedy_sample_hand_enumerated_golden(golden_dir):
    import json, os
    with open(os.path.join(golden_dir, "markov_chain_v8.json")) as f:
        g = json.load(f)
    w1 = syn.to_bf16_bits(np.array(g["w1"], np.float32))
    w2 = syn.to_bf16_bits(np.array(g["w2"], np.float32))
    # r = 2 is below the kernel's rank granularity of 8: pad with zero columns, which
    # leaves every fma chain unchanged (adding +0 * e keeps the sum bit-identical).
    pad = lambda a: np.concatenate([a, np.zeros((a.shape[0], 6), np.uint16)], axis=1)
    lg = dev(np.array(g["logits"], np.float32))
    d, qs = ds.greedy_sample(lg, dev_bf16(pad(w1)), dev_bf16(pad(w2)), dev(np.array(g["prev"], np.int32)))
    np.testing.assert_array_equal(host(d), np.array(g["expect_draft_tokens"]))
    np.testing.assert_array_equal(host(lg), np.array(g["expect_z"], np.float32))


def test_greedy_sample_no_bias_ties_and_signed_zero():
    x = np.full((2, 1, 4100), -5.0, np.float32)
    x[0, 0, [17, 2000, 4099]] = 3.0          # ties -> 17
    x[1, 0, 5] = -0.0
    x[1, 0, 9] = 0.0
    x[1, 0, 4000] = -0.0                     # -0 == +0 -> 5
    lg = dev(x)
    d, _ = ds.greedy_sample(lg, None, None, dev(np.zeros(2, np.int32)))
    assert host(d).tolist() == [[17], [5]]


# ----------------------------------------------------------------------------- verify

def _verify_inputs(B, k, V, seed):
    z = syn.uniform_logits(seed, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    noise = syn.uniform_logits(seed + 1, (B, k + 1, V), 1.0) * np.linspace(0.5, 3.0, k + 1)[None, :, None].astype(np.float32)
    target = np.concatenate([z, z[:, -1:]], axis=1) + noise
    return z, drafts, target.astype(np.float32)


# the last two cases: many requests, rows of several 16384-entry slices with a ragged tail
@pytest.mark.parametrize("B,k,V", [(1, 7, 4096), (5, 3, 4097), (16, 7, 9000), (4, 16, 301),
                                   (64, 7, 50000), (96, 7, 30001)])
def test_verify_greedy_bit_exact(B, k, V):
    z, drafts, target = _verify_inputs(B, k, V, 41 + V)
    # make some requests accept a long prefix: copy the target argmax into the drafts
    t = target.argmax(axis=-1).astype(np.int32)
    drafts[::2, : k // 2] = t[::2, : k // 2]
    dlen = np.array([(b * 3) % (k + 1) for b in range(B)], np.int32)
    ref = oracle.verify(0, target, drafts, dlen)
    a, n = ds.verify(0, dev(target), dev(drafts), dev(dlen))
    np.testing.assert_array_equal(host(a), ref["accepted_len"])
    np.testing.assert_array_equal(host(n), ref["next_token"])


def _excluded(ref, B):
    """Requests whose outcome floating point may legitimately decide differently: an
    accept test with |u - p/q| < 1e-5, or a Gumbel-max draw whose gap to the runner-up
    is within the oracle's binary32 error bound (negative sample margin)."""
    am = ref["accept_margin"]
    sm = ref["sample_margin"]
    ex = np.zeros(B, bool)
    with np.errstate(invalid="ignore"):
        ex |= np.any(np.nan_to_num(am, nan=1.0) < DECISION_EPS, axis=1)
        ex |= np.nan_to_num(sm, nan=1.0) < 0.0
    return ex


@pytest.mark.parametrize("with_q_stats", [False, True])
# (64, 7, 50001) and (48, 7, 40000): many requests, rows of several slices, ragged tails
@pytest.mark.parametrize("B,k,V", [(1, 7, 4096), (6, 5, 4099), (16, 7, 20000), (64, 2, 128),
                                   (64, 7, 50001), (48, 7, 40000)])
def test_verify_probabilistic_bit_exact(B, k, V, with_q_stats):
    z, drafts, target = _verify_inputs(B, k, V, 51 + V + B)
    t = target.argmax(axis=-1).astype(np.int32)
    drafts[1::3, :] = t[1::3, :k]
    ref = oracle.verify(1, target, drafts, None, z, seed=0xDEADBEEF, step=17)
    qs = None
    if with_q_stats:
        zz = z.astype(np.float64)
        m = zz.max(axis=-1)
        s = np.exp(zz - m[..., None]).sum(axis=-1)
        qs = dev(np.stack([m, s], axis=-1).astype(np.float32))
    a, n = ds.verify(1, dev(target), dev(drafts), None, dev(z), qs, seed=0xDEADBEEF, step=17)
    ex = _excluded(ref, B)
    assert ex.mean() < 0.05
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])


def test_verify_with_masked_vocabulary_bit_exact():
    """A vocabulary mask (about 30% of the entries -inf in the target and draft-logit
    rows, as a sampler's token mask leaves them) over rows of two whole 16384-entry
    slices and a ragged one: greedy and probabilistic decisions match the oracle."""
    B, k, V = 4, 5, 40000
    z, drafts, target = _verify_inputs(B, k, V, 97)
    mask = np.random.default_rng(98).random(V) < 0.3
    z[:, :, mask] = -np.inf
    target[:, :, mask] = -np.inf
    drafts = z.argmax(axis=-1).astype(np.int32)
    t = target.argmax(axis=-1).astype(np.int32)
    drafts[::2, :2] = t[::2, :2]
    ref0 = oracle.verify(0, target, drafts, None)
    a, n = ds.verify(0, dev(target), dev(drafts), None)
    np.testing.assert_array_equal(host(a), ref0["accepted_len"])
    np.testing.assert_array_equal(host(n), ref0["next_token"])
    ref = oracle.verify(1, target, drafts, None, z, seed=0xABCDEF, step=9)
    a, n = ds.verify(1, dev(target), dev(drafts), None, dev(z), None, seed=0xABCDEF, step=9)
    ex = _excluded(ref, B)
    assert ex.mean() < 0.5
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])
    assert not mask[host(n)[~ex]].any()  # no draw lands on a masked token


def test_verify_probabilistic_one_hot_and_request_ids():
    B, k, V = 12, 4, 3000
    z, drafts, target = _verify_inputs(B, k, V, 77)
    rid = (np.arange(B, dtype=np.uint32) * 1000003 + 5).astype(np.uint32)
    dlen = np.array([k, 0, 1, 2, 3, 4] * 2, np.int32)
    ref = oracle.verify(1, target, drafts, dlen, None, seed=5, request_id=rid, step=2)
    a, n = ds.verify(1, dev(target), dev(drafts), dev(dlen), None, None, seed=5,
                     request_id=dev(rid.view(np.int32)), step=2)
    ex = _excluded(ref, B)
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])


def test_verify_rejection_identity_on_gpu():
    """The GPU sampler reproduces the oracle draw for draw on a 10^6-request V = 8
    problem, and its first-token histogram passes the chi-square test against p."""
    from scipy.stats import chisquare
    N, V = 1_000_000, 8
    zl = np.array([1.0, 0.2, -0.5, 2.0, 0.0, -1.0, 0.7, 0.1], np.float32)
    tl = np.array([0.3, 1.1, -0.2, 1.0, 0.5, -2.0, 0.0, 0.9], np.float32)
    p = np.exp(tl.astype(np.float64) - tl.max()); p /= p.sum()
    q = np.exp(zl.astype(np.float64) - zl.max()); q /= q.sum()
    x = np.random.default_rng(123).choice(V, size=N, p=q).astype(np.int32)
    target = np.broadcast_to(np.stack([tl, tl])[None], (N, 2, V)).copy()
    z = np.broadcast_to(zl[None, None], (N, 1, V)).copy()
    ref = oracle.verify(1, target, x[:, None], None, z, seed=0xC0FFEE, step=3)
    a, n = ds.verify(1, dev(target), dev(x[:, None]), None, dev(z), None, seed=0xC0FFEE, step=3)
    a, n = host(a), host(n)
    ex = _excluded(ref, N)
    assert ex.mean() < 1e-3
    np.testing.assert_array_equal(a[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(n[~ex], ref["next_token"][~ex])
    first = np.where(a == 1, x, n)
    counts = np.bincount(first, minlength=V)
    assert chisquare(counts, p * counts.sum()).pvalue > 1e-3


# ----------------------------------------------------------------------------- readout

@pytest.mark.parametrize("B,k,H,tau,bias", [(3, 1, 64, 0.5, 0.0), (5, 16, 5120, 0.5, 0.0),
                                             (4, 7, 2560, 0.3, 0.2), (2, 5, 128, 0.7, -0.1),
                                             (6, 4, 256, 0.0, 0.0), (6, 4, 256, 1.0, 0.0)])
def test_confidence_truncate_matches_oracle(B, k, H, tau, bias):
    """Confidence head alone at block sizes 1..16 (one to 32 warps per position): the
    sigmoid within rtol 1e-5, draft_len and the -1 masking exact wherever no decision
    is within 1e-4 of the threshold; tau <= 0 keeps all, tau >= 1 keeps none."""
    h = syn.normal_bf16(40 + k, (B * k, H))
    cw = syn.normal_bf16(41 + H, (H,), (4.0 / H) ** 0.5)
    d0 = np.tile(np.arange(k, dtype=np.int32), (B, 1)) + 3
    ref = oracle.confidence(h, B, k, cw, bias, tau, d0)
    drafts = dev(d0)
    dl, cf = ds.confidence_truncate(dev_bf16(h), dev_bf16(cw), drafts, B, k, bias, tau,
                                    conf_out=torch.empty((B, k), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    np.testing.assert_allclose(host(cf), ref["conf"], rtol=1e-5, atol=1e-6)
    import math
    thr = -math.inf if tau <= 0 else (math.inf if tau >= 1 else math.log(tau) - math.log1p(-tau))
    safe = np.all(np.abs(ref["zc"] - thr) >= 1e-4, axis=1) if np.isfinite(thr) else np.ones(B, bool)
    np.testing.assert_array_equal(host(dl)[safe], ref["draft_len"][safe])
    np.testing.assert_array_equal(host(drafts)[safe], ref["draft_tokens"][safe])
    if tau <= 0:
        assert (host(dl) == k).all()
    if tau >= 1:
        assert (host(dl) == 0).all() and (host(drafts) == -1).all()


def test_draft_readout_with_confidence_matches_oracle():
    B, k, H, V, r = 4, 7, 256, 5000, 16
    h = syn.normal_bf16(61, (B * k, H))
    lm = syn.normal_bf16(62, (V, H), (1.0 / H) ** 0.5)
    w1 = syn.normal_bf16(63, (V, r))
    w2 = syn.normal_bf16(64, (V, r), (1.0 / r) ** 0.5)
    cw = syn.normal_bf16(65, (H,), (1.0 / H) ** 0.5)
    prev = np.array([1, 2, 3, 4999], np.int32)
    ref_logits = oracle.lm_head(h, lm).reshape(B, k, V)
    ref = oracle.greedy_sample(ref_logits, w1, w2, prev)
    conf = oracle.confidence(h, B, k, cw, 0.0, 0.5, ref["draft_tokens"])
    out = ds.draft_readout(dev_bf16(h), dev_bf16(lm), dev_bf16(w1), dev_bf16(w2), dev(prev), B, k,
                           conf_w=dev_bf16(cw), conf_b=0.0, conf_tau=0.5)
    torch.cuda.synchronize()
    _assert_logits_close(host(out["logits"]), ref["z"])
    # confidence decisions away from the boundary are exact
    safe = np.abs(conf["zc"]) >= 1e-4
    np.testing.assert_allclose(host(out["conf"]), conf["conf"], rtol=1e-5, atol=1e-6)
    gl = host(out["draft_len"])
    for b in range(B):
        if np.all(safe[b, : min(k, conf["draft_len"][b] + 1)]):
            assert gl[b] == conf["draft_len"][b]
    # tokens: equal, or a flip between entries the oracle cannot separate within the
    # logit tolerance (then the rest of that request's chain is not comparable)
    gd = host(out["draft_tokens"])
    for b in range(B):
        for i in range(gl[b]):
            if gd[b, i] != conf["draft_tokens"][b, i]:
                zrow = ref["z"][b, i].astype(np.float64)
                top = zrow.max()
                assert top - zrow[gd[b, i]] <= 2 * (LOGIT_ATOL + LOGIT_RTOL * abs(top))
                break


def test_one_workspace_serves_calls_of_different_shapes():
    """A workspace reused for another shape can hold old partial sums where the new
    shape keeps its counters; results must not depend on the call history."""
    wsp = ds.Workspaces()
    H = 256
    cases = [(7, 4096), (300, 777), (7, 20000), (33, 1000), (7, 4096)]
    for M, V in cases:
        h = syn.normal_bf16(M, (M, H))
        w = syn.normal_bf16(V, (V, H), (1.0 / H) ** 0.5)
        got = host(ds.lm_head(dev_bf16(h), dev_bf16(w), workspaces=wsp))
        _assert_logits_close(got, oracle.lm_head(h, w))
    for B, k, V in [(1, 7, 4096), (9, 3, 30000), (1, 16, 4096), (2, 7, 30000)]:
        z, drafts, target = _verify_inputs(B, k, V, 300 + B * k)
        ref = oracle.verify(0, target, drafts)
        a, n = ds.verify(0, dev(target), dev(drafts), workspaces=wsp)
        np.testing.assert_array_equal(host(a), ref["accepted_len"])
        np.testing.assert_array_equal(host(n), ref["next_token"])
        logits = syn.uniform_logits(400 + B, (B, k, V), 1.0)
        w1 = syn.normal_bf16(5, (V, 16))
        w2 = syn.normal_bf16(6, (V, 16), 0.25)
        prev = np.arange(B, dtype=np.int32)
        refc = oracle.greedy_sample(logits, w1, w2, prev)
        d, _ = ds.greedy_sample(dev(logits), dev_bf16(w1), dev_bf16(w2), dev(prev), workspaces=wsp)
        np.testing.assert_array_equal(host(d), refc["draft_tokens"])
