"""Row statistics and the one-kernel verify from precomputed statistics (the split of
verify the step pipeline runs: target-row statistics beside the GEMMs, then one decision
kernel after drafting), through the C ABI against the CPU oracle.

Tolerances: the row max and argmax are exact (the max of fp32 values is one of them; the
argmax is the lowest index holding it); the sum of exp(x - max) is reduced in fp32 per
16384-entry slice and merged in fp64 on the GPU, in fp64 throughout by the oracle:
within rtol 1e-5.  Verify decisions on identical inputs are bit-exact except the
oracle-flagged ones (|u - p/q| < 1e-5, draw gaps within its binary32 bound), counted.
"""
import numpy as np
import pytest
import torch

import oracle
import parity_log
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import dev, dev_bf16, host
from step_util import decision_mask

pytestmark = pytest.mark.gpu


# rows of one partial slice, exactly one slice, several slices with a ragged tail, odd V
# (scalar loads), the 27B vocabulary
@pytest.mark.parametrize("rows,V", [(3, 100), (5, 16384), (7, 40001), (9, 4099), (16, 151936),
                                    (1, 1), (130, 3000)])
def test_row_stats_matches_oracle(rows, V):
    x = syn.uniform_logits(900 + V + rows, (rows, V), 2.0)
    if V > 10:
        x[0, V // 3] = x[0].max() + 1.0
        x[0, V // 2] = x[0, V // 3]              # tie: the lower index wins
    if rows > 2 and V > 20:
        x[1, ::5] = -np.inf                      # masked entries
        x[2, :] = -np.inf                        # a fully masked row
    ms, arg = ds.row_stats(dev(x))
    ms, arg = host(ms), host(arg)
    ref = oracle.row_stats(x)
    np.testing.assert_array_equal(arg, ref["argmax"])
    np.testing.assert_array_equal(ms[:, 0].astype(np.float64), ref["max"])
    np.testing.assert_allclose(ms[:, 1], ref["sumexp"], rtol=1e-5, atol=0)


def test_row_stats_argmax_only_and_3d_rows():
    B, k1, V = 4, 8, 20000
    x = syn.uniform_logits(77, (B, k1, V), 1.0)
    ms, arg = ds.row_stats(dev(x), want_ms=False)
    assert ms is None
    np.testing.assert_array_equal(host(arg), oracle.row_stats(x)["argmax"])


def _inputs(B, k, V, seed):
    z = syn.uniform_logits(seed, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    noise = syn.uniform_logits(seed + 1, (B, k + 1, V), 1.0) * \
        np.linspace(0.5, 3.0, k + 1)[None, :, None].astype(np.float32)
    target = (np.concatenate([z, z[:, -1:]], axis=1) + noise).astype(np.float32)
    t = target.argmax(axis=-1).astype(np.int32)
    drafts[1::3, :] = t[1::3, :k]       # some requests accept long prefixes
    return z, drafts, target


@pytest.mark.parametrize("B,k,V", [(1, 7, 151936), (16, 7, 151936), (5, 3, 4099), (64, 4, 20001),
                                   (3, 16, 1000)])
@pytest.mark.parametrize("mode", [0, 1])
def test_verify_from_stats_matches_oracle_and_verify(B, k, V, mode):
    z, drafts, target = _inputs(B, k, V, 1000 + B * k + V)
    dlen = np.array([(k - b) % (k + 1) for b in range(B)], np.int32)
    rid = (np.arange(B, dtype=np.uint32) * 7919 + 3).astype(np.uint32)
    gt, gz, gd, gl = dev(target), dev(z), dev(drafts), dev(dlen)
    grid = dev(rid.view(np.int32))
    tms, targ = ds.row_stats(gt)
    qms, _ = ds.row_stats(gz, want_argmax=False)
    a, n = ds.verify_from_stats(mode, gt, tms, targ, gd, gl, gz if mode == 1 else None,
                                qms if mode == 1 else None, seed=99, request_id=grid, step=4)
    a2, n2 = ds.verify(mode, gt, gd, gl, gz if mode == 1 else None, None, seed=99,
                       request_id=grid, step=4)
    np.testing.assert_array_equal(host(a), host(a2))
    np.testing.assert_array_equal(host(n), host(n2))
    ref = oracle.verify(mode, target, drafts, dlen, z if mode == 1 else None, seed=99,
                        request_id=rid, step=4)
    if mode == 0:
        np.testing.assert_array_equal(host(a), ref["accepted_len"])
        np.testing.assert_array_equal(host(n), ref["next_token"])
        return
    ex_a, ex_d = decision_mask(ref)
    ex = ex_a | ex_d
    parity_log.record("verify_from_stats B=%d k=%d V=%d" % (B, k, V), "request", B,
                      accept=ex_a.sum(), draw=ex_d.sum())
    assert ex.sum() <= max(1, B // 16)
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])


def test_verify_from_stats_one_hot_q():
    """draft_logits NULL: q is one-hot at the draft (accept with probability p(d),
    residual = p without d)."""
    B, k, V = 12, 5, 30000
    z, drafts, target = _inputs(B, k, V, 555)
    gt = dev(target)
    tms, targ = ds.row_stats(gt)
    a, n = ds.verify_from_stats(1, gt, tms, targ, dev(drafts), None, None, None, seed=3, step=8)
    ref = oracle.verify(1, target, drafts, None, None, seed=3, step=8)
    ex_a, ex_d = decision_mask(ref)
    ex = ex_a | ex_d
    parity_log.record("verify_from_stats one-hot q B=12", "request", B, accept=ex_a.sum(),
                      draw=ex_d.sum())
    assert ex.sum() <= 1
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])


def test_chain_q_stats_feed_verify_from_stats():
    """The pipeline of the benchmark at a reduced vocabulary: the chain's own q
    statistics (not a separate pass over the draft logits) drive the decisions."""
    B, k, V, r = 8, 7, 50000, 64
    logits = syn.uniform_logits(31, (B, k, V), 1.0)
    w1 = syn.normal_bf16(32, (V, r))
    w2 = syn.normal_bf16(33, (V, r), (1.0 / r) ** 0.5)
    prev = np.arange(B, dtype=np.int32) * 17
    lg = dev(logits)
    d, qs = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev))
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
    np.testing.assert_allclose(host(qs)[..., 1], ref["q_sumexp"], rtol=1e-5)
    noise = syn.uniform_logits(34, (B, k + 1, V), 1.5)
    target = (np.concatenate([ref["z"], ref["z"][:, -1:]], axis=1) + noise).astype(np.float32)
    gt = dev(target)
    tms, targ = ds.row_stats(gt)
    a, n = ds.verify_from_stats(1, gt, tms, targ, d, None, lg, qs, seed=11, step=2)
    ver = oracle.verify(1, target, ref["draft_tokens"], None, ref["z"], seed=11, step=2)
    ex_a, ex_d = decision_mask(ver)
    ex = ex_a | ex_d
    parity_log.record("chain q_stats -> verify_from_stats B=8", "request", B, accept=ex_a.sum(),
                      draw=ex_d.sum())
    assert ex.sum() <= 1
    np.testing.assert_array_equal(host(a)[~ex], ver["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ver["next_token"][~ex])
