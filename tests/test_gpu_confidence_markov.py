"""Confidence head with the Markov context and the cumulative truncation rule, through
the C ABI against the CPU oracle.

Tolerances: the sigmoid within rtol 1e-5 (fp32 dot products vs fp64); draft lengths and
the -1 masking exact wherever no decision lies within 1e-4 of its threshold (per
position: |zc - logit tau|; cumulative: |sum of log sigmoid - log tau|), those counted.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import parity_log
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cumulative", [False, True])
@pytest.mark.parametrize("B,k,H,V,r,tau", [(16, 7, 5120, 151936, 64, 0.5), (5, 16, 256, 4096, 16, 0.3),
                                           (3, 1, 64, 1000, 8, 0.5), (8, 7, 2560, 151936, 128, 0.1)])
def test_confidence_markov_matches_oracle(B, k, H, V, r, tau, cumulative):
    h = syn.normal_bf16(70 + k, (B * k, H))
    # a head whose Markov part matters: weights of comparable size on both parts
    cw = np.concatenate([syn.normal_bf16(71 + H, (H,), (1.0 / H) ** 0.5),
                         syn.normal_bf16(72 + r, (r,), (1.0 / r) ** 0.5)])
    w1 = syn.normal_bf16(73, (V, r))
    prev = np.random.default_rng(B).integers(0, V, B).astype(np.int32)
    d0 = np.random.default_rng(B + 1).integers(0, V, (B, k)).astype(np.int32)
    ref = oracle.confidence_markov(h, B, k, cw, 0.2, tau, d0, cumulative, w1, prev)
    drafts = dev(d0)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    dl, cf = ds.confidence_truncate_markov(dev_bf16(h), dev_bf16(cw), drafts, B, k, 0.2, tau,
                                           cumulative=cumulative, w1=dev_bf16(w1), prev_token=dev(prev),
                                           conf_out=torch.empty((B, k), dtype=torch.float32, device="cuda"),
                                           status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_allclose(host(cf), ref["conf"], rtol=1e-5, atol=1e-6)
    if cumulative:
        dist = np.abs(ref["cum"] - math.log(tau))
    else:
        dist = np.abs(ref["zc"] - (math.log(tau) - math.log1p(-tau)))
    safe = np.array([not (dist[b, :min(k, ref["draft_len"][b] + 1)] < 1e-4).any() for b in range(B)])
    parity_log.record("confidence_markov B=%d k=%d H=%d %s" % (B, k, H, "cum" if cumulative else "pos"),
                      "request", B, confidence=(~safe).sum())
    assert safe.sum() >= B - max(1, B // 8)
    np.testing.assert_array_equal(host(dl)[safe], ref["draft_len"][safe])
    np.testing.assert_array_equal(host(drafts)[safe], ref["draft_tokens"][safe])
    # the product of the prefix's confidences is at most each of them, so the
    # cumulative rule never keeps more positions than the per-position rule
    if cumulative:
        per = oracle.confidence_markov(h, B, k, cw, 0.2, tau, d0, False, w1, prev)
        assert (ref["draft_len"] <= per["draft_len"]).all()


def test_confidence_markov_without_w1_is_the_plain_head():
    B, k, H = 6, 5, 512
    h = syn.normal_bf16(90, (B * k, H))
    cw = syn.normal_bf16(91, (H,), (4.0 / H) ** 0.5)
    d0 = np.tile(np.arange(k, dtype=np.int32), (B, 1))
    a_drafts, b_drafts = dev(d0), dev(d0)
    dl1, _ = ds.confidence_truncate(dev_bf16(h), dev_bf16(cw), a_drafts, B, k, 0.0, 0.5)
    dl2, _ = ds.confidence_truncate_markov(dev_bf16(h), dev_bf16(cw), b_drafts, B, k, 0.0, 0.5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(dl1), host(dl2))
    np.testing.assert_array_equal(host(a_drafts), host(b_drafts))


def test_confidence_markov_bad_context_is_recorded():
    B, k, H, V, r = 2, 3, 64, 100, 8
    h = syn.normal_bf16(95, (B * k, H))
    cw = syn.normal_bf16(96, (H + r,), 0.1)
    w1 = syn.normal_bf16(97, (V, r))
    prev = np.array([5, 100], np.int32)       # 100 is outside [0, V)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    ds.confidence_truncate_markov(dev_bf16(h), dev_bf16(cw), dev(np.zeros((B, k), np.int32)), B, k,
                                  0.0, 0.5, w1=dev_bf16(w1), prev_token=dev(prev), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -7   # DSPARK_ERR_BAD_TOKEN
