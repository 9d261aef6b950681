"""Failure detection on the GPU without a fault: errors the kernels find (a token id
outside [0, V), a draft length outside [0, k], a bounded wait running out) are recorded
in the workspace's status word, read back with dspark_workspace_status, while the
kernels skip the offending access and return.  The timeout is provoked by giving the
chain's waits a zero budget (DSPARK_CHAIN_WAIT_CYCLES), so they give up at once; no
kernel is left spinning and the context stays usable."""
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu

OK, BAD_TOKEN, TIMEOUT, INVALID_ARG = 0, -7, -6, -1


def _status(wsp, kind):
    return ds.workspace_status(wsp.buffer(kind, "cuda"))


def test_bad_prev_token_is_recorded_and_others_are_exact():
    B, k, V, r = 4, 5, 20000, 16
    logits = syn.uniform_logits(5, (B, k, V), 1.0)
    w1 = syn.normal_bf16(6, (V, r))
    w2 = syn.normal_bf16(7, (V, r), 0.25)
    prev = np.array([3, -1, V, 1234], np.int32)
    wsp = ds.Workspaces()
    lg = dev(logits)
    d, _ = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev), workspaces=wsp)
    assert _status(wsp, "chain") == BAD_TOKEN
    assert _status(wsp, "chain") == OK          # the read cleared it
    good = np.array([0, 3])
    ref = oracle.greedy_sample(logits[good], w1, w2, prev[good])
    np.testing.assert_array_equal(host(d)[good], ref["draft_tokens"])
    np.testing.assert_array_equal(host(lg)[good], ref["z"])
    # a request with an invalid context is drafted without bias at position 0, then
    # conditioned on its own drafts as usual
    for b in (1, 2):
        first = oracle.greedy_sample(logits[b:b + 1, :1], None, None, np.zeros(1, np.int32))
        assert host(d)[b, 0] == first["draft_tokens"][0, 0]
        rest = oracle.greedy_sample(logits[b:b + 1, 1:], w1, w2, first["draft_tokens"][:, 0])
        np.testing.assert_array_equal(host(d)[b, 1:], rest["draft_tokens"][0])


@pytest.mark.parametrize("split", [False, True])
def test_bad_draft_token_in_verify(split):
    """A draft outside [0, V) stops its block there (the draws of the other requests are
    untouched); the next token is then drawn from p of that row, which is what the oracle
    does for a block of that many drafts."""
    B, k, V = 6, 4, 9000
    z = syn.uniform_logits(21, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    target = (np.concatenate([z, z[:, -1:]], axis=1) + syn.uniform_logits(22, (B, k + 1, V), 0.3)).astype(np.float32)
    drafts[2, 1] = V + 5
    drafts[4, 0] = -3
    wsp = ds.Workspaces()
    gt, gz, gd = dev(target), dev(z), dev(drafts)
    if split:
        tms, targ = ds.row_stats(gt, workspaces=wsp)
        qms, _ = ds.row_stats(gz, want_argmax=False, workspaces=wsp)
        a, n = ds.verify_from_stats(1, gt, tms, targ, gd, None, gz, qms, seed=1, step=1, workspaces=wsp)
        kind = "verify_fs"
    else:
        a, n = ds.verify(1, gt, gd, None, gz, None, seed=1, step=1, workspaces=wsp)
        kind = "verify"
    assert _status(wsp, kind) == BAD_TOKEN
    dlen = np.full(B, k, np.int32)
    dlen[2], dlen[4] = 1, 0
    ref = oracle.verify(1, target, np.where(drafts >= 0, np.minimum(drafts, V - 1), 0), dlen, z,
                        seed=1, step=1)
    a, n = host(a), host(n)
    assert a[4] == 0 and a[2] <= 1
    np.testing.assert_array_equal(a, ref["accepted_len"])
    np.testing.assert_array_equal(n, ref["next_token"])


def test_draft_len_out_of_range_is_recorded():
    B, k, V = 3, 4, 5000
    z = syn.uniform_logits(41, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    target = np.concatenate([z, z[:, -1:]], axis=1).astype(np.float32)
    dlen = np.array([k + 3, 2, -1], np.int32)
    wsp = ds.Workspaces()
    a, n = ds.verify(0, dev(target), dev(drafts), dev(dlen), workspaces=wsp)
    assert _status(wsp, "verify") == INVALID_ARG
    ref = oracle.verify(0, target, drafts, np.array([k, 2, 0], np.int32))  # clamped
    np.testing.assert_array_equal(host(a), ref["accepted_len"])
    np.testing.assert_array_equal(host(n), ref["next_token"])


@pytest.mark.parametrize("B", [2, 16])   # 16: the two-halves kernel
def test_chain_wait_timeout_is_recorded_and_the_context_survives(B):
    k, V, r = 7, 151936, 64
    logits = syn.uniform_logits(51, (B, k, V), 1.0)
    w1 = dev_bf16(syn.normal_bf16(52, (V, r)))
    w2 = dev_bf16(syn.normal_bf16(53, (V, r), 0.125))
    prev = dev((np.arange(B) * 7 + 5).astype(np.int32))
    old = os.environ.get("DSPARK_CHAIN_WAIT_CYCLES")
    seen = []
    try:
        os.environ["DSPARK_CHAIN_WAIT_CYCLES"] = "0"
        for _ in range(5):              # a wait gives up as soon as one word is missing
            wsp = ds.Workspaces()
            ds.greedy_sample(dev(logits), w1, w2, prev, workspaces=wsp)
            torch.cuda.synchronize()
            seen.append(_status(wsp, "chain"))
            if seen[-1] == TIMEOUT:
                break
    finally:
        if old is None:
            del os.environ["DSPARK_CHAIN_WAIT_CYCLES"]
        else:
            os.environ["DSPARK_CHAIN_WAIT_CYCLES"] = old
    assert TIMEOUT in seen, seen
    # the same call with the normal budget on a fresh workspace is exact
    wsp = ds.Workspaces()
    lg = dev(logits)
    d, _ = ds.greedy_sample(lg, w1, w2, prev, workspaces=wsp)
    assert _status(wsp, "chain") == OK
    ref = oracle.greedy_sample(logits, syn.normal_bf16(52, (V, r)), syn.normal_bf16(53, (V, r), 0.125),
                               (np.arange(B) * 7 + 5).astype(np.int32))
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
