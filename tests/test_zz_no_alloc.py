"""The allocation-free verify entry point, called through the C ABI, gives the same
accepted lengths and next tokens as dspark_verify with a caller workspace, on calls of
different shapes in a row (each later call finds the earlier call's leftovers in the
shared scratch).

For callers that are handed only input and output buffers by a framework that owns all
other device memory, or that must not call cudaMalloc while they run.  Outputs are
integers computed by the same kernels, so the comparison is exact.

Collected last on purpose (file name), so that a run stopping at the first failure has
run every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_fc_gb300 as ds
import synthetic as syn

pytestmark = pytest.mark.gpu

_vp = ctypes.c_void_p


def _entry():
    f = ds.lib().dspark_verify_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_uint64, _vp, ctypes.c_uint32,
                  _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]
    return f


def _p(t):
    return None if t is None else _vp(t.data_ptr())


def _inputs(B, k, V, seed):
    z = syn.uniform_logits(seed, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    noise = syn.uniform_logits(seed + 1, (B, k + 1, V), 1.0)
    target = (np.concatenate([z, z[:, -1:]], axis=1) + noise).astype(np.float32)
    t = target.argmax(axis=-1).astype(np.int32)
    drafts[::2, :2] = t[::2, :2]
    return (torch.from_numpy(target).cuda(), torch.from_numpy(drafts).cuda(),
            torch.from_numpy(z).cuda())


def _call(f, mode, target, drafts, dlen, z, qs, seed, step, B, k, V):
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    rc = f(mode, _p(target), _p(drafts), _p(dlen), _p(z), _p(qs), seed, None, step, _p(acc),
           _p(nxt), B, k, V, _vp(stream.cuda_stream))
    assert rc == 0, ds.lib().dspark_status_string(rc)
    return acc, nxt


def test_noalloc_verify_matches_workspace_verify_on_calls_in_a_row():
    """Calls of different shapes in a row share the one scratch array: the first call
    (64 requests, 16 positions, 65536 entries) leaves tickets and partial sums laid out
    for its shape where the next call (3 requests, 5 positions, a ragged 20001-entry
    vocabulary, draft lengths, q statistics from the drafting kernel) keeps other data;
    a greedy call of a third shape follows.  Each must equal dspark_verify with its own
    workspace."""
    f = _entry()
    cases = [(1, 64, 16, 65536, False, False), (1, 3, 5, 20001, True, True),
             (0, 9, 7, 4099, True, False)]
    for call, (mode, B, k, V, with_len, chain_q) in enumerate(cases):
        target, drafts, z = _inputs(B, k, V, 900 + 10 * call)
        dlen = torch.tensor([(k - b) % (k + 1) for b in range(B)], dtype=torch.int32,
                            device="cuda") if with_len else None
        qs = None
        if chain_q:
            # q's statistics as the drafting kernel writes them (unbiased chain here)
            z2 = z.clone()
            prev = torch.zeros((B,), dtype=torch.int32, device="cuda")
            d2, qs = ds.greedy_sample(z2, None, None, prev)
            drafts = d2
        seed, step = 0xABCDEF + call, 3 + call
        ref_a, ref_n = ds.verify(mode, target, drafts, dlen, z if mode == 1 else None, qs,
                                 seed=seed, step=step, workspaces=ds.Workspaces())
        acc, nxt = _call(f, mode, target, drafts, dlen, z if mode == 1 else None, qs, seed, step,
                         B, k, V)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(acc.cpu().numpy(), ref_a.cpu().numpy())
        np.testing.assert_array_equal(nxt.cpu().numpy(), ref_n.cpu().numpy())


def test_noalloc_verify_rejects_sizes_beyond_its_scratch():
    f = _entry()
    need = ds.lib().dspark_verify_workspace_size(4096, 16, 151936)
    assert need > 4 << 20
    fake = _vp(1 << 20)   # rejected on the host before any pointer is used
    rc = f(1, fake, fake, None, fake, None, 0, None, 0, fake, fake, 4096, 16, 151936, None)
    assert rc == -4   # DSPARK_ERR_WORKSPACE
