"""The allocation-free verify entry point, called through the C ABI, gives the same
accepted lengths and next tokens as dspark_verify with a caller workspace, on two calls
in a row (the second call finds the first call's leftovers in the shared scratch).

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


@pytest.mark.parametrize("mode", [1, 0])
def test_noalloc_verify_matches_workspace_verify_twice(mode):
    f = _entry()
    B, k, V = 16, 7, 20000
    stream = torch.cuda.current_stream()
    for call in range(2):
        target, drafts, z = _inputs(B, k, V, 900 + 10 * call + mode)
        seed, step = 0xABCDEF + call, 3 + call
        ref_a, ref_n = ds.verify(mode, target, drafts, None, z if mode == 1 else None, None,
                                 seed=seed, step=step)
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        rc = f(mode, _p(target), _p(drafts), None, _p(z) if mode == 1 else None, None, seed, None,
               step, _p(acc), _p(nxt), B, k, V, _vp(stream.cuda_stream))
        assert rc == 0, ds.lib().dspark_status_string(rc)
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
