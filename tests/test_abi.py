"""The C ABI library loads and exports every function declared in include/dspark.h,
and its host-side argument checks answer without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def libdspark():
    from speculative_decoding_fc_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(dspark_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("dspark_fc_project", "dspark_lm_head", "dspark_greedy_sample", "dspark_draft_readout",
              "dspark_verify", "dspark_status_string", "dspark_workspace_status"):
        assert n in names


def test_every_declared_symbol_is_exported(libdspark):
    missing = [n for n in declared_functions() if not hasattr(libdspark, n)]
    assert not missing, missing


def test_status_strings(libdspark):
    f = libdspark.dspark_status_string
    f.restype = ctypes.c_char_p
    f.argtypes = [ctypes.c_int]
    assert f(0) == b"DSPARK_OK"
    assert f(-1) == b"DSPARK_ERR_INVALID_ARG"
    assert f(-6) == b"DSPARK_ERR_DEVICE_TIMEOUT"
    assert f(12345) == b"DSPARK_ERR_UNKNOWN"


def test_workspace_sizes_are_host_only(libdspark):
    sz = ctypes.c_size_t
    libdspark.dspark_lm_head_workspace_size.restype = sz
    libdspark.dspark_verify_workspace_size.restype = sz
    libdspark.dspark_draft_readout_workspace_size.restype = sz
    libdspark.dspark_fc_project_workspace_size.restype = sz
    assert libdspark.dspark_lm_head_workspace_size(7, 5120, 151936) > 0
    assert libdspark.dspark_fc_project_workspace_size(7, 5120, 5) > 0
    assert libdspark.dspark_draft_readout_workspace_size(16, 7, 5120, 151936, 64) > 0
    assert libdspark.dspark_verify_workspace_size(16, 7, 151936) > 0
    assert libdspark.dspark_verify_workspace_size(16, 17, 151936) == 0   # k > 16
    assert libdspark.dspark_lm_head_workspace_size(0, 5120, 151936) == 0


def test_argument_errors_are_caught_before_any_launch(libdspark):
    vp = ctypes.c_void_p
    f = libdspark.dspark_verify
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_uint64, vp, ctypes.c_uint32, vp, vp,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    fake = vp(1 << 20)  # never dereferenced: the checks reject the call first
    assert f(2, fake, fake, None, None, None, 0, None, 0, fake, fake, 1, 7, 100, fake, 1 << 20, None) == -1
    assert f(0, None, fake, None, None, None, 0, None, 0, fake, fake, 1, 7, 100, fake, 1 << 20, None) == -1
    assert f(0, fake, fake, None, None, None, 0, None, 0, fake, fake, 1, 17, 100, fake, 1 << 20, None) == -2
    assert f(0, vp((1 << 20) + 2), fake, None, None, None, 0, None, 0, fake, fake, 1, 7, 100, fake,
             1 << 20, None) == -3
    assert f(0, fake, fake, None, None, None, 0, None, 0, fake, fake, 1, 7, 100, fake, 16, None) == -4
    g = libdspark.dspark_lm_head
    g.restype = ctypes.c_int
    g.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    assert g(fake, fake, fake, 7, 100, 1000, fake, 1 << 30, None) == -2   # H not a multiple of 64
    assert g(fake, fake, fake, 0, 128, 1000, fake, 1 << 30, None) == -1


def test_fp8_argument_errors_are_caught_before_any_launch(libdspark):
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    fake = vp(1 << 20)
    q = libdspark.dspark_quantize_fp8
    q.restype = ctypes.c_int
    q.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, vp,
                  vp, vp]
    segs = (vp * 2)(1 << 20, 1 << 21)
    assert q(segs, 0, 64, 4, 64, fake, fake, None) == -1          # no segment
    assert q(segs, 2, 64, 4, 24, fake, fake, None) == -2          # seg_cols % 16
    assert q(segs, 2, 60, 4, 48, fake, fake, None) == -3          # seg_ld % 8
    assert q(segs, 2, 64, 4, 64, vp((1 << 20) + 8), fake, None) == -3   # codes not 16-B aligned
    libdspark.dspark_lm_head_fp8_workspace_size.restype = sz
    libdspark.dspark_fc_project_fp8_workspace_size.restype = sz
    assert libdspark.dspark_lm_head_fp8_workspace_size(7, 5120, 151936) > 7 * 5120
    assert libdspark.dspark_fc_project_fp8_workspace_size(7, 5120, 5) > 7 * 5 * 5120
    assert libdspark.dspark_fc_project_fp8_workspace_size(7, 5120, 9) == 0
    g = libdspark.dspark_lm_head_fp8
    g.restype = ctypes.c_int
    g.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, sz, vp]
    assert g(fake, fake, fake, fake, 7, 192, 1000, fake, 1 << 30, None) == -2   # H % 128
    assert g(fake, fake, None, fake, 7, 256, 1000, fake, 1 << 30, None) == -1   # no scales
    assert g(fake, fake, fake, fake, 7, 256, 1000, fake, 16, None) == -4        # workspace
    f = libdspark.dspark_fc_project_fp8
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, vp, vp, vp, ctypes.c_int,
                  ctypes.c_int, vp, sz, vp]
    taps = (vp * 2)(1 << 20, 1 << 21)
    assert f(taps, 2, 256, fake, fake, fake, 4, 192, fake, 1 << 30, None) == -2   # H % 128
    assert f(taps, 2, 256, fake, fake, fake, 4, 256, fake, 16, None) == -4


def test_fc_lm_head_sizes_and_argument_errors(libdspark):
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    libdspark.dspark_fc_lm_head_workspace_size.restype = sz
    n = libdspark.dspark_fc_lm_head_workspace_size(7, 5120, 5, 151936)
    libdspark.dspark_fc_project_workspace_size.restype = sz
    libdspark.dspark_lm_head_workspace_size.restype = sz
    assert n >= libdspark.dspark_fc_project_workspace_size(7, 5120, 5) + \
        libdspark.dspark_lm_head_workspace_size(7, 5120, 151936) - 256
    assert libdspark.dspark_fc_lm_head_workspace_size(7, 5120, 9, 151936) == 0
    f = libdspark.dspark_fc_lm_head
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, vp, vp, vp, vp, ctypes.c_int,
                  ctypes.c_int, ctypes.c_int, vp, sz, vp]
    fake = vp(1 << 20)
    taps = (vp * 2)(1 << 20, 1 << 21)
    assert f(taps, 2, 128, fake, fake, fake, None, 4, 128, 100, fake, 1 << 30, None) == -1
    assert f(taps, 2, 128, fake, fake, fake, fake, 4, 96, 100, fake, 1 << 30, None) == -2
    assert f(taps, 2, 128, fake, vp((1 << 20) + 8), fake, fake, 4, 128, 100, fake, 1 << 30,
             None) == -3
    assert f(taps, 2, 128, fake, fake, fake, fake, 4, 128, 100, fake, 16, None) == -4


def test_row_stats_and_verify_from_stats_argument_errors(libdspark):
    vp, sz, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
    libdspark.dspark_row_stats_workspace_size.restype = sz
    libdspark.dspark_row_stats_workspace_size.argtypes = [i64, ctypes.c_int]
    libdspark.dspark_verify_from_stats_workspace_size.restype = sz
    assert libdspark.dspark_row_stats_workspace_size(128, 151936) > 128 * 10 * 16
    assert libdspark.dspark_row_stats_workspace_size(0, 151936) == 0
    assert libdspark.dspark_row_stats_workspace_size(8, (1 << 26) + 1) == 0
    assert libdspark.dspark_verify_from_stats_workspace_size(16, 7, 151936) > 16 * 149 * 16
    assert libdspark.dspark_verify_from_stats_workspace_size(16, 17, 151936) == 0
    fake = vp(1 << 20)
    r = libdspark.dspark_row_stats
    r.restype = ctypes.c_int
    r.argtypes = [vp, i64, ctypes.c_int, vp, vp, vp, sz, vp]
    assert r(fake, 8, 100, None, None, fake, 1 << 30, None) == -1              # no output
    assert r(fake, 0, 100, fake, None, fake, 1 << 30, None) == -1              # no rows
    assert r(fake, 8, 100, vp((1 << 20) + 4), None, fake, 1 << 30, None) == -3  # ms not 8-B aligned
    assert r(fake, 8, 100, fake, fake, fake, 16, None) == -4                    # workspace too small
    f = libdspark.dspark_verify_from_stats
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, ctypes.c_uint64, vp, ctypes.c_uint32,
                  vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, sz, vp]
    big = 1 << 30
    # greedy needs the target argmax; probabilistic the target (max, sum) and, with draft
    # logits, q's statistics
    assert f(0, fake, fake, None, fake, None, None, None, 0, None, 0, fake, fake, 2, 7, 100, fake, big, None) == -1
    assert f(1, fake, None, fake, fake, None, None, None, 0, None, 0, fake, fake, 2, 7, 100, fake, big, None) == -1
    assert f(1, fake, fake, fake, fake, None, fake, None, 0, None, 0, fake, fake, 2, 7, 100, fake, big, None) == -1
    assert f(1, fake, fake, fake, fake, None, fake, vp((1 << 20) + 4), 0, None, 0, fake, fake, 2, 7,
             100, fake, big, None) == -3
    assert f(0, fake, fake, fake, fake, None, None, None, 0, None, 0, fake, fake, 2, 17, 100, fake, big, None) == -2
    assert f(0, fake, fake, fake, fake, None, None, None, 0, None, 0, fake, fake, 2, 7, 100, fake, 16, None) == -4


def test_verify_noalloc_rejects_before_enqueueing(libdspark):
    """Argument and size errors of the allocation-free verify come back before any GPU
    work is queued (the checks run on the host; no device is needed to reach them)."""
    vp = ctypes.c_void_p
    f = libdspark.dspark_verify_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_uint64, vp, ctypes.c_uint32, vp, vp,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    fake = vp(1 << 20)
    assert f(3, fake, fake, None, None, None, 0, None, 0, fake, fake, 2, 7, 100, None) == -1
    assert f(0, fake, fake, None, None, None, 0, None, 0, fake, fake, 2, 17, 100, None) == -2
    assert f(0, vp((1 << 20) + 2), fake, None, None, None, 0, None, 0, fake, fake, 2, 7, 100, None) == -3
    # beyond the fixed scratch: 1024 requests of 16 positions over 2^20 entries
    assert f(0, fake, fake, None, None, None, 0, None, 0, fake, fake, 1024, 16, 1 << 20, None) == -4


def test_backbone_block_sizes_and_argument_errors(libdspark):
    """dspark_backbone_block: the workspace size and every argument check answer on the
    host (fake, never dereferenced pointers)."""
    vp, c = ctypes.c_void_p, ctypes.c_int

    class Layer(ctypes.Structure):
        _fields_ = [(n, vp) for n in ("w_in", "w_post", "w_qn", "w_kn", "w_qkv", "w_o", "w_gu", "w_d",
                                      "k_cache", "v_cache")] + \
                   [("nq", c), ("nkv", c), ("I", c), ("theta", ctypes.c_float)]

    fake = 1 << 20

    def layers(nq=40, nkv=8, I=17408, theta=1e6, misalign=False):
        arr = (Layer * 1)()
        arr[0] = Layer(*([fake] * 9 + [fake + (2 if misalign else 0)]), nq, nkv, I, theta)
        return arr

    sz = libdspark.dspark_backbone_block_workspace_size
    sz.restype = ctypes.c_size_t
    sz.argtypes = [c, c, c, c, vp, c, c]
    p = lambda a: ctypes.cast(a, vp)
    assert sz(1, 8, 5120, 1, p(layers()), 7, 1024) > 0
    assert sz(1, 1, 5120, 1, p(layers()), 7, 1024) == 0          # a block needs the anchor and a mask row
    assert sz(1, 8, 5100, 1, p(layers()), 7, 1024) == 0          # H not a multiple of 64
    assert sz(1, 8, 5120, 1, p(layers(nq=40, nkv=7)), 7, 1024) == 0   # nq % nkv != 0
    assert sz(1, 8, 5120, 1, p(layers(nq=64, nkv=8)), 7, 1024) == 0   # 8 rows x 8 heads > 48 queries

    f = libdspark.dspark_backbone_block
    f.restype = c
    f.argtypes = [vp, c, c, vp, c, c, c, vp, vp, c, c, vp, c, c, vp, vp, ctypes.c_size_t, vp]
    ok = dict(tokens=fake, B=1, nr=8, embed=fake, V=151936, H=5120, L=1, layers=p(layers()), wf=fake,
              cache_len=1032, C=1024, ctx=fake, nctx=7, pos0=1017, out=fake, ws=fake, wsb=1 << 40)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["tokens"], a["B"], a["nr"], a["embed"], a["V"], a["H"], a["L"], a["layers"], a["wf"],
                 a["cache_len"], a["C"], a["ctx"], a["nctx"], a["pos0"], a["out"], a["ws"], a["wsb"], None)

    assert call(tokens=None) == -1
    assert call(C=1025) == -1                     # the block's slots pass the cache's end
    assert call(pos0=1026) == -1                  # the context rows' slots pass it
    assert call(H=5100) == -2
    assert call(out=fake + 2) == -3
    assert call(layers=p(layers(misalign=True))) == -3
    assert call(layers=p(layers(theta=1.0))) == -1
    assert call(L=0) == -1
    assert call(wsb=16) == -4
