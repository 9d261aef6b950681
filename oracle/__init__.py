"""CPU oracle for the DSpark readout + verify hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the benchmark's CPU-baseline leg, never by the product package.  It shares no
code with the CUDA path.  The arithmetic lives in ``dspark_oracle.c`` (plain
C, fp64 accumulation); this module only marshals numpy arrays into it.

bf16 tensors are passed as ``numpy.uint16`` arrays holding the raw bit
patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.oracle_verify_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                             ctypes.c_uint32, _f64p]
        L.oracle_fc_project.restype = ctypes.c_int
        L.oracle_fc_project.argtypes = [ctypes.POINTER(_u16p), ctypes.c_int, ctypes.c_int64, _u16p,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p, _f32p]
        L.oracle_lm_head.restype = ctypes.c_int
        L.oracle_lm_head.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _u16p, ctypes.c_int64, _f32p]
        L.oracle_greedy_sample.restype = ctypes.c_int
        L.oracle_greedy_sample.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _u16p,
                                           _u16p, ctypes.c_int, _i32p, _i32p, _f64p, _f64p, _f64p]
        L.oracle_confidence.restype = ctypes.c_int
        L.oracle_confidence.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p,
                                        ctypes.c_float, ctypes.c_float, _f64p, _f64p, _i32p, _i32p]
        L.oracle_verify.restype = ctypes.c_int
        L.oracle_verify.argtypes = [ctypes.c_int, _f32p, _i32p, _i32p, _f32p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, _u32p,
                                    ctypes.c_uint32, _i32p, _i32p, _f64p, _f64p, _i32p]
        L.oracle_f32_to_bf16_n.argtypes = [_f32p, ctypes.c_int64, _u16p]
        L.oracle_confidence_markov.restype = ctypes.c_int
        L.oracle_confidence_markov.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _u16p,
                                               ctypes.c_float, ctypes.c_float, ctypes.c_int, _u16p,
                                               ctypes.c_int, ctypes.c_int64, _i32p, _i32p, _f64p,
                                               _f64p, _f64p, _i32p]
        L.oracle_row_stats.restype = ctypes.c_int
        L.oracle_row_stats.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _i32p]
        L.oracle_e4m3_to_f32.restype = ctypes.c_float
        L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.oracle_quantize_fp8_rows.restype = ctypes.c_int
        L.oracle_quantize_fp8_rows.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_uint8), _f32p]
        L.oracle_gemm_fp8.restype = ctypes.c_int
        L.oracle_gemm_fp8.argtypes = [ctypes.POINTER(ctypes.c_uint8), _f32p, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_uint8), _f32p, ctypes.c_int64,
                                      ctypes.c_int, _f32p]
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def _p(a, ptype):
    if a is None:
        return None
    return a.ctypes.data_as(ptype)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError("%s failed with oracle status %d" % (what, rc))


# ---------------------------------------------------------------- scalars
def f32_to_bf16(x):
    """Round fp32 values to bf16 bit patterns (ties to even), element by element."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    f = lib().oracle_f32_to_bf16
    for i, v in enumerate(flat):
        out[i] = f(float(v))
    return out.reshape(x.shape)


def bf16_to_f32(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    f = lib().oracle_bf16_to_f32
    return np.array([f(int(b)) for b in bits.reshape(-1)], dtype=np.float32).reshape(bits.shape)


def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(v) & 0xffffffff for v in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(v) & 0xffffffff for v in key])
    o = (ctypes.c_uint32 * 4)()
    lib().oracle_philox4x32_10(c, k, o)
    return [int(v) for v in o]


def verify_uniforms(seed, request, pos, step):
    o = (ctypes.c_double * 2)()
    lib().oracle_verify_uniforms(seed, request, pos, step, o)
    return float(o[0]), float(o[1])


# ---------------------------------------------------------------- hot path
def fc_project(taps, fc_w, return_f32=False):
    """taps: list of T uint16 arrays [M, H]; fc_w: uint16 [N, T*H] (N = H, or fewer rows to
    compute only the first N output features) -> h uint16 [M, N]."""
    taps = [_c(t, np.uint16) for t in taps]
    T = len(taps)
    M, H = taps[0].shape
    fc_w = _c(fc_w, np.uint16)
    N = fc_w.shape[0]
    assert fc_w.shape == (N, T * H) and N <= H
    arr = (_u16p * T)(*[_p(t, _u16p) for t in taps])
    h = np.empty((M, N), dtype=np.uint16)
    hf = np.empty((M, N), dtype=np.float32) if return_f32 else None
    _check(lib().oracle_fc_project(arr, T, H, _p(fc_w, _u16p), N, M, H, _p(h, _u16p),
                                   _p(hf, _f32p)), "oracle_fc_project")
    return (h, hf) if return_f32 else h


def lm_head(h, lm_w):
    """h: uint16 [M, H]; lm_w: uint16 [V, H] -> fp32 logits [M, V]."""
    h = _c(h, np.uint16)
    lm_w = _c(lm_w, np.uint16)
    M, H = h.shape
    V = lm_w.shape[0]
    assert lm_w.shape[1] == H
    out = np.empty((M, V), dtype=np.float32)
    _check(lib().oracle_lm_head(_p(h, _u16p), M, H, _p(lm_w, _u16p), V, _p(out, _f32p)),
           "oracle_lm_head")
    return out


def greedy_sample(logits, w1, w2, prev):
    """logits fp32 [B, k, V] (not modified); returns dict with z, draft_tokens, q_max,
    q_sumexp, top2_gap."""
    z = np.array(logits, dtype=np.float32, copy=True, order="C")
    B, k, V = z.shape
    prev = _c(np.asarray(prev, dtype=np.int32), np.int32)
    r = 0
    if w1 is not None:
        w1 = _c(w1, np.uint16)
        w2 = _c(w2, np.uint16)
        r = w1.shape[1]
        assert w1.shape == (V, r) and w2.shape == (V, r)
    d = np.empty((B, k), dtype=np.int32)
    qm = np.empty((B, k), dtype=np.float64)
    qs = np.empty((B, k), dtype=np.float64)
    gap = np.empty((B, k), dtype=np.float64)
    _check(lib().oracle_greedy_sample(_p(z, _f32p), B, k, V, _p(w1, _u16p), _p(w2, _u16p), r,
                                      _p(prev, _i32p), _p(d, _i32p), _p(qm, _f64p), _p(qs, _f64p),
                                      _p(gap, _f64p)), "oracle_greedy_sample")
    return {"z": z, "draft_tokens": d, "q_max": qm, "q_sumexp": qs, "top2_gap": gap}


def row_stats(x):
    """fp32 rows [..., V] -> dict max (fp64), sumexp (fp64 sum of exp(x - max)), argmax
    (int32, lowest index of the max), each of shape [...]."""
    x = _c(np.asarray(x), np.float32)
    V = x.shape[-1]
    lead = x.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    mx = np.empty(n, np.float64)
    se = np.empty(n, np.float64)
    arg = np.empty(n, np.int32)
    _check(lib().oracle_row_stats(_p(x, _f32p), n, V, _p(mx, _f64p), _p(se, _f64p), _p(arg, _i32p)),
           "oracle_row_stats")
    return {"max": mx.reshape(lead), "sumexp": se.reshape(lead), "argmax": arg.reshape(lead)}


def confidence(h, B, k, conf_w, conf_b, tau, draft_tokens=None):
    """h uint16 [B*k, H]; returns dict zc, conf, draft_len, draft_tokens (masked copy)."""
    h = _c(h, np.uint16)
    H = h.shape[1]
    conf_w = _c(conf_w, np.uint16)
    zc = np.empty((B, k), dtype=np.float64)
    cf = np.empty((B, k), dtype=np.float64)
    L = np.empty((B,), dtype=np.int32)
    dt = None if draft_tokens is None else np.array(draft_tokens, dtype=np.int32, copy=True)
    _check(lib().oracle_confidence(_p(h, _u16p), B, k, H, _p(conf_w, _u16p), float(conf_b),
                                   float(tau), _p(zc, _f64p), _p(cf, _f64p), _p(L, _i32p),
                                   _p(dt, _i32p)), "oracle_confidence")
    return {"zc": zc, "conf": cf, "draft_len": L, "draft_tokens": dt}


def confidence_markov(h, B, k, conf_w, conf_b, tau, draft_tokens, cumulative=False, w1=None,
                      prev=None):
    """Confidence head over [h ; markov_w1[context]] (w1 given: conf_w has H + r entries)
    or over h alone, with the per-position or cumulative truncation rule.  draft_tokens
    [B, k] are the chain's drafts (contexts of positions 1..k-1); returns dict zc, conf,
    cum (running sum of log sigmoid), draft_len, draft_tokens (masked copy)."""
    h = _c(h, np.uint16)
    H = h.shape[1]
    conf_w = _c(conf_w, np.uint16)
    r, V = 0, 0
    if w1 is not None:
        w1 = _c(w1, np.uint16)
        V, r = w1.shape
        assert conf_w.shape == (H + r,)
        prev = _c(np.asarray(prev, np.int32), np.int32)
    else:
        assert conf_w.shape[0] >= H
    dt = np.array(draft_tokens, dtype=np.int32, copy=True)
    zc = np.empty((B, k), np.float64)
    cf = np.empty((B, k), np.float64)
    cum = np.empty((B, k), np.float64)
    L = np.empty((B,), np.int32)
    _check(lib().oracle_confidence_markov(_p(h, _u16p), B, k, H, _p(conf_w, _u16p), float(conf_b),
                                          float(tau), int(bool(cumulative)), _p(w1, _u16p), r, V,
                                          _p(prev, _i32p), _p(dt, _i32p), _p(zc, _f64p), _p(cf, _f64p),
                                          _p(cum, _f64p), _p(L, _i32p)), "oracle_confidence_markov")
    return {"zc": zc, "conf": cf, "cum": cum, "draft_len": L, "draft_tokens": dt}


def verify(mode, target, drafts, draft_len=None, z=None, seed=0, request_id=None, step=0):
    """mode 0 greedy / 1 probabilistic.  target fp32 [B, k+1, V]; drafts int32 [B, k];
    z fp32 [B, k, V] or None (one-hot q)."""
    target = _c(target, np.float32)
    B, k1, V = target.shape
    k = k1 - 1
    drafts = _c(np.asarray(drafts, dtype=np.int32), np.int32)
    assert drafts.shape == (B, k)
    if draft_len is not None:
        draft_len = _c(np.asarray(draft_len, dtype=np.int32), np.int32)
    if z is not None:
        z = _c(z, np.float32)
        assert z.shape == (B, k, V)
    if request_id is not None:
        request_id = _c(np.asarray(request_id, dtype=np.uint32), np.uint32)
    acc = np.empty((B,), dtype=np.int32)
    nxt = np.empty((B,), dtype=np.int32)
    am = np.empty((B, k), dtype=np.float64)
    sm = np.empty((B,), dtype=np.float64)
    sr = np.empty((B,), dtype=np.int32)
    _check(lib().oracle_verify(int(mode), _p(target, _f32p), _p(drafts, _i32p), _p(draft_len, _i32p),
                               _p(z, _f32p), B, k, V, int(seed) & (2**64 - 1), _p(request_id, _u32p),
                               int(step) & 0xffffffff, _p(acc, _i32p), _p(nxt, _i32p), _p(am, _f64p),
                               _p(sm, _f64p), _p(sr, _i32p)), "oracle_verify")
    return {"accepted_len": acc, "next_token": nxt, "accept_margin": am, "sample_margin": sm,
            "sample_row": sr}


def readout(inputs, B, k, conf=None):
    """The drafter half of one step on host arrays: fc -> LM head -> Markov greedy chain
    -> optional confidence truncation.  ``inputs`` holds taps, fc_w, lm_w, w1, w2, prev;
    ``conf`` is None or a dict with w, b, tau.  Returns every intermediate."""
    h = fc_project(inputs["taps"], inputs["fc_w"])
    logits = lm_head(h, inputs["lm_w"]).reshape(B, k, -1)
    gs = greedy_sample(logits, inputs.get("w1"), inputs.get("w2"), inputs["prev"])
    out = {"h": h, "logits": logits, "draft_len": None, **gs}
    if conf is not None:
        c = confidence(h, B, k, conf["w"], conf["b"], conf["tau"], gs["draft_tokens"])
        out.update({"conf": c["conf"], "zc": c["zc"], "draft_len": c["draft_len"],
                    "draft_tokens": c["draft_tokens"]})
    return out


def step(inputs, B, k, mode, target, seed=0, step=0, conf=None):
    """One whole draft+verify step: ``readout`` then ``verify`` against the given target
    logits [B, k+1, V]."""
    out = readout(inputs, B, k, conf)
    out.update(verify(mode, target, out["draft_tokens"], out["draft_len"],
                      out["z"] if mode == 1 else None, seed=seed, step=step))
    return out


# ---------------------------------------------------------------- FP8 (E4M3) weights
_u8p = ctypes.POINTER(ctypes.c_uint8)


def f32_to_e4m3(x):
    x = np.asarray(x, dtype=np.float32)
    f = lib().oracle_f32_to_e4m3
    return np.array([f(float(v)) for v in x.reshape(-1)], dtype=np.uint8).reshape(x.shape)


def e4m3_to_f32(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    f = lib().oracle_e4m3_to_f32
    return np.array([f(int(c)) for c in codes.reshape(-1)], dtype=np.float32).reshape(codes.shape)


def quantize_fp8_rows(x):
    """bf16 bits [R, C] -> (E4M3 codes uint8 [R, C], fp32 scales [R])."""
    x = _c(x, np.uint16)
    R, C = x.shape
    codes = np.empty((R, C), dtype=np.uint8)
    scales = np.empty((R,), dtype=np.float32)
    _check(lib().oracle_quantize_fp8_rows(_p(x, _u16p), R, C, C, _p(codes, _u8p), _p(scales, _f32p)),
           "oracle_quantize_fp8_rows")
    return codes, scales


def gemm_fp8(a, a_scale, w, w_scale):
    """fp32 [M, N] = a_scale[m] * w_scale[n] * sum_k e4m3(a[m,k]) * e4m3(w[n,k])."""
    a = _c(a, np.uint8)
    w = _c(w, np.uint8)
    a_scale = _c(np.asarray(a_scale, np.float32), np.float32)
    w_scale = _c(np.asarray(w_scale, np.float32), np.float32)
    M, K = a.shape
    N = w.shape[0]
    assert w.shape[1] == K
    out = np.empty((M, N), dtype=np.float32)
    _check(lib().oracle_gemm_fp8(_p(a, _u8p), _p(a_scale, _f32p), M, _p(w, _u8p), _p(w_scale, _f32p),
                                 N, K, _p(out, _f32p)), "oracle_gemm_fp8")
    return out


def f32_to_bf16_array(x):
    """bf16 rounding (ties to even) of a whole fp32 array, in C."""
    x = _c(np.asarray(x, np.float32), np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_n(_p(x, _f32p), x.size, _p(out, _u16p))
    return out


def fc_project_fp8(taps, fc_w8, fc_scale):
    """FP8 fc: the concatenated taps are quantised per row; h = bf16(gemm)."""
    x = np.concatenate([_c(t, np.uint16) for t in taps], axis=1)
    a8, a_s = quantize_fp8_rows(x)
    return f32_to_bf16_array(gemm_fp8(a8, a_s, fc_w8, fc_scale))


def lm_head_fp8(h, lm_w8, lm_scale):
    """FP8 LM head: h (bf16 bits [M, H]) quantised per row -> fp32 logits [M, V]."""
    a8, a_s = quantize_fp8_rows(h)
    return gemm_fp8(a8, a_s, lm_w8, lm_scale)
