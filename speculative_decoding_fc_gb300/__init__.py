"""GB300 (sm_103a) DSpark / DFlash speculative-decoding readout + verify.

Thin Python binding over ``libdspark.so`` (C ABI in ``include/dspark.h``).  This
module only checks tensors and marshals pointers; every step of the path runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or no sm_103 GPU is present, calls raise.

Functions follow the pages' notation:
  fc_project      concat(taps) . fc.weight^T -> h (bf16)
  lm_head         h . lm_head.weight^T -> fp32 logits for every block position
  greedy_sample   Markov-biased, semi-autoregressive argmax drafting (in place)
  draft_readout   lm_head + greedy_sample + optional confidence truncation
  verify          greedy exact match or probabilistic rejection sampling
  row_stats       (max, sum exp) and argmax of fp32 rows (target or draft logits)
  verify_from_stats  verify's decisions and draw from precomputed row statistics
"""
import ctypes
import os
import threading

import torch

__all__ = ["DSparkError", "lib", "fc_project", "lm_head", "greedy_sample", "confidence_truncate",
           "draft_readout", "confidence_truncate_markov", "quantize_fp8", "fc_project_fp8", "lm_head_fp8", "fc_lm_head",
           "verify", "row_stats", "verify_from_stats", "workspace_status", "launch_count",
           "Workspaces", "library_path", "linear", "embed_rmsnorm", "add_rmsnorm", "rmsnorm_bf16",
           "qk_norm_rope", "attention", "silu_mul", "BackboneLayer", "backbone_context", "backbone_block"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libdspark.so")
_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class DSparkError(RuntimeError):
    """A libdspark call returned a non-zero status."""


def library_path():
    return _LIB_PATH


def lib():
    """The loaded libdspark (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise DSparkError("libdspark.so is not built (%s); build it with "
                              "`python -m speculative_decoding_fc_gb300._build`" % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        L.dspark_status_string.restype = ctypes.c_char_p
        L.dspark_status_string.argtypes = [ctypes.c_int]
        L.dspark_version.restype = ctypes.c_int
        L.dspark_launch_count.restype = ctypes.c_longlong
        L.dspark_workspace_status.restype = ctypes.c_int
        L.dspark_workspace_status.argtypes = [_vp, _vp, ctypes.POINTER(_i32)]
        L.dspark_fc_project_workspace_size.restype = _sz
        L.dspark_fc_project_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_fc_project.restype = ctypes.c_int
        L.dspark_fc_project.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i64, _vp, _vp,
                                        ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_lm_head_workspace_size.restype = _sz
        L.dspark_lm_head_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_lm_head.restype = ctypes.c_int
        L.dspark_lm_head.argtypes = [_vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp,
                                     _sz, _vp]
        L.dspark_greedy_sample_workspace_size.restype = _sz
        L.dspark_greedy_sample_workspace_size.argtypes = [ctypes.c_int] * 4
        L.dspark_greedy_sample.restype = ctypes.c_int
        L.dspark_greedy_sample.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_confidence_truncate.restype = ctypes.c_int
        L.dspark_confidence_truncate.argtypes = [_vp, _vp, ctypes.c_float, ctypes.c_float, _vp, _vp,
                                                 _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp]
        L.dspark_confidence_truncate_markov.restype = ctypes.c_int
        L.dspark_confidence_truncate_markov.argtypes = [_vp, _vp, ctypes.c_float, ctypes.c_float,
                                                        ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int,
                                                        _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                                        ctypes.c_int, _vp, _vp]
        L.dspark_draft_readout_workspace_size.restype = _sz
        L.dspark_draft_readout_workspace_size.argtypes = [ctypes.c_int] * 5
        L.dspark_draft_readout.restype = ctypes.c_int
        L.dspark_draft_readout.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, ctypes.c_float,
                                           ctypes.c_float, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_verify_workspace_size.restype = _sz
        L.dspark_verify_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_verify.restype = ctypes.c_int
        L.dspark_verify.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_uint64, _vp,
                                    ctypes.c_uint32, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, _vp, _sz, _vp]
        L.dspark_row_stats_workspace_size.restype = _sz
        L.dspark_row_stats_workspace_size.argtypes = [_i64, ctypes.c_int]
        L.dspark_row_stats.restype = ctypes.c_int
        L.dspark_row_stats.argtypes = [_vp, _i64, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]
        L.dspark_verify_from_stats_workspace_size.restype = _sz
        L.dspark_verify_from_stats_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_verify_from_stats.restype = ctypes.c_int
        L.dspark_verify_from_stats.argtypes = [ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                               ctypes.c_uint64, _vp, ctypes.c_uint32, _vp, _vp,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_fc_lm_head_workspace_size.restype = _sz
        L.dspark_fc_lm_head_workspace_size.argtypes = [ctypes.c_int] * 4
        L.dspark_fc_lm_head.restype = ctypes.c_int
        L.dspark_fc_lm_head.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i64, _vp, _vp, _vp, _vp,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_quantize_fp8.restype = ctypes.c_int
        L.dspark_quantize_fp8.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i64, ctypes.c_int,
                                          ctypes.c_int, _vp, _vp, _vp]
        L.dspark_fc_project_fp8_workspace_size.restype = _sz
        L.dspark_fc_project_fp8_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_fc_project_fp8.restype = ctypes.c_int
        L.dspark_fc_project_fp8.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _i64, _vp, _vp, _vp,
                                            ctypes.c_int, ctypes.c_int, _vp, _sz, _vp]
        L.dspark_lm_head_fp8_workspace_size.restype = _sz
        L.dspark_lm_head_fp8_workspace_size.argtypes = [ctypes.c_int] * 3
        L.dspark_lm_head_fp8.restype = ctypes.c_int
        L.dspark_lm_head_fp8.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _vp, _sz, _vp]
        _c = ctypes.c_int
        L.dspark_linear_workspace_size.restype = _sz
        L.dspark_linear_workspace_size.argtypes = [_c] * 3
        L.dspark_linear.restype = _c
        L.dspark_linear.argtypes = [_vp, _i64, _vp, _vp, _i64, _c, _c, _c, _c, _vp, _sz, _vp]
        L.dspark_embed_rmsnorm.restype = _c
        L.dspark_embed_rmsnorm.argtypes = [_vp, _c, _vp, _vp, _vp, _vp, _c, _c, _vp, _vp]
        L.dspark_add_rmsnorm.restype = _c
        L.dspark_add_rmsnorm.argtypes = [_vp, _vp, _i64, _vp, _vp, _i64, _c, _c, _c, _vp]
        L.dspark_rmsnorm_bf16.restype = _c
        L.dspark_rmsnorm_bf16.argtypes = [_vp, _i64, _vp, _vp, _i64, _c, _c, _vp]
        L.dspark_qk_norm_rope.restype = _c
        L.dspark_qk_norm_rope.argtypes = [_vp, _i64, _c, _c, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                          _c, _c, _c, _c, _vp]
        L.dspark_block_context_rmsnorm.restype = _c
        L.dspark_block_context_rmsnorm.argtypes = [_vp, _vp, _i64, _vp, _c, _vp, _vp, _i64, _c, _vp, _vp, _i64,
                                                   _c, _c, _vp, _vp]
        L.dspark_qk_norm_rope_block_context.restype = _c
        L.dspark_qk_norm_rope_block_context.argtypes = [_vp, _i64, _c, _c, _vp, _vp, ctypes.c_float, _vp, _vp,
                                                        _vp, _c, _c, _c, _c, _vp, _i64, _c, _c, _vp]
        L.dspark_backbone_block_workspace_size.restype = _sz
        L.dspark_backbone_block_workspace_size.argtypes = [_c, _c, _c, _c, _vp, _c, _c]
        L.dspark_backbone_block.restype = _c
        L.dspark_backbone_block.argtypes = [_vp, _c, _c, _vp, _c, _c, _c, _vp, _vp, _c, _c, _vp, _c, _c, _vp, _vp,
                                            _sz, _vp]
        L.dspark_attention_workspace_size.restype = _sz
        L.dspark_attention_workspace_size.argtypes = [_c] * 5
        L.dspark_attention.restype = _c
        L.dspark_attention.argtypes = [_vp, _vp, _vp, _vp, _c, _c, _c, _c, _c, _c, _vp, _sz, _vp]
        L.dspark_silu_mul.restype = _c
        L.dspark_silu_mul.argtypes = [_vp, _vp, _c, _c, _vp]
        _lib = L
    return _lib


def _check(rc, what):
    if rc != 0:
        name = lib().dspark_status_string(rc).decode()
        raise DSparkError("%s failed: %s (%d)" % (what, name, rc))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise DSparkError("%s must be a CUDA tensor (no CPU path exists)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


class Workspaces:
    """Zero-initialised device workspaces, one per (call kind, device), grown on
    demand.  Calls that share a workspace must be ordered on the GPU (one stream,
    or events); pass a separate Workspaces object to run calls concurrently."""

    def __init__(self):
        self._bufs = {}

    def buffer(self, kind, device):
        """The workspace tensor of a call kind on a device (None before its first call);
        pass it to workspace_status() to read the device-side status word."""
        idx = torch.device(device).index
        if idx is None:
            idx = torch.cuda.current_device()
        return self._bufs.get((kind, idx))

    def get(self, kind, device, nbytes):
        key = (kind, torch.device(device).index)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
            self._bufs[key] = buf
        return buf


_default_ws = Workspaces()


def launch_count():
    """Kernels the library has enqueued in this process so far."""
    return int(lib().dspark_launch_count())


def workspace_status(ws, stream=None):
    """Reads and clears the device-side status word of a workspace tensor."""
    out = _i32(0)
    _check(lib().dspark_workspace_status(_ptr(ws), _stream(stream, ws.device), ctypes.byref(out)),
           "dspark_workspace_status")
    return int(out.value)


def fc_project(taps, fc_w, out=None, stream=None, workspaces=None):
    """h[M, H] (bf16) = concat(taps) . fc_w^T.  taps: T bf16 tensors [M, H] (row stride
    may exceed H); fc_w: [H, T*H] bf16."""
    T = len(taps)
    M, H = taps[0].shape
    dev = fc_w.device
    _need(fc_w, "fc_w", torch.bfloat16, (H, T * H))
    ld = taps[0].stride(0)
    for j, t in enumerate(taps):
        if not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (M, H) \
                or t.stride(1) != 1 or t.stride(0) != ld:
            raise ValueError("tap %d must be a CUDA bf16 [%d, %d] tensor with row stride %d" % (j, M, H, ld))
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (M, H))
    L = lib()
    nbytes = L.dspark_fc_project_workspace_size(M, H, T)
    ws = (workspaces or _default_ws).get("fc", dev, nbytes)
    arr = (_vp * T)(*[t.data_ptr() for t in taps])
    _check(L.dspark_fc_project(arr, T, ld, _ptr(fc_w), _ptr(out), M, H, _ptr(ws), ws.numel(),
                               _stream(stream, dev)), "dspark_fc_project")
    return out


def fc_lm_head(taps, fc_w, lm_w, h_out=None, logits=None, stream=None, workspaces=None):
    """fc projection and LM head in one launch: returns (h [M, H] bf16, fp32 logits
    [M, V]).  taps: T bf16 tensors [M, H] with a common row stride."""
    T = len(taps)
    M, H = taps[0].shape
    V = lm_w.shape[0]
    dev = fc_w.device
    _need(fc_w, "fc_w", torch.bfloat16, (H, T * H))
    _need(lm_w, "lm_w", torch.bfloat16, (V, H))
    ld = taps[0].stride(0)
    for j, t in enumerate(taps):
        if not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (M, H) \
                or t.stride(1) != 1 or t.stride(0) != ld:
            raise ValueError("tap %d must be a CUDA bf16 [%d, %d] tensor with row stride %d" % (j, M, H, ld))
    if h_out is None:
        h_out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    if logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    _need(h_out, "h_out", torch.bfloat16, (M, H))
    _need(logits, "logits", torch.float32)
    if logits.numel() != M * V:
        raise ValueError("logits must hold M*V floats")
    L = lib()
    ws = (workspaces or _default_ws).get("fclm", dev, L.dspark_fc_lm_head_workspace_size(M, H, T, V))
    arr = (_vp * T)(*[t.data_ptr() for t in taps])
    _check(L.dspark_fc_lm_head(arr, T, ld, _ptr(fc_w), _ptr(lm_w), _ptr(h_out), _ptr(logits), M, H,
                               V, _ptr(ws), ws.numel(), _stream(stream, dev)), "dspark_fc_lm_head")
    return h_out, logits


def lm_head(h, lm_w, out=None, stream=None, workspaces=None):
    """fp32 logits [M, V] = h . lm_w^T (h [M, H] bf16, lm_w [V, H] bf16)."""
    M, H = h.shape
    V = lm_w.shape[0]
    _need(h, "h", torch.bfloat16)
    _need(lm_w, "lm_w", torch.bfloat16, (V, H))
    if out is None:
        out = torch.empty((M, V), dtype=torch.float32, device=h.device)
    _need(out, "out", torch.float32)
    if out.numel() != M * V:
        raise ValueError("out must hold M*V floats")
    L = lib()
    ws = (workspaces or _default_ws).get("lm", h.device, L.dspark_lm_head_workspace_size(M, H, V))
    _check(L.dspark_lm_head(_ptr(h), _ptr(lm_w), _ptr(out), M, H, V, _ptr(ws), ws.numel(),
                            _stream(stream, h.device)), "dspark_lm_head")
    return out


def greedy_sample(logits, w1, w2, prev_token, draft_tokens=None, q_stats=None, stream=None,
                  workspaces=None, want_q_stats=True):
    """Markov-biased greedy drafting.  logits fp32 [B, k, V] is biased in place; returns
    (draft_tokens int32 [B, k], q_stats fp32 [B, k, 2]).  want_q_stats=False passes no
    q_stats buffer (the kernel then reduces only the argmax) and returns None for it."""
    B, k, V = logits.shape
    _need(logits, "logits", torch.float32)
    r = 0
    if w1 is not None:
        r = w1.shape[1]
        _need(w1, "w1", torch.bfloat16, (V, r))
        _need(w2, "w2", torch.bfloat16, (V, r))
    _need(prev_token, "prev_token", torch.int32, (B,))
    dev = logits.device
    if draft_tokens is None:
        draft_tokens = torch.empty((B, k), dtype=torch.int32, device=dev)
    if not want_q_stats:
        q_stats = None
    elif q_stats is None:
        q_stats = torch.empty((B, k, 2), dtype=torch.float32, device=dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if q_stats is not None:
        _need(q_stats, "q_stats", torch.float32, (B, k, 2))
    L = lib()
    ws = (workspaces or _default_ws).get("chain", dev, L.dspark_greedy_sample_workspace_size(B, k, V, r))
    _check(L.dspark_greedy_sample(_ptr(logits), _ptr(w1), _ptr(w2), r, _ptr(prev_token),
                                  _ptr(draft_tokens), _ptr(q_stats), B, k, V, _ptr(ws), ws.numel(),
                                  _stream(stream, dev)), "dspark_greedy_sample")
    return draft_tokens, q_stats


def confidence_truncate(h, conf_w, draft_tokens, B, k, conf_b=0.0, conf_tau=0.5, draft_len=None,
                        conf_out=None, stream=None):
    """Confidence head + adaptive truncation: c = sigmoid(conf_w . h + conf_b) per block
    position; draft_len[b] = first position with c < conf_tau; later drafts become -1 (in
    place).  Returns (draft_len int32 [B], conf fp32 [B, k] or None)."""
    M, H = h.shape
    if M != B * k:
        raise ValueError("h must have B*k rows")
    _need(h, "h", torch.bfloat16)
    _need(conf_w, "conf_w", torch.bfloat16, (H,))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if draft_len is None:
        draft_len = torch.empty((B,), dtype=torch.int32, device=h.device)
    _need(draft_len, "draft_len", torch.int32, (B,))
    if conf_out is not None:
        _need(conf_out, "conf_out", torch.float32, (B, k))
    _check(lib().dspark_confidence_truncate(_ptr(h), _ptr(conf_w), float(conf_b), float(conf_tau),
                                            _ptr(draft_tokens), _ptr(draft_len), _ptr(conf_out), B,
                                            k, H, _stream(stream, h.device)),
           "dspark_confidence_truncate")
    return draft_len, conf_out


def confidence_truncate_markov(h, conf_w, draft_tokens, B, k, conf_b=0.0, conf_tau=0.5,
                               cumulative=False, w1=None, prev_token=None, draft_len=None,
                               conf_out=None, status=None, stream=None):
    """Confidence head over [h ; markov_w1[context]] (w1 given: conf_w has H + r entries)
    or over h alone, with the per-position or the cumulative (product of confidences)
    truncation rule.  Returns (draft_len int32 [B], conf fp32 [B, k] or None)."""
    M, H = h.shape
    if M != B * k:
        raise ValueError("h must have B*k rows")
    _need(h, "h", torch.bfloat16)
    r, V = 0, 0
    if w1 is not None:
        V, r = w1.shape
        _need(w1, "w1", torch.bfloat16, (V, r))
        _need(prev_token, "prev_token", torch.int32, (B,))
    _need(conf_w, "conf_w", torch.bfloat16, (H + r,))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if draft_len is None:
        draft_len = torch.empty((B,), dtype=torch.int32, device=h.device)
    _need(draft_len, "draft_len", torch.int32, (B,))
    if conf_out is not None:
        _need(conf_out, "conf_out", torch.float32, (B, k))
    if status is not None:
        _need(status, "status", torch.int32, (1,))
    _check(lib().dspark_confidence_truncate_markov(
        _ptr(h), _ptr(conf_w), float(conf_b), float(conf_tau), int(bool(cumulative)), _ptr(w1), r, V,
        _ptr(prev_token), _ptr(draft_tokens), _ptr(draft_len), _ptr(conf_out), B, k, H,
        _ptr(status), _stream(stream, h.device)), "dspark_confidence_truncate_markov")
    return draft_len, conf_out


def draft_readout(h, lm_w, w1, w2, prev_token, B, k, conf_w=None, conf_b=0.0, conf_tau=0.5,
                  out=None, stream=None, workspaces=None):
    """LM head + Markov greedy drafting + optional confidence truncation.

    h: [B*k, H] bf16.  Returns a dict with logits (biased, fp32 [B, k, V]), q_stats,
    draft_tokens (-1 past the truncation point), draft_len, conf (or None)."""
    M, H = h.shape
    if M != B * k:
        raise ValueError("h must have B*k rows")
    V = lm_w.shape[0]
    dev = h.device
    _need(h, "h", torch.bfloat16)
    _need(lm_w, "lm_w", torch.bfloat16, (V, H))
    r = 0
    if w1 is not None:
        r = w1.shape[1]
        _need(w1, "w1", torch.bfloat16, (V, r))
        _need(w2, "w2", torch.bfloat16, (V, r))
    _need(prev_token, "prev_token", torch.int32, (B,))
    if conf_w is not None:
        _need(conf_w, "conf_w", torch.bfloat16, (H,))
    o = out if out is not None else {}
    logits = o.get("logits")
    if logits is None:
        logits = torch.empty((B, k, V), dtype=torch.float32, device=dev)
    q_stats = o.get("q_stats")
    if q_stats is None:
        q_stats = torch.empty((B, k, 2), dtype=torch.float32, device=dev)
    drafts = o.get("draft_tokens")
    if drafts is None:
        drafts = torch.empty((B, k), dtype=torch.int32, device=dev)
    dlen = o.get("draft_len")
    if dlen is None:
        dlen = torch.empty((B,), dtype=torch.int32, device=dev)
    conf = o.get("conf")
    if conf is None and conf_w is not None:
        conf = torch.empty((B, k), dtype=torch.float32, device=dev)
    _need(logits, "logits", torch.float32, (B, k, V))
    _need(q_stats, "q_stats", torch.float32, (B, k, 2))
    _need(drafts, "draft_tokens", torch.int32, (B, k))
    _need(dlen, "draft_len", torch.int32, (B,))
    L = lib()
    ws = (workspaces or _default_ws).get("readout", dev,
                                         L.dspark_draft_readout_workspace_size(B, k, H, V, r))
    _check(L.dspark_draft_readout(_ptr(h), _ptr(lm_w), _ptr(w1), _ptr(w2), r, _ptr(prev_token),
                                  _ptr(conf_w), float(conf_b), float(conf_tau), _ptr(logits),
                                  _ptr(q_stats), _ptr(drafts), _ptr(dlen), _ptr(conf), B, k, H, V,
                                  _ptr(ws), ws.numel(), _stream(stream, dev)), "dspark_draft_readout")
    return {"logits": logits, "q_stats": q_stats, "draft_tokens": drafts, "draft_len": dlen,
            "conf": conf}


def verify(mode, target_logits, draft_tokens, draft_len=None, draft_logits=None, q_stats=None,
           seed=0, request_id=None, step=0, accepted_len=None, next_token=None, stream=None,
           workspaces=None):
    """Verify one draft block per request.  mode 0 greedy, 1 probabilistic.
    target_logits fp32 [B, k+1, V]; returns (accepted_len int32 [B], next_token int32 [B])."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    _need(target_logits, "target_logits", torch.float32)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if draft_len is not None:
        _need(draft_len, "draft_len", torch.int32, (B,))
    if draft_logits is not None:
        _need(draft_logits, "draft_logits", torch.float32, (B, k, V))
    if q_stats is not None:
        _need(q_stats, "q_stats", torch.float32, (B, k, 2))
    if request_id is not None:
        if request_id.dtype not in (torch.int32, torch.uint32):
            raise TypeError("request_id must be int32/uint32")
        if not request_id.is_cuda or not request_id.is_contiguous() or tuple(request_id.shape) != (B,):
            raise ValueError("request_id must be a contiguous CUDA [B] tensor")
    if accepted_len is None:
        accepted_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(accepted_len, "accepted_len", torch.int32, (B,))
    _need(next_token, "next_token", torch.int32, (B,))
    L = lib()
    ws = (workspaces or _default_ws).get("verify", dev, L.dspark_verify_workspace_size(B, k, V))
    _check(L.dspark_verify(int(mode), _ptr(target_logits), _ptr(draft_tokens), _ptr(draft_len),
                           _ptr(draft_logits), _ptr(q_stats), int(seed) & (2 ** 64 - 1),
                           _ptr(request_id), int(step) & 0xFFFFFFFF, _ptr(accepted_len),
                           _ptr(next_token), B, k, V, _ptr(ws), ws.numel(), _stream(stream, dev)),
           "dspark_verify")
    return accepted_len, next_token


def _request_ids(request_id, B):
    if request_id is not None:
        if request_id.dtype not in (torch.int32, torch.uint32):
            raise TypeError("request_id must be int32/uint32")
        if not request_id.is_cuda or not request_id.is_contiguous() or tuple(request_id.shape) != (B,):
            raise ValueError("request_id must be a contiguous CUDA [B] tensor")


def row_stats(rows, ms=None, argmax=None, want_ms=True, want_argmax=True, stream=None,
              workspaces=None):
    """Softmax statistics and argmax of every row of an fp32 tensor [..., V]:
    returns (ms fp32 [..., 2] = (max, sum exp(x - max)) or None, argmax int32 [...] or None)."""
    _need(rows, "rows", torch.float32)
    V = rows.shape[-1]
    lead = tuple(rows.shape[:-1])
    n = rows.numel() // V
    dev = rows.device
    if want_ms and ms is None:
        ms = torch.empty(lead + (2,), dtype=torch.float32, device=dev)
    if want_argmax and argmax is None:
        argmax = torch.empty(lead, dtype=torch.int32, device=dev)
    if ms is not None:
        _need(ms, "ms", torch.float32, lead + (2,))
    if argmax is not None:
        _need(argmax, "argmax", torch.int32, lead)
    L = lib()
    ws = (workspaces or _default_ws).get("rows", dev, L.dspark_row_stats_workspace_size(n, V))
    _check(L.dspark_row_stats(_ptr(rows), n, V, _ptr(ms), _ptr(argmax), _ptr(ws), ws.numel(),
                              _stream(stream, dev)), "dspark_row_stats")
    return ms, argmax


def verify_from_stats(mode, target_logits, target_ms, target_argmax, draft_tokens, draft_len=None,
                      draft_logits=None, q_stats=None, seed=0, request_id=None, step=0,
                      accepted_len=None, next_token=None, stream=None, workspaces=None):
    """verify() with the target rows' statistics already computed (row_stats of the target
    logits): one kernel.  Returns (accepted_len int32 [B], next_token int32 [B])."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    _need(target_logits, "target_logits", torch.float32)
    if target_ms is not None:
        _need(target_ms, "target_ms", torch.float32, (B, k1, 2))
    if target_argmax is not None:
        _need(target_argmax, "target_argmax", torch.int32, (B, k1))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if draft_len is not None:
        _need(draft_len, "draft_len", torch.int32, (B,))
    if draft_logits is not None:
        _need(draft_logits, "draft_logits", torch.float32, (B, k, V))
    if q_stats is not None:
        _need(q_stats, "q_stats", torch.float32, (B, k, 2))
    _request_ids(request_id, B)
    if accepted_len is None:
        accepted_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(accepted_len, "accepted_len", torch.int32, (B,))
    _need(next_token, "next_token", torch.int32, (B,))
    L = lib()
    ws = (workspaces or _default_ws).get("verify_fs", dev,
                                         L.dspark_verify_from_stats_workspace_size(B, k, V))
    _check(L.dspark_verify_from_stats(int(mode), _ptr(target_logits), _ptr(target_ms),
                                      _ptr(target_argmax), _ptr(draft_tokens), _ptr(draft_len),
                                      _ptr(draft_logits), _ptr(q_stats), int(seed) & (2 ** 64 - 1),
                                      _ptr(request_id), int(step) & 0xFFFFFFFF, _ptr(accepted_len),
                                      _ptr(next_token), B, k, V, _ptr(ws), ws.numel(),
                                      _stream(stream, dev)), "dspark_verify_from_stats")
    return accepted_len, next_token


# ---------------------------------------------------------------- FP8 (E4M3) weights
def _segments(segs, name):
    rows, cols = segs[0].shape
    ld = segs[0].stride(0)
    for j, t in enumerate(segs):
        if not t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != (rows, cols) \
                or t.stride(1) != 1 or t.stride(0) != ld:
            raise ValueError("%s %d must be a CUDA bf16 [%d, %d] tensor with row stride %d"
                             % (name, j, rows, cols, ld))
    return rows, cols, ld


def quantize_fp8(x, codes=None, scales=None, stream=None):
    """Per-row E4M3 quantisation of a bf16 matrix (or a list of column segments of
    one): returns (codes uint8 [R, C], scales fp32 [R])."""
    segs = list(x) if isinstance(x, (list, tuple)) else [x]
    R, C, ld = _segments(segs, "segment")
    dev = segs[0].device
    if codes is None:
        codes = torch.empty((R, C * len(segs)), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((R,), dtype=torch.float32, device=dev)
    _need(codes, "codes", torch.uint8, (R, C * len(segs)))
    _need(scales, "scales", torch.float32, (R,))
    arr = (_vp * len(segs))(*[t.data_ptr() for t in segs])
    _check(lib().dspark_quantize_fp8(arr, len(segs), ld, R, C, _ptr(codes), _ptr(scales),
                                     _stream(stream, dev)), "dspark_quantize_fp8")
    return codes, scales


def fc_project_fp8(taps, fc_w8, fc_scale, out=None, stream=None, workspaces=None):
    """FP8 fc: h[M, H] (bf16) from bf16 taps (quantised per row on the fly) and the
    E4M3 weight fc_w8 [H, T*H] with per-row scales fc_scale [H]."""
    T = len(taps)
    M, H, ld = _segments(taps, "tap")
    dev = fc_w8.device
    _need(fc_w8, "fc_w8", torch.uint8, (H, T * H))
    _need(fc_scale, "fc_scale", torch.float32, (H,))
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (M, H))
    L = lib()
    ws = (workspaces or _default_ws).get("fc8", dev, L.dspark_fc_project_fp8_workspace_size(M, H, T))
    arr = (_vp * T)(*[t.data_ptr() for t in taps])
    _check(L.dspark_fc_project_fp8(arr, T, ld, _ptr(fc_w8), _ptr(fc_scale), _ptr(out), M, H,
                                   _ptr(ws), ws.numel(), _stream(stream, dev)),
           "dspark_fc_project_fp8")
    return out


def lm_head_fp8(h, lm_w8, lm_scale, out=None, stream=None, workspaces=None):
    """FP8 LM head: fp32 logits [M, V] from h [M, H] bf16 (quantised per row on the fly)
    and the E4M3 weight lm_w8 [V, H] with per-row scales lm_scale [V]."""
    M, H = h.shape
    V = lm_w8.shape[0]
    _need(h, "h", torch.bfloat16)
    _need(lm_w8, "lm_w8", torch.uint8, (V, H))
    _need(lm_scale, "lm_scale", torch.float32, (V,))
    if out is None:
        out = torch.empty((M, V), dtype=torch.float32, device=h.device)
    _need(out, "out", torch.float32)
    if out.numel() != M * V:
        raise ValueError("out must hold M*V floats")
    L = lib()
    ws = (workspaces or _default_ws).get("lm8", h.device, L.dspark_lm_head_fp8_workspace_size(M, H, V))
    _check(L.dspark_lm_head_fp8(_ptr(h), _ptr(lm_w8), _ptr(lm_scale), _ptr(out), M, H, V,
                                _ptr(ws), ws.numel(), _stream(stream, h.device)),
           "dspark_lm_head_fp8")
    return out


# ----------------------------------------------------------------------------- backbone
def linear(x, w, out=None, out_bf16=True, stream=None, workspaces=None, kind="linear"):
    """out[M, N] = x[M, K] . w[N, K]^T (bf16 in, fp32 accumulate; bf16 or fp32 out).
    `kind` names the workspace (calls of different shapes keep separate ones)."""
    M, K = x.shape
    N = w.shape[0]
    dev = w.device
    _need(w, "w", torch.bfloat16, (N, K))
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.stride(1) != 1:
        raise ValueError("x must be a CUDA bf16 [M, K] tensor with unit column stride")
    odt = torch.bfloat16 if out_bf16 else torch.float32
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=dev)
    if out.dtype != odt or tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be %s [%d, %d] with unit column stride" % (odt, M, N))
    L = lib()
    ws = (workspaces or _default_ws).get(kind, dev, L.dspark_linear_workspace_size(M, N, K))
    _check(L.dspark_linear(_ptr(x), x.stride(0), _ptr(w), _ptr(out), out.stride(0), 1 if out_bf16 else 0,
                           M, N, K, _ptr(ws), ws.numel(), _stream(stream, dev)), "dspark_linear")
    return out


def embed_rmsnorm(table, tokens, w, x_out=None, n_out=None, status=None, stream=None):
    """x_out = table[tokens] (fp32 [rows, H]); n_out = bf16(rmsnorm(x_out) * w)."""
    V, H = table.shape
    rows = tokens.numel()
    dev = table.device
    _need(table, "table", torch.bfloat16)
    _need(tokens, "tokens", torch.int32)
    _need(w, "w", torch.bfloat16, (H,))
    if x_out is None:
        x_out = torch.empty((rows, H), dtype=torch.float32, device=dev)
    if n_out is None:
        n_out = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    _need(x_out, "x_out", torch.float32, (rows, H))
    _need(n_out, "n_out", torch.bfloat16, (rows, H))
    _check(lib().dspark_embed_rmsnorm(_ptr(table), V, _ptr(tokens), _ptr(w), _ptr(x_out), _ptr(n_out), rows, H,
                                      _ptr(status), _stream(stream, dev)), "dspark_embed_rmsnorm")
    return x_out, n_out


def add_rmsnorm(x, delta, w, out=None, group=0, stream=None):
    """x += delta (fp32 add of bf16, delta may be None); out = bf16(rmsnorm(x) * w).
    group > 0: the first row of every group is not written, the others compacted."""
    rows, H = x.shape
    dev = x.device
    _need(x, "x", torch.float32)
    _need(w, "w", torch.bfloat16, (H,))
    if delta is not None:
        _need(delta, "delta", torch.bfloat16, (rows, H))
    orows = rows if group == 0 else rows // group * (group - 1)
    if out is None:
        out = torch.empty((orows, H), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (orows, H))
    _check(lib().dspark_add_rmsnorm(_ptr(x), _ptr(delta), H, _ptr(w), _ptr(out), H, group, rows, H,
                                    _stream(stream, dev)), "dspark_add_rmsnorm")
    return out


def rmsnorm_bf16(inp, w, out=None, stream=None):
    """out = bf16(rmsnorm(inp) * w) of bf16 rows [rows, H]."""
    rows, H = inp.shape
    dev = inp.device
    _need(inp, "inp", torch.bfloat16)
    _need(w, "w", torch.bfloat16, (H,))
    if out is None:
        out = torch.empty_like(inp)
    _need(out, "out", torch.bfloat16, (rows, H))
    _check(lib().dspark_rmsnorm_bf16(_ptr(inp), H, _ptr(w), _ptr(out), H, rows, H, _stream(stream, dev)),
           "dspark_rmsnorm_bf16")
    return out


def block_context_rmsnorm(x, w, out, ctx=None, table=None, tokens=None, delta=None, status=None, stream=None):
    """One launch for the block rows' and the new context rows' input norms: x [rows, H]
    fp32 is set to table[tokens] (table given) or gets delta added (delta given, else
    left); out[:rows] = bf16(rmsnorm(x) * w); out[rows:] = bf16(rmsnorm(ctx) * w) of the
    bf16 context rows ctx [n, H] (optional).  out: bf16 [rows + n, H]."""
    rows, H = x.shape
    dev = x.device
    n = 0 if ctx is None else ctx.shape[0]
    _need(x, "x", torch.float32)
    _need(w, "w", torch.bfloat16, (H,))
    _need(out, "out", torch.bfloat16, (rows + n, H))
    V = 0
    if table is not None:
        V = table.shape[0]
        _need(table, "table", torch.bfloat16, (V, H))
        _need(tokens, "tokens", torch.int32)
        if tokens.numel() != rows:
            raise ValueError("tokens must hold one id per block row")
    if delta is not None:
        _need(delta, "delta", torch.bfloat16, (rows, H))
    if n:
        _need(ctx, "ctx", torch.bfloat16, (n, H))
    _check(lib().dspark_block_context_rmsnorm(_ptr(x), _ptr(delta), H, _ptr(table), V, _ptr(tokens), _ptr(ctx), H,
                                              n, _ptr(w), _ptr(out), H, rows, H, _ptr(status),
                                              _stream(stream, dev)), "dspark_block_context_rmsnorm")
    return out


def qk_norm_rope_block_context(qkv, nq, nkv, q_norm_w, k_norm_w, theta, k_cache, v_cache, rows_per_req, pos0,
                               ctx_kv, ctx_rows_per_req, ctx_pos0, q_out=None, stream=None):
    """qk_norm_rope of the block rows qkv [B * rows_per_req, (nq + 2 nkv) * 128] and of the
    context rows ctx_kv [B * ctx_rows_per_req, 2 nkv * 128] (key and value heads, cache
    slots ctx_pos0 + j) in one launch; both may be column slices of a wider GEMM output.
    Returns q [B * rows_per_req, nq, 128]."""
    rows = qkv.shape[0]
    B, cache_len = k_cache.shape[0], k_cache.shape[1]
    dev = qkv.device
    for t, width, name in ((qkv, (nq + 2 * nkv) * 128, "qkv"), (ctx_kv, 2 * nkv * 128, "ctx_kv")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 \
                or t.dim() != 2 or t.shape[1] != width or t.stride(1) != 1:
            raise ValueError("%s must be a CUDA bf16 [rows, %d] tensor with unit column stride" % (name, width))
    _need(k_norm_w, "k_norm_w", torch.bfloat16, (128,))
    _need(q_norm_w, "q_norm_w", torch.bfloat16, (128,))
    _need(k_cache, "k_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    _need(v_cache, "v_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    if rows != B * rows_per_req or ctx_kv.shape[0] != B * ctx_rows_per_req:
        raise ValueError("qkv and ctx_kv must hold B * rows_per_req and B * ctx_rows_per_req rows")
    if q_out is None:
        q_out = torch.empty((rows, nq, 128), dtype=torch.bfloat16, device=dev)
    _need(q_out, "q_out", torch.bfloat16, (rows, nq, 128))
    _check(lib().dspark_qk_norm_rope_block_context(
        _ptr(qkv), qkv.stride(0), nq, nkv, _ptr(q_norm_w), _ptr(k_norm_w), float(theta), _ptr(q_out), _ptr(k_cache),
        _ptr(v_cache), B, cache_len, rows_per_req, pos0, _ptr(ctx_kv), ctx_kv.stride(0), ctx_rows_per_req, ctx_pos0,
        _stream(stream, dev)), "dspark_qk_norm_rope_block_context")
    return q_out


def qk_norm_rope(qkv, nq, nkv, q_norm_w, k_norm_w, theta, k_cache, v_cache, rows_per_req, pos0,
                 q_out=None, stream=None):
    """Per-head q/k rmsnorm + rotary embedding of qkv rows [B * rows_per_req, (nq + 2 nkv) * 128]
    (nq = 0: key/value rows only); k and v go to cache slots pos0 .. pos0 + rows_per_req - 1
    of each request; returns q [rows, nq, 128] (None when nq == 0)."""
    rows = qkv.shape[0]
    B, cache_len = k_cache.shape[0], k_cache.shape[1]
    dev = qkv.device
    # qkv may be a column slice of a wider GEMM output (row stride > its width)
    if not isinstance(qkv, torch.Tensor) or not qkv.is_cuda or qkv.dtype != torch.bfloat16 \
            or tuple(qkv.shape) != (rows, (nq + 2 * nkv) * 128) or qkv.stride(1) != 1:
        raise ValueError("qkv must be a CUDA bf16 [rows, (nq + 2 nkv) * 128] tensor with unit column stride")
    _need(k_norm_w, "k_norm_w", torch.bfloat16, (128,))
    _need(k_cache, "k_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    _need(v_cache, "v_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    if rows != B * rows_per_req:
        raise ValueError("qkv has %d rows, expected B * rows_per_req = %d" % (rows, B * rows_per_req))
    if nq > 0:
        _need(q_norm_w, "q_norm_w", torch.bfloat16, (128,))
        if q_out is None:
            q_out = torch.empty((rows, nq, 128), dtype=torch.bfloat16, device=dev)
        _need(q_out, "q_out", torch.bfloat16, (rows, nq, 128))
    _check(lib().dspark_qk_norm_rope(_ptr(qkv), qkv.stride(0), nq, nkv, _ptr(q_norm_w if nq > 0 else None),
                                     _ptr(k_norm_w), float(theta), _ptr(q_out if nq > 0 else None),
                                     _ptr(k_cache), _ptr(v_cache), B, cache_len, rows_per_req, pos0,
                                     _stream(stream, dev)), "dspark_qk_norm_rope")
    return q_out if nq > 0 else None


def attention(q, k_cache, v_cache, nkeys, out=None, stream=None, workspaces=None):
    """Grouped-query attention of q [B, nr, nq, 128] over cache keys 0 .. nkeys - 1
    (k_cache, v_cache [B, cache_len, nkv, 128]); returns out [B, nr, nq, 128] bf16."""
    B, nr, nq, hd = q.shape
    cache_len, nkv = k_cache.shape[1], k_cache.shape[2]
    dev = q.device
    _need(q, "q", torch.bfloat16, (B, nr, nq, 128))
    _need(k_cache, "k_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    _need(v_cache, "v_cache", torch.bfloat16, (B, cache_len, nkv, 128))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (B, nr, nq, 128))
    L = lib()
    ws = (workspaces or _default_ws).get("attention", dev,
                                        L.dspark_attention_workspace_size(B, nr, nq, nkv, nkeys))
    _check(L.dspark_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), B, nr, nq, nkv, cache_len, nkeys,
                              _ptr(ws), ws.numel(), _stream(stream, dev)), "dspark_attention")
    return out


def silu_mul(gu, out=None, stream=None):
    """act[M, I] = bf16(silu(gu[:, :I]) * gu[:, I:]) of the gate|up GEMM output gu [M, 2I]."""
    M, I2 = gu.shape
    dev = gu.device
    _need(gu, "gu", torch.bfloat16)
    if out is None:
        out = torch.empty((M, I2 // 2), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (M, I2 // 2))
    _check(lib().dspark_silu_mul(_ptr(gu), _ptr(out), M, I2 // 2, _stream(stream, dev)), "dspark_silu_mul")
    return out


class BackboneLayer:
    """One decoder layer's device weights (bf16): w_in, w_post [H]; w_qn, w_kn [128];
    w_qkv [(nq + 2 nkv) * 128, H]; w_o [H, nq * 128]; w_gu [2I, H]; w_d [H, I]."""

    def __init__(self, nq, nkv, w_in, w_post, w_qn, w_kn, w_qkv, w_o, w_gu, w_d, theta=1e6):
        self.nq, self.nkv, self.theta = nq, nkv, theta
        self.w_in, self.w_post, self.w_qn, self.w_kn = w_in, w_post, w_qn, w_kn
        self.w_qkv, self.w_o, self.w_gu, self.w_d = w_qkv, w_o, w_gu, w_d

    @property
    def w_kv(self):
        """The [Wk; Wv] rows of w_qkv (a view)."""
        return self.w_qkv[self.nq * 128:]


def backbone_context(ctx, layers, k_caches, v_caches, pos0, stream=None, workspaces=None):
    """Writes the keys and values of context rows ctx [B * n, H] (bf16, the fc output of
    n verified tokens per request) into each layer's caches at slots pos0 .. pos0 + n - 1:
    input norm, the [Wk; Wv] GEMM, k-norm + rotary."""
    rows = ctx.shape[0]
    B = k_caches[0].shape[0]
    n = rows // B
    for li, (ly, kc, vc) in enumerate(zip(layers, k_caches, v_caches)):
        nrm = rmsnorm_bf16(ctx, ly.w_in, stream=stream)
        kv = linear(nrm, ly.w_kv, stream=stream, workspaces=workspaces, kind="bb_kv%d" % li)
        qk_norm_rope(kv, 0, ly.nkv, None, ly.w_kn, ly.theta, kc, vc, n, pos0, stream=stream)


class _BackboneLayerC(ctypes.Structure):
    """dspark_backbone_layer_t."""
    _fields_ = [("w_in", _vp), ("w_post", _vp), ("w_qn", _vp), ("w_kn", _vp), ("w_qkv", _vp), ("w_o", _vp),
                ("w_gu", _vp), ("w_d", _vp), ("k_cache", _vp), ("v_cache", _vp), ("nq", ctypes.c_int),
                ("nkv", ctypes.c_int), ("I", ctypes.c_int), ("theta", ctypes.c_float)]


def backbone_block(tokens, embed, layers, w_final, k_caches, v_caches, C, out=None, stream=None,
                   workspaces=None, ctx=None, ctx_pos0=None):
    """Runs the draft block through the layers and the final norm (dspark_backbone_block:
    one call).  tokens [B, k+1] int32 (anchor, then mask tokens); embed [V, H] bf16 (the
    LM head's weight); the caches hold each layer's context keys/values at slots 0 .. C - 1,
    the block's go to C .. C + k.  Returns h [B * k, H] bf16 (mask positions), the LM head's
    input.  ctx [B * n, H] (optional): n new context rows per request (the fc output of the
    verified tokens), written to cache slots ctx_pos0 .. ctx_pos0 + n - 1 of every layer
    before its attention; their keys and values come out of the same GEMM as the block's
    q, k, v (one pass over each layer's [Wq; Wk; Wv])."""
    B, nr = tokens.shape
    V, H = embed.shape
    dev = embed.device
    _need(tokens, "tokens", torch.int32, (B, nr))
    _need(embed, "embed", torch.bfloat16, (V, H))
    _need(w_final, "w_final", torch.bfloat16, (H,))
    if len(layers) != len(k_caches) or len(layers) != len(v_caches) or not layers:
        raise ValueError("one key and one value cache per layer")
    cache_len = k_caches[0].shape[1]
    arr = (_BackboneLayerC * len(layers))()
    for i, (ly, kc, vc) in enumerate(zip(layers, k_caches, v_caches)):
        _need(kc, "k_cache", torch.bfloat16, (B, cache_len, ly.nkv, 128))
        _need(vc, "v_cache", torch.bfloat16, (B, cache_len, ly.nkv, 128))
        I = ly.w_d.shape[1]
        for t, nm, shape in ((ly.w_in, "w_in", (H,)), (ly.w_post, "w_post", (H,)), (ly.w_qn, "w_qn", (128,)),
                             (ly.w_kn, "w_kn", (128,)), (ly.w_qkv, "w_qkv", ((ly.nq + 2 * ly.nkv) * 128, H)),
                             (ly.w_o, "w_o", (H, ly.nq * 128)), (ly.w_gu, "w_gu", (2 * I, H)),
                             (ly.w_d, "w_d", (H, I))):
            _need(t, nm, torch.bfloat16, shape)
        arr[i] = _BackboneLayerC(ly.w_in.data_ptr(), ly.w_post.data_ptr(), ly.w_qn.data_ptr(), ly.w_kn.data_ptr(),
                                 ly.w_qkv.data_ptr(), ly.w_o.data_ptr(), ly.w_gu.data_ptr(), ly.w_d.data_ptr(),
                                 kc.data_ptr(), vc.data_ptr(), ly.nq, ly.nkv, I, float(ly.theta))
    n = 0
    if ctx is not None:
        _need(ctx, "ctx", torch.bfloat16)
        if ctx.shape[0] % B != 0 or ctx.shape[1] != H:
            raise ValueError("ctx must be [B * n, H]")
        n = ctx.shape[0] // B
    if out is None:
        out = torch.empty((B * (nr - 1), H), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B * (nr - 1), H))
    L = lib()
    parr = ctypes.cast(arr, ctypes.c_void_p)
    nbytes = L.dspark_backbone_block_workspace_size(B, nr, H, len(layers), parr, n, C)
    if nbytes == 0:
        raise DSparkError("dspark_backbone_block: unsupported shape")
    ws = (workspaces or _default_ws).get("backbone", dev, nbytes)
    _check(L.dspark_backbone_block(_ptr(tokens), B, nr, _ptr(embed), V, H, len(layers), parr, _ptr(w_final),
                                   cache_len, C, _ptr(ctx), n, int(ctx_pos0 or 0), _ptr(out), _ptr(ws), ws.numel(),
                                   _stream(stream, dev)), "dspark_backbone_block")
    return out

