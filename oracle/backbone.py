"""Oracle of the drafter backbone (test infrastructure only: tests, the smoke check and
the benchmark's CPU baseline use it; the product path never does).

Plain numpy in float64, with a bf16 rounding (ties to even) wherever the step stores
a bf16 tensor, so that a result can be compared with the GPU's up to the order of its
fp32 sums.  The pages name the drafter class (a DFlash Qwen3 model: "DSparkDraftModel
(DFlashQwen3ForCausalLM)"; "Qwen3DSparkModel selects the Qwen3 implementation") and
its config fields (`layer_types`, `head_dim`, `mask_token_id`, `projector_type`)
without values or a forward pass; the readings taken here are listed with the
functions (and in the design notes, reading R13):

* Decoder layer of the Qwen3 form, pre-norm:
    n   = bf16(rmsnorm(x) * w_in)
    q, k, v = bf16(n Wq^T), bf16(n Wk^T), bf16(n Wv^T)       (one GEMM over [Wq; Wk; Wv])
    q_h = bf16(rope(rmsnorm(q_h) * w_qn)), k_h = bf16(rope(rmsnorm(k_h) * w_kn))   per head
    o   = bf16(attention(q, [K_ctx; k], [V_ctx; v]))          (grouped-query heads)
    x  += bf16(o Wo^T)
    n2  = bf16(rmsnorm(x) * w_post)
    g, u = bf16(n2 Wg^T), bf16(n2 Wu^T)                      (one GEMM over [Wg; Wu])
    x  += bf16(bf16(silu(g) * u) Wd^T)
  rmsnorm(x) = x / sqrt(mean(x^2) + 1e-6); the residual x is kept in fp32.
* Rotary embedding of the NeoX form: dims (d, d + hd/2), angle pos * theta^(-2d/hd),
  theta = 1e6.
* The block: position 0 is the anchor (the bonus token), positions 1..k the mask
  token; their inputs are rows of the LM head's weight (tied embeddings).
* Context: the fc output of each verified token; a layer's context keys and values
  are that row through the layer's input norm and Wk, Wv (k-norm and rotary at the
  token's position).  Context token j sits at position j, block position i at C + i;
  every block query attends to all C context keys and all k + 1 block keys (no mask
  inside the block).
* Output: h = bf16(rmsnorm(x) * w_final) of the mask positions 1..k, the LM head's
  input.
"""
import numpy as np

from . import f32_to_bf16_array

EPS = 1e-6
THETA = 1e6


def bf16_round(x):
    """Values -> the float64 value of their bf16 rounding (ties to even, via fp32)."""
    return bf16_to_f32_array(f32_to_bf16_array(np.asarray(x, dtype=np.float32)))


def bf16_to_f32_array(bits):
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm(x, w):
    """x / sqrt(mean(x^2) + eps) * w over the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS)
    return x * inv * np.asarray(w, dtype=np.float64)


def rope(x, pos):
    """NeoX rotary embedding of x [..., n, hd] at integer positions pos (broadcast to
    x's leading axes): (x1, x2) -> (x1 cos - x2 sin, x2 cos + x1 sin) with x1 = dims
    0..hd/2-1, x2 = the rest, angle pos * THETA^(-2d/hd)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = THETA ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[..., None, None] * inv_freq  # [..., 1, half]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def attention(q, K, V):
    """Grouped-query attention of one request.  q [nq_rows, nq, hd], K, V [nk, nkv, hd]
    (float64 values); query head j reads kv head j // (nq / nkv); scale 1/sqrt(hd);
    softmax over all nk keys.  Returns [nq_rows, nq, hd]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    rows, nq, hd = q.shape
    nkv = K.shape[1]
    grp = nq // nkv
    out = np.empty_like(q)
    for j in range(nq):
        g = j // grp
        s = q[:, j, :] @ K[:, g, :].T / np.sqrt(hd)         # [rows, nk]
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, j, :] = p @ V[:, g, :]
    return out


def qk_norm_rope(x, w_norm, pos):
    """Per-head rmsnorm then rotary embedding of x [rows, n, hd] at positions pos [rows];
    bf16 result (as float64 values)."""
    return bf16_round(rope(rmsnorm(x, w_norm), pos))


def context_kv(ctx, layer, pos):
    """A layer's keys and values of context rows ctx [rows, H] (float64 values of bf16)
    at positions pos [rows]: (K [rows, nkv, hd], V [rows, nkv, hd]), bf16 values."""
    nq, nkv, hd = layer["nq"], layer["nkv"], layer["hd"]
    n = bf16_round(rmsnorm(ctx, layer["w_in"]))
    kv = bf16_round(n @ layer["w_qkv"][nq * hd:].T)
    k = kv[:, :nkv * hd].reshape(-1, nkv, hd)
    v = kv[:, nkv * hd:].reshape(-1, nkv, hd)
    return qk_norm_rope(k, layer["w_kn"], pos), v


def decoder_layer(x, layer, K_ctx, V_ctx, C):
    """One layer over one request's block rows x [k+1, H] (fp32 residual values).
    K_ctx, V_ctx [C, nkv, hd]: the layer's context keys and values (bf16 values).
    Returns the new residual (float64 values of fp32) and the block's (K, V)."""
    nq, nkv, hd = layer["nq"], layer["nkv"], layer["hd"]
    rows = x.shape[0]
    pos = C + np.arange(rows)
    n = bf16_round(rmsnorm(x, layer["w_in"]))
    qkv = bf16_round(n @ layer["w_qkv"].T)
    q = qk_norm_rope(qkv[:, :nq * hd].reshape(rows, nq, hd), layer["w_qn"], pos)
    k = qk_norm_rope(qkv[:, nq * hd:(nq + nkv) * hd].reshape(rows, nkv, hd), layer["w_kn"], pos)
    v = qkv[:, (nq + nkv) * hd:].reshape(rows, nkv, hd)
    o = bf16_round(attention(q, np.concatenate([K_ctx, k]), np.concatenate([V_ctx, v])))
    x = (x + bf16_round(o.reshape(rows, nq * hd) @ layer["w_o"].T)).astype(np.float32).astype(np.float64)
    n2 = bf16_round(rmsnorm(x, layer["w_post"]))
    gu = bf16_round(n2 @ layer["w_gu"].T)
    I = gu.shape[1] // 2
    act = bf16_round(silu(gu[:, :I]) * gu[:, I:])
    x = (x + bf16_round(act @ layer["w_d"].T)).astype(np.float32).astype(np.float64)
    return x, k, v


def backbone(block_tokens, ctx, layers, w_final, embed):
    """The drafter backbone of one request.  block_tokens [k+1] (anchor, then mask
    tokens); ctx [C, H] context features (bf16 values); embed [V, H] (bf16 values);
    layers: dicts of float64 weights (bf16 values) and the geometry nq, nkv, hd.
    Returns h [k, H] (bf16 values) for the mask positions."""
    C = ctx.shape[0]
    x = embed[np.asarray(block_tokens)].astype(np.float64)
    for layer in layers:
        K_ctx, V_ctx = context_kv(ctx, layer, np.arange(C))
        x, _, _ = decoder_layer(x, layer, K_ctx, V_ctx, C)
    return bf16_round(rmsnorm(x[1:], w_final))
