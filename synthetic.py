"""Seeded synthetic inputs for the DSpark readout + verify path.

Shared by the tests, the smoke check and the benchmark.  This module holds no
arithmetic of the method itself: it only draws random tensors of the shapes,
scales and dtypes of the workloads and hands them out as numpy arrays (bf16
as uint16 bit patterns, rounded to nearest-even by ``torch``'s cast).

Workload recipe (weights are random-init: no trained drafter is used):
  - fc weight  W_fc [H, T*H]  ~ N(0, 1/(T*H))   bf16
  - LM head    W_lm [V, H]    ~ N(0, 1/H)       bf16
  - markov_w1  W1   [V, r]    ~ N(0, 1)         bf16  (embedding)
  - markov_w2  W2   [V, r]    ~ N(0, 1/r)       bf16  (Linear r -> V)
  - confidence w    [H]       ~ N(0, 1/H)       bf16, b = 0
  - taps       T x [B*k, H]   ~ N(0, 1)         bf16, redrawn every step
  - prev token [B]            ~ U[0, V)         int32 (step 0)
  - target noise [B, k+1, V]  = sigma_j * N(0, 1) fp32; the target logits of
    block row j are the draft logits of row min(j, k-1) plus this noise
    (whoever holds the draft logits adds them).
Seeds: tensor i of the weights uses seed 1 + i; step s uses seed 1000 + s.
"""
import os

import numpy as np
import torch

# Named workloads: the model shapes of the pages (Qwen3.8-27B DSpark drafter,
# Qwen3.8-Flash-Next DFlash2 drafter) and a tiny one for exhaustive checks.
CONFIGS = {
    "tiny": dict(H=256, T=5, V=4096, r=16, k=7, B=1, steps=8, mode=0,
                 sigma=("const", 1.0), conf=False),
    "27b_b1": dict(H=5120, T=5, V=151936, r=64, k=7, B=1, steps=1, mode=1,
                   sigma=("ramp", 0.5, 3.0), conf=False),
    # the same workload with the fc and LM-head weights held as E4M3 codes + row scales
    "27b_b1_fp8": dict(H=5120, T=5, V=151936, r=64, k=7, B=1, steps=1, mode=1,
                       sigma=("ramp", 0.5, 3.0), conf=False, fp8=True),
    "27b_b16": dict(H=5120, T=5, V=151936, r=64, k=7, B=16, steps=1, mode=1,
                    sigma=("ramp", 0.5, 3.0), conf=True),
    "flash_b4": dict(H=2560, T=5, V=151936, r=64, k=7, B=4, steps=1, mode=1,
                     sigma=("ramp", 0.5, 3.0), conf=False),
    # the 27B batch-1 step with one drafter backbone layer between the fc and the LM
    # head, over a 1024-token context (the block's keys/values follow it in the cache)
    "27b_b1_backbone": dict(H=5120, T=5, V=151936, r=64, k=7, B=1, steps=1, mode=1,
                            sigma=("ramp", 0.5, 3.0), conf=False, backbone=dict(L=1, C=1024)),
}
FLASH_PREFILL = dict(H=2560, T=5, M=4096)


def sigma_schedule(spec, k):
    """Per-row noise scale of the k+1 target rows."""
    if spec[0] == "const":
        return np.full(k + 1, float(spec[1]))
    lo, hi = float(spec[1]), float(spec[2])
    return lo + (hi - lo) * np.arange(k + 1) / k


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


_BLOCK = 1 << 22  # elements per independently seeded block of a large draw


def normal_f32(seed, shape, std=1.0):
    """N(0, std^2) fp32.  Large arrays are drawn in blocks of 2^22 elements, block i from
    the i-th child of SeedSequence(seed), in parallel threads; the result depends only on
    (seed, shape)."""
    n = int(np.prod(shape))
    if n <= _BLOCK:
        a = _rng(seed).standard_normal(size=shape, dtype=np.float32)
    else:
        from concurrent.futures import ThreadPoolExecutor
        a = np.empty(n, dtype=np.float32)
        nb = (n + _BLOCK - 1) // _BLOCK
        kids = np.random.SeedSequence(seed).spawn(nb)

        def fill(i):
            lo, hi = i * _BLOCK, min(n, (i + 1) * _BLOCK)
            np.random.Generator(np.random.PCG64(kids[i])).standard_normal(
                size=hi - lo, dtype=np.float32, out=a[lo:hi])

        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nb)))
        a = a.reshape(shape)
    if std != 1.0:
        a *= np.float32(std)
    return a


def to_bf16_bits(a):
    """fp32 numpy -> bf16 bit patterns (uint16), round to nearest even (torch cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed, shape, std=1.0):
    return to_bf16_bits(normal_f32(seed, shape, std))


def weights(H, T, V, r, with_conf=False, with_markov=True):
    """Drafter weights (numpy uint16 bf16 bits)."""
    w = {
        "fc_w": normal_bf16(1, (H, T * H), (1.0 / (T * H)) ** 0.5),
        "lm_w": normal_bf16(2, (V, H), (1.0 / H) ** 0.5),
    }
    if with_markov:
        w["w1"] = normal_bf16(3, (V, r), 1.0)
        w["w2"] = normal_bf16(4, (V, r), (1.0 / r) ** 0.5)
    if with_conf:
        w["conf_w"] = normal_bf16(5, (H,), (1.0 / H) ** 0.5)
        w["conf_b"] = 0.0
        w["conf_tau"] = 0.5
    return w


# Geometry of the drafter backbone's layers per hidden size (128-wide heads, 5 query
# heads per key/value head, the MLP width of the Qwen3 model of that hidden size).
BACKBONE_GEOMETRY = {5120: dict(nq=40, nkv=8, I=17408), 2560: dict(nq=20, nkv=4, I=9728)}


def backbone_weights(H, nq, nkv, I, L, seed=200):
    """Random backbone weights (numpy uint16 bf16 bits), one dict per layer, and the
    final norm weight: norms ~ 1 + N(0, 0.1^2), projections ~ N(0, 1/fan_in)."""
    layers = []
    for li in range(L):
        s = seed + 16 * li
        layers.append({
            "nq": nq, "nkv": nkv,
            "w_in": to_bf16_bits(1.0 + normal_f32(s, (H,), 0.1)),
            "w_post": to_bf16_bits(1.0 + normal_f32(s + 1, (H,), 0.1)),
            "w_qn": to_bf16_bits(1.0 + normal_f32(s + 2, (128,), 0.1)),
            "w_kn": to_bf16_bits(1.0 + normal_f32(s + 3, (128,), 0.1)),
            "w_qkv": normal_bf16(s + 4, ((nq + 2 * nkv) * 128, H), (1.0 / H) ** 0.5),
            "w_o": normal_bf16(s + 5, (H, nq * 128), (1.0 / (nq * 128)) ** 0.5),
            "w_gu": normal_bf16(s + 6, (2 * I, H), (1.0 / H) ** 0.5),
            "w_d": normal_bf16(s + 7, (H, I), (1.0 / I) ** 0.5),
        })
    w_final = to_bf16_bits(1.0 + normal_f32(seed + 15, (H,), 0.1))
    return layers, w_final


def step_inputs(step, B, k, H, T, V, sigma_spec):
    """Per-step activations: taps, initial prev tokens, target noise."""
    s = 1000 + step
    taps = [normal_bf16(s * 16 + j, (B * k, H)) for j in range(T)]
    prev = _rng(s * 16 + 15).integers(0, V, size=(B,), dtype=np.int64).astype(np.int32)
    sig = sigma_schedule(sigma_spec, k).astype(np.float32)
    noise = normal_f32(s * 16 + 14, (B, k + 1, V)) * sig[None, :, None]
    return {"taps": taps, "prev": prev, "noise": noise}


def uniform_logits(seed, shape, scale=1.0):
    """Plain fp32 N(0, scale^2) logits, for checks of the chain and of verify on
    inputs that do not go through the GEMMs."""
    return normal_f32(seed, shape, scale)


def integer_valued_bf16(seed, shape, lo=-3, hi=4):
    """Small-integer bf16 tensors: products and sums of these are exact in fp32, so any
    summation order gives the same bits."""
    a = _rng(seed).integers(lo, hi, size=shape).astype(np.float32)
    return to_bf16_bits(a)
