"""FP8 (E4M3) drafter-weight path through the C ABI against the oracle.

Tolerances (from the arithmetic):
  * Row quantisation: both sides divide in IEEE binary32 and round to the nearest
    E4M3 code (ties to even, saturating), so codes and scales are bit-exact.
  * FP8 GEMMs: E4M3 x E4M3 products are exact in fp32; the tensor cores sum them in
    fp32, the oracle in fp64.  Any fp32 summation order is within
    K * 2^-24 * sum|a_k w_k| of the exact sum; the two fp32 scale multiplications add
    at most 2 ulps of fp32; the fc output's bf16 rounding adds at most one bf16 ulp.
  * Integer-valued codes with power-of-two scales make every partial sum exact, so
    there the result is bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu

_LUT = None


def _dequant(codes):
    global _LUT
    if _LUT is None:
        _LUT = oracle.e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    return _LUT[codes]


def _gemm_bound(a8, sa, w8, sw):
    """Per-output bound on |fp32 result - exact result| (see module docstring)."""
    K = a8.shape[1]
    mag = np.abs(_dequant(a8)) @ np.abs(_dequant(w8)).T
    scale = np.abs(sa.astype(np.float64))[:, None] * np.abs(sw.astype(np.float64))[None, :]
    return K * 2.0 ** -24 * mag * scale


def _rows_with_spread(seed, R, C):
    """bf16 rows whose magnitudes span several binades (so codes cover the normal and
    subnormal E4M3 ranges), plus an all-zero row and a row with a single nonzero."""
    x = syn.normal_f32(seed, (R, C))
    row_scale = 2.0 ** np.linspace(-20, 10, R).astype(np.float32)
    col_scale = 2.0 ** (-(np.arange(C) % 13)).astype(np.float32)   # tiny entries -> subnormal codes
    x = x * row_scale[:, None] * col_scale[None, :]
    if R > 2:
        x[1] = 0.0
        x[2] = 0.0
        x[2, C // 2] = -3.5
    return syn.to_bf16_bits(x)


# ----------------------------------------------------------------------------- quantisation

@pytest.mark.parametrize("R,C", [(1, 128), (37, 256), (300, 1024), (5, 25600)])
def test_quantize_fp8_bit_exact(R, C):
    x = _rows_with_spread(40 + R, R, C)
    ref_codes, ref_scales = oracle.quantize_fp8_rows(x)
    codes, scales = ds.quantize_fp8(dev_bf16(x))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(scales).view(np.uint32), ref_scales.view(np.uint32))
    np.testing.assert_array_equal(host(codes), ref_codes)


def test_quantize_fp8_segments_with_row_stride():
    """The row is the concatenation of column segments read with a row stride wider
    than the segment (the fc taps), as the oracle sees the concatenated matrix."""
    R, C, T, ld = 19, 256, 5, 320
    full = _rows_with_spread(77, R, T * ld)
    full = full.reshape(R, T, ld)
    segs = [full[:, j, :C] for j in range(T)]
    x = np.concatenate(segs, axis=1)
    ref_codes, ref_scales = oracle.quantize_fp8_rows(x)
    base = dev_bf16(full.reshape(R, T * ld))
    views = [base[:, j * ld: j * ld + C] for j in range(T)]
    # one storage, T column windows: every window has row stride T*ld
    codes, scales = ds.quantize_fp8(views)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(scales).view(np.uint32), ref_scales.view(np.uint32))
    np.testing.assert_array_equal(host(codes), ref_codes)


@pytest.mark.parametrize("R,C,T,pad", [(7, 5120, 5, 64), (200, 4096, 2, 0), (3, 8192, 1, 16), (2, 1200, 3, 48)])
def test_quantize_fp8_few_long_rows(R, C, T, pad):
    """Few long rows (the activation rows of a step) are quantised by a cluster of CTAs
    per row that combine their partial maxima; the codes stay bit-exact, also where a
    CTA's range of the row crosses from one segment to the next."""
    ld = C + pad
    full = _rows_with_spread(90 + R, R, T * ld).reshape(R, T, ld)
    segs = [full[:, j, :C] for j in range(T)]
    x = np.concatenate(segs, axis=1)
    ref_codes, ref_scales = oracle.quantize_fp8_rows(x)
    base = dev_bf16(full.reshape(R, T * ld))
    codes, scales = ds.quantize_fp8([base[:, j * ld: j * ld + C] for j in range(T)])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(scales).view(np.uint32), ref_scales.view(np.uint32))
    np.testing.assert_array_equal(host(codes), ref_codes)


# ----------------------------------------------------------------------------- GEMMs

@pytest.mark.parametrize("M,H,V", [(1, 256, 4096), (7, 256, 4097), (33, 512, 1000),
                                   (130, 1024, 3000), (7, 5120, 1536)])
def test_lm_head_fp8_matches_oracle(M, H, V):
    h = syn.normal_bf16(300 + M, (M, H))
    w = syn.normal_bf16(400 + V, (V, H), (1.0 / H) ** 0.5)
    w8, ws = oracle.quantize_fp8_rows(w)
    a8, sa = oracle.quantize_fp8_rows(h)
    ref = oracle.lm_head_fp8(h, w8, ws)
    got = host(ds.lm_head_fp8(dev_bf16(h), dev(w8), dev(ws)))
    torch.cuda.synchronize()
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = _gemm_bound(a8, sa, w8, ws) + 2.0 ** -22 * np.abs(ref.astype(np.float64)) + 1e-30
    assert np.all(err <= bound), "max excess %.3e" % (err - bound).max()


def test_lm_head_fp8_integer_codes_bit_exact():
    """h holds integers in [-7, 7] with a 7 in every row: scale 7/448 = 2^-6 exactly and
    the codes are 64*h; weight codes are E4M3 integers with scale 1.  Every product and
    partial sum is an integer below 2^24, so the result is exact on both sides."""
    M, H, V = 21, 512, 3000
    rng = np.random.default_rng(5)
    hv = rng.integers(-7, 8, size=(M, H)).astype(np.float32)
    hv[:, 3] = 7.0
    h = syn.to_bf16_bits(hv)
    wv = rng.integers(-3, 4, size=(V, H)).astype(np.float32)
    w8 = oracle.f32_to_e4m3(wv)
    ws = np.ones((V,), np.float32)
    ref = oracle.lm_head_fp8(h, w8, ws)
    hd, w8d, wsd = dev_bf16(h), dev(w8), dev(ws)
    a = host(ds.lm_head_fp8(hd, w8d, wsd))
    b = host(ds.lm_head_fp8(hd, w8d, wsd))
    np.testing.assert_array_equal(a, ref)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ref, (hv.astype(np.float64) @ wv.T.astype(np.float64)).astype(np.float32))


def _assert_fc8_close(got_bits, ref_bits, taps, w8, sw):
    x = np.concatenate(taps, axis=1)
    a8, sa = oracle.quantize_fp8_rows(x)
    got = syn.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = syn.bf16_bits_to_f32(ref_bits).astype(np.float64)
    ulp = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7
    bound = ulp + _gemm_bound(a8, sa, w8, sw) * 1.0001 + 2.0 ** -22 * np.abs(ref)
    assert np.all(np.abs(got - ref) <= bound), "max excess %.3e" % (np.abs(got - ref) - bound).max()


@pytest.mark.parametrize("M,H,T", [(1, 256, 5), (7, 256, 5), (28, 512, 5), (130, 128, 3),
                                   (7, 1024, 5)])
def test_fc_project_fp8_matches_oracle(M, H, T):
    taps = [syn.normal_bf16(500 + 10 * j + M, (M, H), 2.0) for j in range(T)]
    fc_w = syn.normal_bf16(600 + H, (H, T * H), (1.0 / (T * H)) ** 0.5)
    w8, sw = oracle.quantize_fp8_rows(fc_w)
    ref = oracle.fc_project_fp8(taps, w8, sw)
    got = host_bf16_bits(ds.fc_project_fp8([dev_bf16(t) for t in taps], dev(w8), dev(sw)))
    torch.cuda.synchronize()
    _assert_fc8_close(got, ref, taps, w8, sw)


def test_fc_project_fp8_strided_taps():
    M, H, T, ld = 9, 256, 5, 384
    full = syn.normal_bf16(711, (M, T * ld), 1.5).reshape(M, T, ld)
    taps = [np.ascontiguousarray(full[:, j, :H]) for j in range(T)]
    fc_w = syn.normal_bf16(712, (H, T * H), (1.0 / (T * H)) ** 0.5)
    w8, sw = oracle.quantize_fp8_rows(fc_w)
    ref = oracle.fc_project_fp8(taps, w8, sw)
    base = dev_bf16(full.reshape(M, T * ld))
    views = [base[:, j * ld: j * ld + H] for j in range(T)]
    got = host_bf16_bits(ds.fc_project_fp8(views, dev(w8), dev(sw)))
    torch.cuda.synchronize()
    _assert_fc8_close(got, ref, taps, w8, sw)


def test_fp8_weights_quantised_on_device_match_oracle_codes():
    """The offline weight quantisation (device) gives the oracle's codes, so an FP8
    LM head fed with device-quantised weights equals the oracle's FP8 LM head."""
    M, H, V = 7, 512, 2053
    h = syn.normal_bf16(801, (M, H))
    w = syn.normal_bf16(802, (V, H), (1.0 / H) ** 0.5)
    w8_ref, ws_ref = oracle.quantize_fp8_rows(w)
    w8d, wsd = ds.quantize_fp8(dev_bf16(w))
    np.testing.assert_array_equal(host(w8d), w8_ref)
    np.testing.assert_array_equal(host(wsd).view(np.uint32), ws_ref.view(np.uint32))
    a8, sa = oracle.quantize_fp8_rows(h)
    ref = oracle.lm_head_fp8(h, w8_ref, ws_ref)
    got = host(ds.lm_head_fp8(dev_bf16(h), w8d, wsd))
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bound = _gemm_bound(a8, sa, w8_ref, ws_ref) + 2.0 ** -22 * np.abs(ref.astype(np.float64)) + 1e-30
    assert np.all(err <= bound)


# ----------------------------------------------------------------------------- 27B shapes
# The FP8 benchmark line's shapes (H 5120, 5 taps, V 151936, k 7; batch 1 and 16):
# weights quantised on the device once, checked against the oracle on sampled rows;
# GEMM outputs checked on sampled outputs.

@pytest.fixture(scope="module")
def w27_fp8():
    w = syn.weights(5120, 5, 151936, 64, with_conf=False, with_markov=False)
    d = {"fc_w": w["fc_w"], "lm_w": w["lm_w"]}
    d["fc_w8"], d["fc_s"] = ds.quantize_fp8(dev_bf16(w["fc_w"]))
    d["lm_w8"], d["lm_s"] = ds.quantize_fp8(dev_bf16(w["lm_w"]))
    torch.cuda.synchronize()
    return d


def test_27b_weight_quantisation_sampled_rows(w27_fp8):
    for name, n in (("fc_w", 5120), ("lm_w", 151936)):
        rows = np.unique(np.concatenate([np.random.default_rng(n).choice(n, 500, replace=False),
                                         [0, n - 1]]))
        ref_codes, ref_scales = oracle.quantize_fp8_rows(w27_fp8[name][rows])
        idx = torch.from_numpy(rows).cuda()
        np.testing.assert_array_equal(host(w27_fp8[name[:-2] + "_w8"].index_select(0, idx)), ref_codes)
        np.testing.assert_array_equal(host(w27_fp8[name[:-2] + "_s"].index_select(0, idx)).view(np.uint32),
                                      ref_scales.view(np.uint32))


@pytest.mark.parametrize("B", [1, 16])
def test_27b_lm_head_fp8_sampled_rows(w27_fp8, B):
    k, H, V = 7, 5120, 151936
    h = syn.normal_bf16(900 + B, (B * k, H))
    logits = host(ds.lm_head_fp8(dev_bf16(h), w27_fp8["lm_w8"], w27_fp8["lm_s"]))
    rows = np.random.default_rng(B).choice(V, 2000, replace=False)
    rows = np.unique(np.concatenate([rows, logits.argmax(axis=1), [0, V - 1]]))
    w8, sw = oracle.quantize_fp8_rows(w27_fp8["lm_w"][rows])
    a8, sa = oracle.quantize_fp8_rows(h)
    ref = oracle.gemm_fp8(a8, sa, w8, sw)
    err = np.abs(logits[:, rows].astype(np.float64) - ref.astype(np.float64))
    bound = _gemm_bound(a8, sa, w8, sw) + 2.0 ** -22 * np.abs(ref.astype(np.float64)) + 1e-30
    assert np.all(err <= bound), "max excess %.3e" % (err - bound).max()


@pytest.mark.parametrize("B", [1, 16])
def test_27b_fc_project_fp8_sampled_columns(w27_fp8, B):
    k, H, T = 7, 5120, 5
    st = syn.step_inputs(0, B, k, H, T, 151936, ("ramp", 0.5, 3.0))
    h = host_bf16_bits(ds.fc_project_fp8([dev_bf16(t) for t in st["taps"]], w27_fp8["fc_w8"],
                                         w27_fp8["fc_s"]))
    cols = np.sort(np.random.default_rng(B).choice(H, 192, replace=False))
    w8, sw = oracle.quantize_fp8_rows(w27_fp8["fc_w"][cols])
    ref = oracle.fc_project_fp8(st["taps"], w8, sw)
    _assert_fc8_close(h[:, cols], ref, st["taps"], w8, sw)
