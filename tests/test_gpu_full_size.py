"""Full-size parity: the workloads' own shapes, through the C ABI in the launch
configuration the benchmark uses, against the CPU oracle on sampled outputs (GEMMs)
or whole (Markov chain, verify, the Tiny end-to-end run).

Workloads: Tiny (H 256, V 4096, r 16, k 7, B 1, 8 chained steps, greedy);
Qwen3.8-27B DSpark shapes (H 5120, 5 taps, V 151936, r 64, k 7) at batch 1 and 16;
Flash-Next DFlash2 shapes (H 2560) at batch 4 and its 4096-token prefill fc; sweep
corners (B 64, k 4..7, r 32/128).
"""
import numpy as np
import pytest
import torch

import oracle
import parity_log
import speculative_decoding_fc_gb300 as ds
import synthetic as syn
from gpu_util import bf16_ulp_diff, dev, dev_bf16, host, host_bf16_bits
from step_util import chain_forced, decision_mask

pytestmark = pytest.mark.gpu

RTOL = ATOL = 2e-3


def _fc_bound_ok(got_bits, ref_bits, taps, w_rows):
    x = np.concatenate([syn.bf16_bits_to_f32(t) for t in taps], axis=1).astype(np.float64)
    w = syn.bf16_bits_to_f32(w_rows).astype(np.float64)
    mag = np.abs(x) @ np.abs(w).T
    got = syn.bf16_bits_to_f32(got_bits).astype(np.float64)
    ref = syn.bf16_bits_to_f32(ref_bits).astype(np.float64)
    bound = np.maximum(np.abs(ref), 2.0 ** -126) * 2.0 ** -7 + x.shape[1] * 2.0 ** -24 * mag
    assert np.all(np.abs(got - ref) <= bound)
    assert (bf16_ulp_diff(got_bits, ref_bits) > 1).mean() < 0.01


def _tokens_match_or_near_tie(gpu_tokens, ref_z, ref_tokens, lens=None):
    """Draft tokens equal the oracle's; a mismatch is accepted only where the oracle's
    own top value and the GPU's choice are within the logit tolerance (a near tie),
    and then the rest of that request's chain is not compared.  Returns the count."""
    B, k = ref_tokens.shape
    flips = 0
    for b in range(B):
        L = k if lens is None else lens[b]
        for i in range(L):
            if gpu_tokens[b, i] != ref_tokens[b, i]:
                z = ref_z[b, i].astype(np.float64)
                top = z.max()
                assert top - z[gpu_tokens[b, i]] <= 2 * (ATOL + RTOL * abs(top)), (b, i)
                flips += 1
                break
    return flips


@pytest.fixture(scope="module")
def w27():
    return syn.weights(5120, 5, 151936, 64, with_conf=True)


@pytest.fixture(scope="module")
def w27_dev(w27):
    return {k: dev_bf16(v) for k, v in w27.items() if isinstance(v, np.ndarray)}


# ----------------------------------------------------------------------------- 27B shapes

@pytest.mark.parametrize("B", [1, 16])
def test_27b_fc_sampled_columns(w27, w27_dev, B):
    k, H, T = 7, 5120, 5
    st = syn.step_inputs(0, B, k, H, T, 151936, ("ramp", 0.5, 3.0))
    h = host_bf16_bits(ds.fc_project([dev_bf16(t) for t in st["taps"]], w27_dev["fc_w"]))
    cols = np.sort(np.random.default_rng(B).choice(H, 192, replace=False))
    ref = oracle.fc_project(st["taps"], w27["fc_w"][cols])
    _fc_bound_ok(h[:, cols], ref, st["taps"], w27["fc_w"][cols])


@pytest.mark.parametrize("B", [1, 16])
def test_27b_lm_head_sampled_rows(w27, w27_dev, B):
    k, H, V = 7, 5120, 151936
    h = syn.normal_bf16(77 + B, (B * k, H))
    logits = host(ds.lm_head(dev_bf16(h), w27_dev["lm_w"]))
    rows = np.random.default_rng(B).choice(V, 3000, replace=False)
    rows = np.unique(np.concatenate([rows, logits.argmax(axis=1), [0, V - 1]]))
    ref = oracle.lm_head(h, w27["lm_w"][rows])
    err = np.abs(logits[:, rows].astype(np.float64) - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref))


@pytest.mark.parametrize("B", [1, 16])
def test_27b_fc_lm_head_one_launch(w27, w27_dev, B):
    """The single-launch fc + LM head at the workload's shapes gives the bits of the two
    separate launches (one CTA per SM in both), sampled against the oracle."""
    k, H, T, V = 7, 5120, 5, 151936
    st = syn.step_inputs(3, B, k, H, T, V, ("ramp", 0.5, 3.0))
    taps = [dev_bf16(t) for t in st["taps"]]
    h, logits = ds.fc_lm_head(taps, w27_dev["fc_w"], w27_dev["lm_w"])
    h2 = ds.fc_project(taps, w27_dev["fc_w"])
    l2 = ds.lm_head(h2, w27_dev["lm_w"])
    torch.cuda.synchronize()
    hb = host_bf16_bits(h)
    np.testing.assert_array_equal(hb, host_bf16_bits(h2))
    np.testing.assert_array_equal(host(logits), host(l2))
    rows = np.random.default_rng(B + 7).choice(V, 1000, replace=False)
    ref = oracle.lm_head(hb, w27["lm_w"][rows])
    err = np.abs(host(logits)[:, rows].astype(np.float64) - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref))


@pytest.mark.parametrize("B", [1, 16])
def test_27b_markov_chain_bit_exact(w27, w27_dev, B):
    k, V = 7, 151936
    logits = syn.uniform_logits(500 + B, (B, k, V), 1.0)
    prev = syn.step_inputs(1, B, k, 64, 1, V, ("const", 1.0))["prev"]
    ref = oracle.greedy_sample(logits, w27["w1"], w27["w2"], prev)
    lg = dev(logits)
    d, qs = ds.greedy_sample(lg, w27_dev["w1"], w27_dev["w2"], dev(prev))
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
    np.testing.assert_array_equal(host(lg), ref["z"])
    np.testing.assert_allclose(host(qs)[..., 1], ref["q_sumexp"], rtol=1e-5)


def test_27b_b1_readout_from_h_end_to_end(w27, w27_dev):
    """LM head + chain on the full vocabulary from one fc output h, then probabilistic
    verify against target logits built from the oracle's draft logits.  Every request is
    compared; only counted exclusions are skipped."""
    B, k, H, V = 1, 7, 5120, 151936
    st = syn.step_inputs(3, B, k, H, 5, V, ("ramp", 0.5, 3.0))
    h = oracle.fc_project(st["taps"], w27["fc_w"])
    logits = oracle.lm_head(h, w27["lm_w"]).reshape(B, k, V)
    out = ds.draft_readout(dev_bf16(h), w27_dev["lm_w"], w27_dev["w1"], w27_dev["w2"],
                           dev(st["prev"]), B, k)
    gd = host(out["draft_tokens"])
    ref = chain_forced(logits, w27["w1"], w27["w2"], st["prev"], gd)
    z = host(out["logits"])
    err = np.abs(z.astype(np.float64) - ref["z"])
    assert np.all(err <= ATOL + RTOL * np.abs(ref["z"]))
    assert ref["flip"] == 0   # a flip would need a gap below ~1e-5 at this size
    target = (np.concatenate([ref["z"], ref["z"][:, -1:]], axis=1) + st["noise"]).astype(np.float32)
    ver = oracle.verify(1, target, ref["tokens"], None, ref["z"], seed=0, step=3)
    a, n = ds.verify(1, dev(target), out["draft_tokens"], None, out["logits"], out["q_stats"],
                     seed=0, step=3)
    # the GPU verifies its own z (within ~1e-5 of the oracle's): decisions must agree
    # wherever the oracle's margin exceeds the propagated logit difference
    ex_a, ex_d = decision_mask(ver, 1e-5 + 4 * float(err.max()))
    ex = ex_a | ex_d
    parity_log.record("27b_b1 readout from h + verify(prob)", "request", B, near_tie=ref["near_tie"],
                      flip=ref["flip"], accept=ex_a.sum(), draw=ex_d.sum())
    assert ex.sum() == 0
    np.testing.assert_array_equal(host(a), ver["accepted_len"])
    np.testing.assert_array_equal(host(n), ver["next_token"])


def test_27b_b16_confidence_and_truncation(w27, w27_dev):
    B, k, H, V = 16, 7, 5120, 151936
    h = syn.normal_bf16(91, (B * k, H))
    d0 = np.tile(np.arange(k, dtype=np.int32), (B, 1))
    ref = oracle.confidence(h, B, k, w27["conf_w"], 0.0, 0.5, d0)
    drafts = dev(d0)
    dl, cf = ds.confidence_truncate(dev_bf16(h), w27_dev["conf_w"], drafts, B, k, 0.0, 0.5,
                                    conf_out=torch.empty((B, k), dtype=torch.float32, device="cuda"))
    np.testing.assert_allclose(host(cf), ref["conf"], rtol=1e-5, atol=1e-6)
    safe = np.all(np.abs(ref["zc"]) >= 1e-4, axis=1)
    np.testing.assert_array_equal(host(dl)[safe], ref["draft_len"][safe])
    np.testing.assert_array_equal(host(drafts)[safe], ref["draft_tokens"][safe])
    assert (ref["draft_len"] < k).any() and (ref["draft_len"] > 0).any()


@pytest.mark.parametrize("B", [1, 16])
def test_27b_verify_probabilistic_full_vocab(B):
    k, V = 7, 151936
    z = syn.uniform_logits(700 + B, (B, k, V), 1.0)
    drafts = z.argmax(axis=-1).astype(np.int32)
    sig = syn.sigma_schedule(("ramp", 0.5, 3.0), k).astype(np.float32)
    target = (np.concatenate([z, z[:, -1:]], axis=1)
              + syn.uniform_logits(701 + B, (B, k + 1, V), 1.0) * sig[None, :, None]).astype(np.float32)
    ref = oracle.verify(1, target, drafts, None, z, seed=0, step=11)
    a, n = ds.verify(1, dev(target), dev(drafts), None, dev(z), None, seed=0, step=11)
    ex_a, ex_d = decision_mask(ref)
    ex = ex_a | ex_d
    parity_log.record("27b verify(prob) full vocab B=%d" % B, "request", B, accept=ex_a.sum(),
                      draw=ex_d.sum())
    assert ex.sum() <= max(1, B // 16)
    np.testing.assert_array_equal(host(a)[~ex], ref["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ref["next_token"][~ex])
    a0, n0 = ds.verify(0, dev(target), dev(drafts))
    ref0 = oracle.verify(0, target, drafts)
    np.testing.assert_array_equal(host(a0), ref0["accepted_len"])
    np.testing.assert_array_equal(host(n0), ref0["next_token"])


# ----------------------------------------------------------------------------- whole steps

def _bb_vals(bits):
    return syn.bf16_bits_to_f32(bits).astype(np.float64)


def _backbone_from_fc(bbc, w, wd, hd, gh, prev, B, k, H, V, seed):
    """The drafter backbone between the fc and the LM head, as the benchmark runs it: the
    caches hold C - k older context rows (written by backbone_context), the fc output
    hd becomes each request's newest k context rows inside backbone_block, and the
    block is [prev, mask x k] with the LM head's weight as the embedding table.  Checked
    against the oracle's backbone on the same context (the older rows, then the GPU's fc
    rows, which the fc check covers) within the chained-layer bound: rms error at most
    2^-7 and max error at most 2^-4 of the reference's rms, per request.  Returns the
    GPU's h (the LM head's input)."""
    from oracle import backbone as bb
    g = syn.BACKBONE_GEOMETRY[H]
    L, C = bbc["L"], bbc["C"]
    layers, wf = syn.backbone_weights(H, g["nq"], g["nkv"], g["I"], L, seed=seed + 300)
    lay_d = [ds.BackboneLayer(l["nq"], l["nkv"], *[dev_bf16(l[x]) for x in (
        "w_in", "w_post", "w_qn", "w_kn", "w_qkv", "w_o", "w_gu", "w_d")]) for l in layers]
    old = syn.normal_bf16(seed + 301, (B, C - k, H))
    kcs = [torch.zeros((B, C + k + 1, g["nkv"], 128), dtype=torch.bfloat16, device="cuda") for _ in layers]
    vcs = [torch.zeros_like(t) for t in kcs]
    wsp = ds.Workspaces()
    ds.backbone_context(dev_bf16(old.reshape(-1, H)), lay_d, kcs, vcs, 0, workspaces=wsp)
    toks = np.concatenate([np.asarray(prev)[:, None], np.full((B, k), V - 1)], axis=1).astype(np.int32)
    hb = ds.backbone_block(dev(toks), wd["lm_w"], lay_d, dev_bf16(wf), kcs, vcs, C, workspaces=wsp,
                           ctx=hd, ctx_pos0=C - k)
    got = _bb_vals(host_bf16_bits(hb)).reshape(B, k, H)
    ref_layers = []
    for l in layers:
        ref_layers.append({n: (_bb_vals(v) if isinstance(v, np.ndarray) else v) for n, v in l.items()})
        ref_layers[-1]["hd"] = 128
    new = gh.reshape(B, k, H)
    for b in range(B):
        ctx_b = _bb_vals(np.concatenate([old[b], new[b]]))
        emb = _bb_vals(w["lm_w"][toks[b]])        # the block's rows of the tied table
        ref = bb.backbone(np.arange(k + 1), ctx_b, ref_layers, _bb_vals(wf), emb)
        err = got[b] - ref
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.sqrt(np.mean(err ** 2)) <= rms * 2.0 ** -7, (b, np.sqrt(np.mean(err ** 2)) / rms)
        assert np.abs(err).max() <= rms * 2.0 ** -4, (b, np.abs(err).max() / rms)
    return hb


def _whole_step(label, w, wd, B, k, H, T, V, seed, conf, split, backbone=None):
    """One step through the GPU path exactly as the benchmark runs it (GPU fc -> [drafter
    backbone ->] LM head -> chain with q statistics -> [confidence] -> probabilistic
    verify), against the oracle from scratch on the same inputs.  Checks, in order: h
    within the fc bound; [the backbone's output within its chained bound, after which the
    oracle's readout starts from the GPU's backbone output;] the draft logits within the
    logit tolerance and the tokens equal (near-tie flips counted, the oracle then
    teacher-forced); draft lengths equal away from the confidence window; verify
    bit-exact against the oracle on the GPU's own drafts and draft logits (only the
    oracle's margin exclusions skipped); and against the oracle's from-scratch step,
    where a request also counts as excluded when the oracle's own decision changes
    between its draft logits and the GPU's."""
    st = syn.step_inputs(seed, B, k, H, T, V, ("ramp", 0.5, 3.0))
    hd = ds.fc_project([dev_bf16(t) for t in st["taps"]], wd["fc_w"])
    gh = host_bf16_bits(hd)
    h_ref = oracle.fc_project(st["taps"], w["fc_w"])
    _fc_bound_ok(gh, h_ref, st["taps"], w["fc_w"])
    if backbone is not None:
        hd = _backbone_from_fc(backbone, w, wd, hd, gh, st["prev"], B, k, H, V, seed)
        gh = h_ref = host_bf16_bits(hd)
    out = ds.draft_readout(hd, wd["lm_w"], wd["w1"], wd["w2"], dev(st["prev"]), B, k,
                           conf_w=wd["conf_w"] if conf else None, conf_b=0.0, conf_tau=0.5)
    gz = host(out["logits"])
    gd = host(out["draft_tokens"])
    gl = host(out["draft_len"])
    logits = oracle.lm_head(h_ref, w["lm_w"]).reshape(B, k, V)
    ch = chain_forced(logits, w["w1"], w["w2"], st["prev"], gd, lens=gl)
    zerr = np.abs(gz.astype(np.float64) - ch["z"])
    for b in range(B):   # positions up to the draft length run on the same context
        assert np.all(zerr[b, :gl[b]] <= ATOL + RTOL * np.abs(ch["z"][b, :gl[b]]))
    n_conf = 0
    if conf:
        c = oracle.confidence(h_ref, B, k, w["conf_w"], 0.0, 0.5, ch["tokens"])
        # the two sides' h differ by bf16 roundings: widen the window by their effect
        dh = np.abs(syn.bf16_bits_to_f32(gh).astype(np.float64) - syn.bf16_bits_to_f32(h_ref))
        dzc = (dh @ np.abs(syn.bf16_bits_to_f32(w["conf_w"]).astype(np.float64))).reshape(B, k)
        amb = np.abs(c["zc"]) < 1e-4 + dzc
        ok = np.array([not amb[b, :min(k, c["draft_len"][b] + 1)].any() for b in range(B)])
        n_conf = int((~ok).sum())
        np.testing.assert_array_equal(gl[ok], c["draft_len"][ok])
        ref_len = np.where(ok, c["draft_len"], gl).astype(np.int32)
    else:
        assert (gl == k).all()
        ref_len = gl.astype(np.int32)
    target = (np.concatenate([ch["z"], ch["z"][:, -1:]], axis=1) + st["noise"]).astype(np.float32)
    gdt = dev(target)
    if split:
        tms, targ = ds.row_stats(gdt)
        a, n = ds.verify_from_stats(1, gdt, tms, targ, out["draft_tokens"], out["draft_len"],
                                    out["logits"], out["q_stats"], seed=7, step=seed)
    else:
        a, n = ds.verify(1, gdt, out["draft_tokens"], out["draft_len"], out["logits"],
                         out["q_stats"], seed=7, step=seed)
    a, n = host(a), host(n)
    # level 1: the oracle on the GPU's own drafts, draft lengths and draft logits
    same = oracle.verify(1, target, gd, gl, gz, seed=7, step=seed)
    ex_a1, ex_d1 = decision_mask(same)
    ex1 = ex_a1 | ex_d1
    np.testing.assert_array_equal(a[~ex1], same["accepted_len"][~ex1])
    np.testing.assert_array_equal(n[~ex1], same["next_token"][~ex1])
    # level 2: the oracle's from-scratch step (its drafts forced only at counted flips)
    scratch = oracle.verify(1, target, np.where(np.arange(k)[None] < ref_len[:, None], ch["tokens"], -1),
                            ref_len, ch["z"], seed=7, step=seed)
    ex_a2, ex_d2 = decision_mask(scratch, 1e-5 + 4 * float(zerr.max()))
    zsens = (scratch["accepted_len"] != same["accepted_len"]) | (scratch["next_token"] != same["next_token"])
    ex2 = ex1 | ex_a2 | ex_d2 | zsens | (ref_len != gl)
    np.testing.assert_array_equal(a[~ex2], scratch["accepted_len"][~ex2])
    np.testing.assert_array_equal(n[~ex2], scratch["next_token"][~ex2])
    parity_log.record(label, "request", B, near_tie=ch["near_tie"], flip=ch["flip"],
                      accept=(ex_a1 | ex_a2).sum(), draw=(ex_d1 | ex_d2).sum(), z_sensitive=zsens.sum(),
                      confidence=n_conf)
    assert ex1.sum() <= max(1, B // 16)
    assert ex2.sum() <= max(1, B // 8)
    return a, n


@pytest.mark.parametrize("split", [True, False])
def test_27b_b16_whole_step(w27, w27_dev, split):
    """27B batch 16, confidence head on, probabilistic verify: the benchmark's batch-16
    step, through the split verify (target statistics, then one decision kernel) and the
    all-in-one verify."""
    _whole_step("27b_b16 whole step (%s verify)" % ("split" if split else "inline"),
                w27, w27_dev, 16, 7, 5120, 5, 151936, 21, True, split)


def test_27b_b1_whole_step(w27, w27_dev):
    _whole_step("27b_b1 whole step (split verify)", w27, w27_dev, 1, 7, 5120, 5, 151936, 22,
                False, True)


@pytest.mark.parametrize("B,conf", [(1, False), (2, True)])
def test_27b_whole_step_with_backbone(w27, w27_dev, B, conf):
    """The benchmark's backbone step: one 27B drafter layer over a 1024-token context
    between the fc and the LM head (batch 1), and batch 2 with the confidence head
    reading the backbone's output."""
    _whole_step("27b_b%d_backbone whole step (split verify)" % B, w27, w27_dev, B, 7, 5120, 5, 151936,
                24 + B, conf, True, backbone=dict(L=1, C=1024))


# ----------------------------------------------------------------------------- Flash-Next

def test_flash_prefill_fc_4096_tokens():
    M, H, T = 4096, 2560, 5
    fc_w = syn.normal_bf16(1, (H, T * H), (1.0 / (T * H)) ** 0.5)
    taps = [syn.normal_bf16(6000 + j, (M, H)) for j in range(T)]
    h = host_bf16_bits(ds.fc_project([dev_bf16(t) for t in taps], dev_bf16(fc_w)))
    cols = np.sort(np.random.default_rng(5).choice(H, 24, replace=False))
    rows = np.sort(np.random.default_rng(6).choice(M, 1024, replace=False))
    sub_taps = [t[rows] for t in taps]
    ref = oracle.fc_project(sub_taps, fc_w[cols])
    _fc_bound_ok(h[np.ix_(rows, cols)], ref, sub_taps, fc_w[cols])


def test_flash_b4_whole_step():
    """Flash-Next DFlash2 shapes (H 2560), batch 4: the whole step with verify."""
    B, k, H, T, V, r = 4, 7, 2560, 5, 151936, 64
    w = syn.weights(H, T, V, r, with_conf=True)
    wd = {n: dev_bf16(v) for n, v in w.items() if isinstance(v, np.ndarray)}
    _whole_step("flash_b4 whole step (split verify)", w, wd, B, k, H, T, V, 23, False, True)


def test_flash_b2_whole_step_with_two_backbone_layers():
    """Flash-Next geometry (H 2560, 20 query / 4 key-value heads), two backbone layers over
    a 200-token context, batch 2, confidence head on."""
    B, k, H, T, V, r = 2, 7, 2560, 5, 151936, 64
    w = syn.weights(H, T, V, r, with_conf=True)
    wd = {n: dev_bf16(v) for n, v in w.items() if isinstance(v, np.ndarray)}
    _whole_step("flash_b2_backbone whole step (inline verify)", w, wd, B, k, H, T, V, 27, True, False,
                backbone=dict(L=2, C=200))


# ----------------------------------------------------------------------------- Tiny, 8 steps

def test_tiny_eight_steps_end_to_end():
    """Eight chained steps of the Tiny workload (greedy): each step's prev token is the
    GPU's own verify output of the step before.  The oracle runs the same chain from
    scratch and is teacher-forced only at counted near ties; greedy verify on the same
    drafts and target must then agree exactly, including the next token both carry on."""
    cfg = syn.CONFIGS["tiny"]
    B, k, H, T, V, r = (cfg[x] for x in ("B", "k", "H", "T", "V", "r"))
    w = syn.weights(H, T, V, r)
    wd = {n: dev_bf16(v) for n, v in w.items()}
    prev = syn.step_inputs(0, B, k, H, T, V, cfg["sigma"])["prev"]
    near = flips = 0
    for step in range(cfg["steps"]):
        st = syn.step_inputs(step, B, k, H, T, V, cfg["sigma"])
        h = ds.fc_project([dev_bf16(t) for t in st["taps"]], wd["fc_w"])
        out = ds.draft_readout(h, wd["lm_w"], wd["w1"], wd["w2"], dev(prev), B, k)
        gd = host(out["draft_tokens"])
        h_ref = oracle.fc_project(st["taps"], w["fc_w"])
        _fc_bound_ok(host_bf16_bits(h), h_ref, st["taps"], w["fc_w"])
        ch = chain_forced(oracle.lm_head(h_ref, w["lm_w"]).reshape(B, k, V), w["w1"], w["w2"], prev, gd)
        near += ch["near_tie"]
        flips += ch["flip"]
        z = host(out["logits"])
        assert np.all(np.abs(z.astype(np.float64) - ch["z"]) <= ATOL + RTOL * np.abs(ch["z"]))
        np.testing.assert_array_equal(gd, ch["tokens"])
        target = (np.concatenate([ch["z"], ch["z"][:, -1:]], axis=1) + st["noise"]).astype(np.float32)
        ver = oracle.verify(0, target, ch["tokens"])
        a, n = ds.verify(0, dev(target), out["draft_tokens"])
        assert host(a)[0] == ver["accepted_len"][0] and host(n)[0] == ver["next_token"][0]
        prev = host(n).astype(np.int32)   # the GPU's own output feeds the next step
    parity_log.record("tiny 8 chained steps (greedy)", "position", cfg["steps"] * B * k,
                      near_tie=near, flip=flips)


# ----------------------------------------------------------------------------- sweep corners

@pytest.mark.parametrize("B,k,r", [(64, 7, 128), (32, 4, 32), (8, 6, 128), (2, 7, 32)])
def test_sweep_chain_and_verify(B, k, r):
    V = 151936
    w1 = syn.normal_bf16(3, (V, r))
    w2 = syn.normal_bf16(4, (V, r), (1.0 / r) ** 0.5)
    logits = syn.uniform_logits(800 + B * r + k, (B, k, V), 1.0)
    prev = syn.step_inputs(2, B, k, 64, 1, V, ("const", 1.0))["prev"]
    ref = oracle.greedy_sample(logits, w1, w2, prev)
    lg = dev(logits)
    d, qs = ds.greedy_sample(lg, dev_bf16(w1), dev_bf16(w2), dev(prev))
    np.testing.assert_array_equal(host(d), ref["draft_tokens"])
    np.testing.assert_array_equal(host(lg), ref["z"])
    sig = np.full(k + 1, 2.0 if B % 2 == 0 else 0.5, np.float32)
    target = (np.concatenate([ref["z"], ref["z"][:, -1:]], axis=1)
              + syn.uniform_logits(900 + B, (B, k + 1, V), 1.0) * sig[None, :, None]).astype(np.float32)
    ver = oracle.verify(1, target, ref["draft_tokens"], None, ref["z"], seed=5, step=1)
    a, n = ds.verify(1, dev(target), d, None, lg, qs, seed=5, step=1)
    ex_a, ex_d = decision_mask(ver)
    ex = ex_a | ex_d
    parity_log.record("sweep B=%d k=%d r=%d chain + verify(prob)" % (B, k, r), "request", B,
                      accept=ex_a.sum(), draw=ex_d.sum())
    assert ex.sum() <= max(1, B // 16)
    np.testing.assert_array_equal(host(a)[~ex], ver["accepted_len"][~ex])
    np.testing.assert_array_equal(host(n)[~ex], ver["next_token"][~ex])


@pytest.mark.parametrize("M", [448, 256, 257])
def test_large_batch_lm_head_tiles(M):
    """B*k above one 256-row tile (two N tiles of 224, ragged 257) on a vocab slice."""
    H, V = 5120, 20000
    h = syn.normal_bf16(40 + M, (M, H))
    w = syn.normal_bf16(41, (V, H), (1.0 / H) ** 0.5)
    got = host(ds.lm_head(dev_bf16(h), dev_bf16(w)))
    rows = np.sort(np.random.default_rng(M).choice(V, 600, replace=False))
    ref = oracle.lm_head(h, w[rows])
    assert np.all(np.abs(got[:, rows].astype(np.float64) - ref) <= ATOL + RTOL * np.abs(ref))
