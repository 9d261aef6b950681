#!/usr/bin/env python3
"""Draft+verify step benchmark of the GB300 DSpark readout + verify path.

One step = the whole hot path for one batch: fc projection of the 5 tapped hidden
states -> LM head over every block position -> Markov-biased semi-autoregressive
greedy drafting (k positions) -> [confidence truncation] -> verification against the
target logits.  Every step goes through the C ABI (libdspark.so).

Prints ONE JSON line (rank 0).  Default workload: Qwen3.8-27B-DSpark shapes at batch 1
(H=5120, 5 taps, V=151936, r=64, k=7, probabilistic verify).  Weights are random-init
and inputs synthetic (seeded); see synthetic.py for the recipe.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Under torchrun (N > 1) every rank runs an independent replica on its own requests
(the path has no cross-request exchange); value = all ranks' steps / max time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as syn  # noqa: E402

METRIC = "draft+verify steps/sec and drafted tok/s at batch 1/16; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------------------- helpers

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="27b_b1", choices=sorted(syn.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", type=int, default=None, help="verify mode override (0 greedy, 1 prob)")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sets", type=int, default=3,
                    help="minimum input sets rotated across steps (more are used when needed "
                         "to exceed 2x the L2 cache)")
    ap.add_argument("--no-backbone", action="store_true",
                    help="leave out the 27B batch-1 sub-record with one drafter backbone layer")
    ap.add_argument("--profile-sets", type=int, default=0,
                    help="profiling runs only: rotate this many input sets instead of enough to "
                         "exceed 2x the L2 cache (fewer set-up launches before the profiled ones)")
    ap.add_argument("--min-time", type=float, default=1.0,
                    help="seconds of repeated K-step timed loops (the median loop is reported)")
    ap.add_argument("--no-b16", action="store_true",
                    help="27b_b1: skip the batch-16 sub-record")
    ap.add_argument("--no-graph", action="store_true", help="time un-captured steps only")
    ap.add_argument("--sweep", action="store_true",
                    help="run the 27B sweep grid instead (one JSON line per cell, not the "
                         "headline line): B x k x r x sigma, probabilistic verify")
    ap.add_argument("--sweep-steps", type=int, default=200, help="timed steps per sweep cell")
    ap.add_argument("--fused-gemms", action="store_true",
                    help="bf16 weights: run the fc and the LM head as one two-phase GEMM "
                         "launch (dspark_fc_lm_head) instead of two launches")
    ap.add_argument("--q-stats", default="verify", choices=["verify", "chain"],
                    help="where the softmax statistics of q are reduced: in verify's row-"
                         "statistics launch (with the target rows), or in the Markov chain kernel")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def replica_step_seed(step, rank):
    """Input-set seed of a replica: every rank drafts for its own requests."""
    return step + 100 * rank


def max_over_ranks(x, world, device=None):
    """The slowest rank's value (timings are taken as the max over ranks)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_seconds):
    """Units all ranks processed divided by the slowest rank's time."""
    return world * units_per_rank / max_seconds


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, tflops, src = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"
    try:
        with open(path) as f:
            d = json.load(f)
        flat = {}

        def walk(x, pre=""):
            if isinstance(x, dict):
                for kk, vv in x.items():
                    walk(vv, pre + kk + ".")
            else:
                flat[pre[:-1]] = x
        walk(d)
        for kk, vv in flat.items():
            if isinstance(vv, (int, float)) and "hbm" in kk.lower() and "gbs" in kk.lower():
                hbm, src = float(vv), "measured"
                break
        for kk, vv in flat.items():
            if isinstance(vv, (int, float)) and kk.lower().endswith("bf16_tflops"):
                tflops = float(vv)
                break
    except (OSError, ValueError):
        pass
    return hbm, tflops, src


def profiled_traffic(workload, stem="gemm_tcgen05_lm_head"):
    """DRAM bytes per LM-head launch from the committed ncu summary of this workload,
    or None when there is none or the kernel source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (stem, workload))
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith(("|", "#", " ")):
                    key, _, val = line.partition(":")
                    fields[key.strip()] = val.strip()
        src = os.path.join(ROOT, fields["source"])
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if sha != fields["source_sha256_16"]:
            return None
        return int(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def step_bytes(cfg, mode):
    """Algorithmic bytes of one step: each weight once, activations, the fp32 draft
    logits written once, the target logits read, one resample row pair per request."""
    B, k, H, T, V, r = (cfg[x] for x in ("B", "k", "H", "T", "V", "r"))
    M = B * k
    if cfg.get("fp8"):
        # E4M3 weights + fp32 row scales; the activation rows are read as bf16, their codes
        # written and read back once, their scales are negligible
        fc = H * T * H + H * 4 + T * M * H * 2 + 2 * T * M * H + M * H * 2
        lm = V * H + V * 4 + M * H * 2 + 2 * M * H + M * V * 4
    else:
        fc = H * T * H * 2 + T * M * H * 2 + M * H * 2
        lm = V * H * 2 + M * H * 2 + M * V * 4
    chain = V * r * 2
    verify = B * (k + 1) * V * 4 + (B * 2 * V * 4 if mode == 1 else 0)
    bb = backbone_bytes(cfg)
    return {"fc": fc, "backbone": bb, "lm_head": lm, "chain": chain, "verify": verify,
            "total": fc + bb + lm + chain + verify}


def backbone_bytes(cfg):
    """Drafter backbone: each layer's weights once, its key/value cache read once (the
    C context rows and the k + 1 block rows), the block's embedding rows."""
    if not cfg.get("backbone"):
        return 0
    B, k, H = cfg["B"], cfg["k"], cfg["H"]
    g, L, C = syn.BACKBONE_GEOMETRY[H], cfg["backbone"]["L"], cfg["backbone"]["C"]
    nq, nkv, I = g["nq"], g["nkv"], g["I"]
    weights = ((nq + 2 * nkv) * 128 * H + H * nq * 128 + 2 * I * H + H * I + 2 * H + 256) * 2
    cache = B * (C + k + 1) * nkv * 128 * 2 * 2
    return L * (weights + cache) + B * (k + 1) * H * 2


def step_flops(cfg):
    B, k, H, T, V, r = (cfg[x] for x in ("B", "k", "H", "T", "V", "r"))
    M = B * k
    f = 2 * M * (T * H * H + V * H + V * r)
    if cfg.get("backbone"):
        g, L, C = syn.BACKBONE_GEOMETRY[H], cfg["backbone"]["L"], cfg["backbone"]["C"]
        nq, nkv, I = g["nq"], g["nkv"], g["I"]
        rows = B * (k + 1)
        per_layer = (2 * rows * ((nq + 2 * nkv) * 128 * H + H * nq * 128 + 3 * I * H)
                     + 2 * M * 2 * nkv * 128 * H                        # the context rows' K/V
                     + 4 * rows * nq * 128 * (C + k + 1))               # scores and P.V
        f += L * per_layer
    return f


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = "/tmp/dspark_clocks_%d_%d.csv" % (os.getpid(), gpu_index)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- CPU oracle sample

def oracle_sample_step(ora, host, cfg, mode, frac, step):
    """The oracle's whole step restricted to a fraction of the output columns of fc and of
    the vocabulary (LM head rows, chain, verify), so its cost is about frac x a full step.
    Returns seconds."""
    B, k, H, V = cfg["B"], cfg["k"], cfg["H"], cfg["V"]
    nh = max(1, int(round(frac * H)))
    nv = max(8, int(round(frac * V)))
    t0 = time.perf_counter()
    if cfg.get("fp8"):
        ora.fc_project_fp8(host["taps"], host["fc_w8"][:nh], host["fc_s"][:nh])
    else:
        ora.fc_project(host["taps"], host["fc_w"][:nh])  # fc over nh output columns
    t1 = time.perf_counter()
    if cfg.get("fp8"):
        logits = ora.lm_head_fp8(host["h"], host["lm_w8"][:nv], host["lm_s"][:nv]).reshape(B, k, nv)
    else:
        logits = ora.lm_head(host["h"], host["lm_w"][:nv]).reshape(B, k, nv)
    prev = (host["prev"] % nv).astype(np.int32)
    gs = ora.greedy_sample(logits, host["w1"][:nv], host["w2"][:nv], prev)
    tgt = np.ascontiguousarray(host["target"][:, :, :nv])
    ora.verify(mode, tgt, gs["draft_tokens"], None, gs["z"] if mode == 1 else None, seed=0,
               step=step)
    t2 = time.perf_counter()
    # the fc slice costs nh/H of the fc; the rest nv/V of its full cost
    return (t1 - t0) * (H / nh) + (t2 - t1) * (V / nv)


def cpu_oracle_baseline(host, cfg, mode, budget_s, steps=None):
    """Times the oracle (as it stands) on bounded samples of the workload; returns
    (full steps/s extrapolated from the samples, cores, sample description, n)."""
    import oracle as ora
    # calibrate: one small sample
    est = oracle_sample_step(ora, host, cfg, mode, 1.0 / 256, 0)
    per_sample = budget_s / (steps if steps else 8)
    frac = min(1.0, max(1.0 / 512, per_sample / max(est, 1e-6)))
    n = steps if steps else 0
    full_times = []
    t_start = time.perf_counter()
    i = 0
    while True:
        full_times.append(oracle_sample_step(ora, host, cfg, mode, frac, i + 1))
        i += 1
        if steps is not None and i >= steps:
            break
        if steps is None and time.perf_counter() - t_start > budget_s and i >= 2:
            break
    mean_full = statistics.mean(full_times)
    desc = ("%d oracle samples, each the whole step on %.4f of the fc output columns and of the "
            "vocabulary (LM head rows, Markov chain, verify), scaled to a full step"
            % (len(full_times), frac))
    return 1.0 / mean_full, ora.num_threads(), desc, len(full_times)


def host_workload(cfg):
    """Host copies of the weights and one step's inputs (for the CPU baseline)."""
    import oracle as ora
    B, k, H, T, V, r = (cfg[x] for x in ("B", "k", "H", "T", "V", "r"))
    w = syn.weights(H, T, V, r, with_conf=cfg["conf"])
    st = syn.step_inputs(0, B, k, H, T, V, cfg["sigma"])
    # target logits: the oracle's own draft logits (on the vocabulary) plus noise
    host = {"taps": st["taps"], "fc_w": w["fc_w"], "lm_w": w["lm_w"], "w1": w["w1"],
            "w2": w["w2"], "prev": st["prev"]}
    add_host_fp8(ora, host, cfg)
    host["h"] = oracle_h(ora, host, cfg)
    host["target"] = st["noise"]  # noise alone stands in: the cost does not depend on values
    return host


def add_host_fp8(ora, host, cfg):
    """FP8 workloads: the oracle's own E4M3 codes and row scales of the fc and LM-head
    weights (the bf16 copies are then dropped)."""
    if cfg.get("fp8"):
        host["fc_w8"], host["fc_s"] = ora.quantize_fp8_rows(host.pop("fc_w"))
        host["lm_w8"], host["lm_s"] = ora.quantize_fp8_rows(host.pop("lm_w"))


def oracle_h(ora, host, cfg):
    if cfg.get("fp8"):
        return ora.fc_project_fp8(host["taps"], host["fc_w8"], host["fc_s"])
    return ora.fc_project(host["taps"], host["fc_w"])


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    cfg = dict(syn.CONFIGS[args.config])
    mode = cfg["mode"] if args.mode is None else args.mode
    host = host_workload(cfg)
    budget = 150.0
    import oracle as ora
    est = oracle_sample_step(ora, host, cfg, mode, 1.0 / 256, 0)
    # size the sample so that warmup + steps finish within the budget
    per_step = budget / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1.0 / 4096, per_step / max(est, 1e-9)))
    for i in range(args.warmup):
        oracle_sample_step(ora, host, cfg, mode, frac, i)
    t0 = time.perf_counter()
    full = [oracle_sample_step(ora, host, cfg, mode, frac, args.warmup + i) for i in range(args.steps)]
    wall = time.perf_counter() - t0
    sps = 1.0 / statistics.mean(full)
    desc = ("each step: the oracle's whole step on %.5f of the fc output columns and of the "
            "vocabulary, scaled to a full step" % frac)
    line = {
        "impl": "reference", "metric": METRIC, "value": sps, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / sps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "wall_s": wall,
        "config": config_of(args.config, cfg, mode, args, world),
        "cpu_baseline": {"value": sps, "unit": "steps/s", "cores": ora.num_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": sps, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm

def n_input_sets(cfg, min_sets, l2_bytes):
    """Input sets rotated across steps: at least min_sets and enough that their per-step
    inputs (taps, prev tokens, target logits) exceed 2.2x the L2 cache, so no step finds
    its inputs in L2 (the 1.8-2.2 GB of weights stream from HBM every step anyway)."""
    B, k, H, T, V = (cfg[x] for x in ("B", "k", "H", "T", "V"))
    per_set = T * B * k * H * 2 + B * 4 + B * (k + 1) * V * 4
    need = -(-int(2.2 * l2_bytes) // per_set)
    return int(min(256, max(min_sets, need))), per_set


def timing_events_supported(torch):
    """Timing events that become event-record nodes when captured in a CUDA graph."""
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


class Pipeline:
    """One draft+verify step through the C ABI.

    draft(): fc -> LM head -> Markov chain [-> confidence] on one stream.
    verify(): the verify of those drafts (row statistics of the target rows, and of the
    draft-logit rows unless the chain reduced q's statistics, then the decision/draw
    kernel) on a given stream.  A serial step runs both on one stream; the decode loop
    of `measure_workload` runs the verify of step i on a second stream beside the fc
    and LM head of step i + 1 (two Pipelines, alternating buffers)."""

    def __init__(self, ds, torch, device, cfg, mode, w, args):
        self.ds, self.torch, self.dev = ds, torch, device
        self.cfg, self.mode, self.w = cfg, mode, w
        B, k, H, V = cfg["B"], cfg["k"], cfg["H"], cfg["V"]
        M = B * k
        self.fp8 = bool(cfg.get("fp8"))
        self.fused = (not self.fp8) and args.fused_gemms
        self.q_in = args.q_stats
        f32, i32 = torch.float32, torch.int32
        self.h = torch.empty((M, H), dtype=torch.bfloat16, device=device)
        self.logits = torch.empty((B, k, V), dtype=f32, device=device)
        self.drafts = torch.empty((B, k), dtype=i32, device=device)
        self.q_stats = torch.empty((B, k, 2), dtype=f32, device=device) if mode == 1 else None
        # drafter backbone (N1): the fc output becomes the context rows; the block
        # (the previous token, then k mask tokens) runs through the layers into hb
        self.bb = w.get("bb_layers")
        if self.bb:
            self.C = cfg["backbone"]["C"]
            self.tokens = torch.full((B, k + 1), V - 1, dtype=i32, device=device)
            self.hb = torch.empty((M, H), dtype=torch.bfloat16, device=device)
        self.wsp = ds.Workspaces()          # drafting calls
        self.wsp_v = ds.Workspaces()        # verify calls (may run beside the next drafting)

    def chain_q(self):
        return self.mode == 1 and self.q_in == "chain"

    def stage_names(self):
        """The stages between consecutive timing events of a step."""
        if self.fused:
            return ["fc_lm_head", "(none)", "greedy_sample", "verify"]
        if self.bb:
            return ["fc_project", "backbone", "lm_head", "greedy_sample", "verify"]
        return ["fc_project", "lm_head", "greedy_sample", "verify"]

    def backbone(self, prev, s):
        """The fc output (self.h) as the newest k context rows of every layer's cache,
        then the block through the layers; returns the LM head's input."""
        ds, w, k = self.ds, self.w, self.cfg["k"]
        with self.torch.cuda.stream(s):
            self.tokens[:, 0].copy_(prev)
        return ds.backbone_block(self.tokens, w["lm_w"], self.bb, w["bb_final"], w["bb_kc"], w["bb_vc"], self.C,
                                 out=self.hb, stream=s, workspaces=self.wsp, ctx=self.h, ctx_pos0=self.C - k)

    def draft(self, st, s, hist, ev=None, chain_after=None):
        """ev: timing events on s at the stage boundaries (start, after fc, [after the
        backbone,] after LM head, after chain; one more for verify).
        chain_after: an event the chain waits for (the previous step's verify)."""
        ds, w, cfg = self.ds, self.w, self.cfg
        B, k, V = cfg["B"], cfg["k"], cfg["V"]
        M = B * k
        dlen_o = hist[2]
        if ev is not None:
            ev[0].record(s)
        if self.fused:
            ds.fc_lm_head(st["taps"], w["fc_w"], w["lm_w"], h_out=self.h, logits=self.logits.view(M, V),
                          stream=s, workspaces=self.wsp)
            if ev is not None:
                ev[1].record(s)
        else:
            if self.fp8:
                ds.fc_project_fp8(st["taps"], w["fc_w8"], w["fc_s"], out=self.h, stream=s, workspaces=self.wsp)
            else:
                ds.fc_project(st["taps"], w["fc_w"], out=self.h, stream=s, workspaces=self.wsp)
            if ev is not None:
                ev[1].record(s)
            h_lm = self.h
            if self.bb:
                h_lm = self.backbone(st["prev"], s)
                if ev is not None:
                    ev[2].record(s)
            if self.fp8:
                ds.lm_head_fp8(h_lm, w["lm_w8"], w["lm_s"], out=self.logits.view(M, V), stream=s,
                               workspaces=self.wsp)
            else:
                ds.lm_head(h_lm, w["lm_w"], out=self.logits.view(M, V), stream=s, workspaces=self.wsp)
        if ev is not None:
            ev[-3].record(s)
        if chain_after is not None:
            s.wait_event(chain_after)
        ds.greedy_sample(self.logits, w["w1"], w["w2"], st["prev"], draft_tokens=self.drafts,
                         q_stats=self.q_stats if self.chain_q() else None, want_q_stats=self.chain_q(),
                         stream=s, workspaces=self.wsp)
        if w.get("conf_w") is not None:
            ds.confidence_truncate(self.hb if self.bb else self.h, w["conf_w"], self.drafts, B, k, 0.0, 0.5,
                                   draft_len=dlen_o, stream=s)
        if ev is not None:
            ev[-2].record(s)

    def verify(self, st, s, hist, step_id, ev=None):
        acc_o, nxt_o, dlen_o = hist
        dl = dlen_o if self.w.get("conf_w") is not None else None
        self.ds.verify(self.mode, st["target"], self.drafts, dl, self.logits if self.mode == 1 else None,
                       self.q_stats if self.chain_q() else None, seed=12345, request_id=None,
                       step=step_id, accepted_len=acc_o, next_token=nxt_o, stream=s,
                       workspaces=self.wsp_v)
        if ev is not None:
            ev.record(s)

    def step(self, st, s, hist, step_id, ev=None):
        """A serial step: draft and verify on stream s (ev: 5 timing events)."""
        self.draft(st, s, hist, ev)
        self.verify(st, s, hist, step_id, ev[-1] if ev is not None else None)


def load_weights(ds, torch, device, cfg, host_cache):
    """Device weights of a workload (bf16, or E4M3 codes + row scales), from seeded host
    draws shared between workloads of the same shapes."""
    H, T, V, r = cfg["H"], cfg["T"], cfg["V"], cfg["r"]
    key = (H, T, V, r)
    if key not in host_cache:
        host_cache.clear()
        host_cache[key] = syn.weights(H, T, V, r, with_conf=True)
    hw = host_cache[key]

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    w = {"w1": d16(hw["w1"]), "w2": d16(hw["w2"]), "conf_w": d16(hw["conf_w"]) if cfg["conf"] else None}
    fc_w, lm_w = d16(hw["fc_w"]), d16(hw["lm_w"])
    if cfg.get("fp8"):
        w["fc_w8"], w["fc_s"] = ds.quantize_fp8(fc_w)
        w["lm_w8"], w["lm_s"] = ds.quantize_fp8(lm_w)
        torch.cuda.synchronize()
        del fc_w, lm_w
    else:
        w["fc_w"], w["lm_w"] = fc_w, lm_w
    if cfg.get("backbone"):
        bbc, g = cfg["backbone"], syn.BACKBONE_GEOMETRY[H]
        bkey = ("backbone", H, bbc["L"])
        if bkey not in host_cache:
            host_cache[bkey] = syn.backbone_weights(H, g["nq"], g["nkv"], g["I"], bbc["L"])
        layers, wf = host_cache[bkey]
        w["bb_layers"] = [ds.BackboneLayer(l["nq"], l["nkv"], *[d16(l[x]) for x in (
            "w_in", "w_post", "w_qn", "w_kn", "w_qkv", "w_o", "w_gu", "w_d")]) for l in layers]
        w["bb_final"] = d16(wf)
        # each layer's key/value cache: a synthetic context of C tokens (unit-scale keys
        # and values, as the k-norm leaves them), then room for the k + 1 block rows;
        # every step writes its k new context rows over the newest k context slots
        shape = (cfg["B"], bbc["C"] + cfg["k"] + 1, g["nkv"], 128)
        w["bb_kc"] = [d16(syn.normal_bf16(900 + li, shape)) for li in range(bbc["L"])]
        w["bb_vc"] = [d16(syn.normal_bf16(950 + li, shape)) for li in range(bbc["L"])]
    return w


def measure_workload(args, name, rank, local_rank, world, host_cache, with_cpu_baseline):
    """Times one workload.

    Headline: a decode loop of K steps captured in one CUDA graph, where the verify of
    step i runs on a second stream beside the fc and LM head of step i + 1 (which need
    only the target forward's outputs) and the Markov chain of step i + 1 waits for
    that verify (its context is the verified token).  The K-step loop is replayed for
    at least --min-time seconds and the median loop is reported.  Also: serial steps
    (draft and verify on one stream, one CUDA graph per step), per-stage times from
    serial graphs carrying timing events, the un-captured serial loop, and the
    end-to-end leg with host buffers."""
    import torch
    import torch.distributed as dist

    import speculative_decoding_fc_gb300 as ds

    device = torch.device("cuda", local_rank)
    cfg = dict(syn.CONFIGS[name])
    mode = cfg["mode"] if args.mode is None else args.mode
    B, k, H, T, V, r = (cfg[x] for x in ("B", "k", "H", "T", "V", "r"))
    M = B * k
    w = load_weights(ds, torch, device, cfg, host_cache)
    pipes = [Pipeline(ds, torch, device, cfg, mode, w, args) for _ in range(2)]
    pipe = pipes[0]
    stream = torch.cuda.current_stream(device)
    vstream = torch.cuda.Stream(device)
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 129 << 20) or (129 << 20))
    nsets, set_bytes = n_input_sets(cfg, args.sets, l2)
    if args.profile_sets > 0:
        nsets = args.profile_sets

    # input sets: taps, prev, target logits = own draft logits + noise (built once)
    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    sets = []
    for si in range(nsets):
        st = syn.step_inputs(replica_step_seed(si, rank), B, k, H, T, V, cfg["sigma"])
        dev_set = {"taps": [d16(t) for t in st["taps"]], "prev": torch.from_numpy(st["prev"]).to(device)}
        # the drafter's own biased logits on this set, then the target = those + noise
        if pipe.fp8:
            h = ds.fc_project_fp8(dev_set["taps"], w["fc_w8"], w["fc_s"])
            lg = ds.lm_head_fp8(h, w["lm_w8"], w["lm_s"]).view(B, k, V)
        else:
            h = ds.fc_project(dev_set["taps"], w["fc_w"])
            if pipe.bb:
                pipe.h.copy_(h)
                h = pipe.backbone(dev_set["prev"], stream).clone()
            lg = ds.lm_head(h, w["lm_w"]).view(B, k, V)
        ds.greedy_sample(lg, w["w1"], w["w2"], dev_set["prev"], want_q_stats=False)
        noise = torch.from_numpy(st["noise"]).to(device)
        dev_set["target"] = (torch.cat([lg, lg[:, -1:]], dim=1) + noise).contiguous()
        dev_set["host"] = st if si == 0 else None
        del h, lg, noise
        sets.append(dev_set)
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    acc_hist = torch.zeros((K + W, B), dtype=torch.int32, device=device)
    nxt_hist = torch.zeros((K + W, B), dtype=torch.int32, device=device)
    dlen_hist = torch.zeros((K + W, B), dtype=torch.int32, device=device)

    def hist(i):
        return acc_hist[i], nxt_hist[i], dlen_hist[i]

    for i in range(W):
        pipe.step(sets[i % nsets], stream, hist(K + i), K + i)
    torch.cuda.synchronize()

    def decode_loop(s, sv, first, nsteps, hist_of):
        """nsteps consecutive steps from input set `first`: step i drafts on s with the
        buffers of pipes[i % 2]; its verify runs on sv once its drafts exist; the chain
        of step i + 1 waits for it, the fc and LM head of step i + 1 do not (they only
        wait, before overwriting the buffers of step i - 1, for that step's verify)."""
        done_d = [torch.cuda.Event(), torch.cuda.Event()]
        done_v = [torch.cuda.Event(), torch.cuda.Event()]
        for i in range(nsteps):
            p = pipes[i % 2]
            st = sets[(first + i) % nsets]
            if i >= 2:
                s.wait_event(done_v[i % 2])      # step i - 2's verify read these buffers
            h_ = hist_of(i)
            # fc + LM head, then the chain once the previous step's verify is done
            p.draft(st, s, h_, chain_after=done_v[(i - 1) % 2] if i >= 1 else None)
            done_d[i % 2].record(s)
            sv.wait_event(done_d[i % 2])
            p.verify(st, sv, h_, i)
            done_v[i % 2].record(sv)
        s.wait_event(done_v[(nsteps - 1) % 2])   # the loop ends with its last verify
        if nsteps >= 2:
            s.wait_event(done_v[(nsteps - 2) % 2])

    # ---------------------------------------------------------------- CUDA graphs
    graphs, loops, staged, graph_error = None, None, None, None
    launches_per_step = None
    ev_ok = timing_events_supported(torch)
    nloops = max(1, -(-nsets // K))
    if not args.no_graph:
        try:
            cap = torch.cuda.Stream(device)
            capv = torch.cuda.Stream(device)
            cap.wait_stream(stream)
            ghist = tuple(torch.zeros((B,), dtype=torch.int32, device=device) for _ in range(3))
            # serial: one graph per input set
            graphs = []
            for st in sets:
                g = torch.cuda.CUDAGraph()
                n0 = ds.launch_count()
                with torch.cuda.graph(g, stream=cap):
                    pipe.step(st, cap, ghist, 0)
                launches_per_step = ds.launch_count() - n0
                graphs.append(g)
            # decode loop: K steps per graph, consecutive graphs start at later sets
            lhist = [tuple(torch.zeros((B,), dtype=torch.int32, device=device) for _ in range(3))
                     for _ in range(2)]
            loops = []
            for li in range(nloops):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    capv.wait_stream(cap)
                    decode_loop(cap, capv, li * K, K, lambda i: lhist[i % 2])
                loops.append(g)
            if ev_ok:
                # serial steps with timing events at the stage boundaries (event-record
                # nodes), for the per-stage times of graph replays
                staged = []
                for st in sets:
                    g = torch.cuda.CUDAGraph()
                    ev = [torch.cuda.Event(enable_timing=True, external=True)
                          for _ in range(len(pipe.stage_names()) + 1)]
                    with torch.cuda.graph(g, stream=cap):
                        pipe.step(st, cap, ghist, 0, ev=ev)
                    staged.append((g, ev))
            stream.wait_stream(cap)
            for g in graphs + loops:      # one untimed replay each
                g.replay()
            torch.cuda.synchronize()
        except Exception as exc:  # noqa: BLE001 - fall back to un-captured timing
            graphs, loops, staged, graph_error = None, None, None, str(exc).splitlines()[0][:200]
            torch.cuda.synchronize()

    def timed(run_steps):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        run_steps()
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return max_over_ranks(t0.elapsed_time(t1), world, device)

    def repeat(run_steps, seconds):
        """K-step timed loops until `seconds` have elapsed (at least 3): their times."""
        out = []
        t_start = time.perf_counter()
        while True:
            out.append(timed(run_steps))
            done = time.perf_counter() - t_start >= seconds and len(out) >= 3
            if world > 1:
                done = max_over_ranks(1.0 if done else 0.0, world, device) > 0.5
            if done:
                return out

    rep_no = [0]

    def run_loop():
        loops[rep_no[0] % len(loops)].replay()
        rep_no[0] += 1

    def run_graphs():
        for i in range(K):
            graphs[i % nsets].replay()

    def run_plain():
        for i in range(K):
            pipe.step(sets[i % nsets], stream, hist(i), i)

    # the headline: the decode loop (K steps per replay), repeated for --min-time
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.1)
    if loops is not None:
        rep_ms = repeat(run_loop, args.min_time)
        launches = launches_per_step * K
    else:
        n0 = ds.launch_count()
        rep_ms = repeat(run_plain, args.min_time)
        launches = (ds.launch_count() - n0) // len(rep_ms)
    clk = clocks.stop()
    max_ms = statistics.median(rep_ms)
    serial_ms = statistics.median(repeat(run_graphs, 0.25)) if graphs is not None else max_ms
    plain_ms = timed(run_plain)

    # per-stage times: replays of the serial graphs with timing events (passes over all
    # input sets, back to back, read after each pass); else the un-captured loop
    stage_names = pipe.stage_names()
    samples = {nm: [] for nm in stage_names}
    samples["step"] = []
    if staged is not None:
        stage_src = "serial CUDA-graph replays (event-record nodes at the stage boundaries)"
        t_s = time.perf_counter()
        while len(samples["step"]) < 200 or time.perf_counter() - t_s < 0.3:
            for g, _ in staged:
                g.replay()
            torch.cuda.synchronize()
            for _, ev in staged:
                for j, nm in enumerate(stage_names):
                    samples[nm].append(ev[j].elapsed_time(ev[j + 1]))
                samples["step"].append(ev[0].elapsed_time(ev[-1]))
            if time.perf_counter() - t_s > 5.0:
                break
    else:
        stage_src = "un-captured serial loop with CUDA events (host launch cost included)"
        for i in range(K):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
            pipe.step(sets[i % nsets], stream, hist(i), i, ev=ev)
            torch.cuda.synchronize()
            for j, nm in enumerate(stage_names):
                samples[nm].append(ev[j].elapsed_time(ev[j + 1]))
            samples["step"].append(ev[0].elapsed_time(ev[-1]))
    stage_ms = {nm: statistics.median(v) for nm, v in samples.items() if v and nm != "(none)"}
    lm_ms = stage_ms["fc_lm_head"] if pipe.fused else stage_ms["lm_head"]

    # ---------------------------------------------------------------- end to end (host buffers)
    Ke = min(args.e2e_steps, K)
    st0 = sets[0]
    pin_taps = torch.empty((T, M, H), dtype=torch.bfloat16).pin_memory()
    for j in range(T):
        pin_taps[j].copy_(st0["taps"][j].cpu())
    pin_prev = st0["prev"].cpu().pin_memory()
    pin_target = st0["target"].cpu().pin_memory()
    out_acc = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_nxt = torch.empty((B,), dtype=torch.int32).pin_memory()
    out_drafts = torch.empty((B, k), dtype=torch.int32).pin_memory()
    dev_taps = torch.empty((T, M, H), dtype=torch.bfloat16, device=device)
    dev_prev = torch.empty((B,), dtype=torch.int32, device=device)
    dev_target = torch.empty_like(st0["target"])
    e2e_set = {"taps": [dev_taps[j] for j in range(T)], "prev": dev_prev, "target": dev_target}
    h2d = pin_taps.numel() * 2 + pin_prev.numel() * 4 + pin_target.numel() * 4
    d2h = (2 * B + B * k) * 4
    # The readout's inputs (taps, previous tokens) go to the device first; the target
    # logits follow on a side stream, under the readout (queued behind the small copies:
    # on one copy engine the 78 MB of batch-16 logits ahead of them held the readout back
    # by their whole transfer); verify waits for them.  The host reads every step's
    # result before the next step.
    copy_stream = torch.cuda.Stream(device)
    target_ready = torch.cuda.Event()

    def e2e_step(s, i):
        with torch.cuda.stream(s):
            dev_taps.copy_(pin_taps, non_blocking=True)
            dev_prev.copy_(pin_prev, non_blocking=True)
        copy_stream.wait_stream(s)
        with torch.cuda.stream(copy_stream):
            dev_target.copy_(pin_target, non_blocking=True)
            target_ready.record(copy_stream)
        pipe.draft(e2e_set, s, hist(i))
        s.wait_event(target_ready)
        pipe.verify(e2e_set, s, hist(i), i)
        with torch.cuda.stream(s):
            out_acc.copy_(acc_hist[i], non_blocking=True)
            out_nxt.copy_(nxt_hist[i], non_blocking=True)
            out_drafts.copy_(pipe.drafts, non_blocking=True)

    def e2e_time(run_one):
        wall = 0.0
        for rep in range(2):
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            n = 3 if rep == 0 else Ke
            t0 = time.perf_counter()
            for i in range(n):
                run_one(i)
                stream.synchronize()  # the host reads this step's result
            wall = time.perf_counter() - t0
        return whole_job_rate(Ke, world, max_over_ranks(wall, world, device))

    e2e_plain = e2e_time(lambda i: e2e_step(stream, i))
    # The same step (copies in, readout, verify, results out) captured once as a CUDA
    # graph, as a serving loop would run it: one graph launch per step, the host still
    # reading every step's result before the next.
    e2e_graph = None
    try:
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=cap):
            e2e_step(cap, 0)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        e2e_graph = e2e_time(lambda i: g_e2e.replay())
    except Exception:  # noqa: BLE001 - report the un-captured loop alone
        torch.cuda.synchronize()
    e2e = {"value": e2e_graph if e2e_graph is not None else e2e_plain, "unit": "steps/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "how": ("each step one CUDA-graph replay of the public-API calls (pinned-host copies in, "
                   "readout, verify, results out), then a host read of the results"
                   if e2e_graph is not None else "each step the public-API calls launched from the host, "
                   "then a host read of the results"),
           "uncaptured": e2e_plain}

    # ---------------------------------------------------------------- acceptance statistics
    acc = acc_hist[:K].cpu().numpy()
    drafted = float(dlen_hist[:K].cpu().numpy().sum()) / K if cfg["conf"] else float(B * k)
    mean_acc_len = float(acc.mean()) + 1.0   # accepted drafts + the bonus/corrected token
    per_pos = [float((acc > j).mean()) for j in range(k)]

    steps_per_s = whole_job_rate(K, world, max_ms / 1000.0)
    peak_gbs, peak_tf, peak_src = measured_peaks()
    sb = step_bytes(cfg, mode)
    lm_bytes = sb["fc"] + sb["lm_head"] if pipe.fused else sb["lm_head"]
    achieved = lm_bytes / (lm_ms / 1000.0) / 1e9
    t_roof = max(sb["total"] / (peak_gbs * 1e9), step_flops(cfg) / (peak_tf * 1e12))
    t_readout = max((sb["fc"] + sb["backbone"] + sb["lm_head"] + sb["chain"]) / (peak_gbs * 1e9),
                    step_flops(cfg) / (peak_tf * 1e12))
    t_verify = sb["verify"] / (peak_gbs * 1e9)
    readout_ms = ((stage_ms["fc_lm_head"] if pipe.fused else stage_ms["fc_project"] + stage_ms["lm_head"])
                  + stage_ms.get("backbone", 0.0) + stage_ms["greedy_sample"])
    traffic_file = "gemm_tcgen05_fc_lm_head" if pipe.fused else "gemm_tcgen05_lm_head"
    traffic = profiled_traffic(name, traffic_file)
    step_roof = {"bytes": sb["total"], "flops": step_flops(cfg), "t_roofline_ms": t_roof * 1000.0,
                 "frac": (t_roof * 1000.0) / (max_ms / K), "peak_source": peak_src,
                 "serial_frac": (t_roof * 1000.0) / (serial_ms / K),
                 "readout_frac": t_readout * 1000.0 / readout_ms,
                 "verify_frac": t_verify * 1000.0 / stage_ms["verify"],
                 "verify_frac_is": "the serial step's verify (row statistics, decision, draw) "
                                   "against its own algorithmic bytes",
                 "stage_times": stage_src}
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": max_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if pipe.fp8 else "bf16",
        "data": "synthetic",
        "config": config_of(name, cfg, mode, args, world, nsets, set_bytes, l2,
                            weights_bytes=sb["fc"] + sb["backbone"] + sb["lm_head"]),
        "drafted_tok_s": steps_per_s * drafted,
        "accepted_tok_s": steps_per_s * B * mean_acc_len,
        "mean_acceptance_length": mean_acc_len,
        "per_position_acceptance": per_pos,
        "roofline": {"bound": "hbm",
                     "kernel": ("quantize_rows + gemm_tcgen05<fp8> (LM head stage)" if pipe.fp8
                                else "gemm_tcgen05, two phases: fc then LM head (one launch)"
                                if pipe.fused else "gemm_tcgen05 (LM head)"),
                     "achieved": achieved,
                     "peak": peak_gbs, "unit": "GB/s", "frac": achieved / peak_gbs,
                     "traffic": traffic,
                     "traffic_source": ("profiled: dram__bytes_read.sum + dram__bytes_write.sum "
                                        "per launch from profiles/%s_%s.md (ncu capture of the same "
                                        "kernel source), not measured in this run"
                                        % (traffic_file, name)) if traffic is not None else None,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": lm_bytes, "ms_per_launch": lm_ms},
        "step_roofline": step_roof,
        "graph": loops is not None,
        "graph_error": graph_error,
        "timing": ("decode loop: K steps per CUDA-graph replay; verify of step i on a second "
                   "stream beside the fc and LM head of step i+1; the chain of step i+1 waits "
                   "for it" if loops is not None else "un-captured serial steps"),
        "timed_reps": {"reps": len(rep_ms), "steps_per_rep": K, "median_ms": max_ms,
                       "min_ms": min(rep_ms), "max_ms": max(rep_ms),
                       "seconds": sum(rep_ms) / 1000.0},
        "serial": {"value": whole_job_rate(K, world, serial_ms / 1000.0), "unit": "steps/s",
                   "ms_per_step": serial_ms / K,
                   "what": "one CUDA graph per step, draft and verify on one stream"},
        "uncaptured": {"value": whole_job_rate(K, world, plain_ms / 1000.0), "unit": "steps/s",
                       "ms_per_step": plain_ms / K},
        "stage_ms": stage_ms,
        "gpu_launches": launches,
        "e2e": e2e,
        "clocks": clk,
    }

    if cfg.get("backbone"):
        with_cpu_baseline = False   # the C oracle's step has no backbone layers
    if with_cpu_baseline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as ora
        hw = host_cache[(H, T, V, r)]
        st = sets[0]["host"]
        host = {"taps": st["taps"], "fc_w": hw["fc_w"], "lm_w": hw["lm_w"],
                "w1": hw["w1"], "w2": hw["w2"], "prev": st["prev"],
                "target": np.ascontiguousarray(sets[0]["target"].cpu().numpy())}
        add_host_fp8(ora, host, cfg)
        host["h"] = oracle_h(ora, host, cfg)
        sps, cores, desc, _ = cpu_oracle_baseline(host, cfg, mode, args.cpu_budget)
        line["cpu_baseline"] = {"value": sps, "unit": "steps/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    del graphs, loops, staged, sets, pipes, pipe
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def config_of(name, cfg, mode, args, world, nsets=None, set_bytes=None, l2=None, weights_bytes=None):
    """The workload description shared by both arms' JSON lines."""
    c = {"workload": name, "B": cfg["B"], "k": cfg["k"], "H": cfg["H"], "taps": cfg["T"],
         "V": cfg["V"], "r": cfg["r"], "verify": "probabilistic" if mode == 1 else "greedy",
         "confidence_head": bool(cfg["conf"]),
         "weights": "e4m3 codes + fp32 row scales (fc, LM head)" if cfg.get("fp8") else "bf16",
         "parallelism": "replicas%d" % world}
    if cfg.get("backbone"):
        g = syn.BACKBONE_GEOMETRY[cfg["H"]]
        c["backbone"] = {"layers": cfg["backbone"]["L"], "context": cfg["backbone"]["C"], "q_heads": g["nq"],
                         "kv_heads": g["nkv"], "head_dim": 128, "mlp": g["I"]}
    if nsets is not None:
        c["q_stats_in"] = args.q_stats
        c["l2"] = ("inputs larger than L2: %.2f GB of weights streamed per step; %d input sets of "
                   "%.1f MB rotated (%.0f MB > 2x the %.0f MB L2)"
                   % (weights_bytes / 1e9, nsets, set_bytes / 1e6, nsets * set_bytes / 1e6, l2 / 1e6))
    return c


def run_ours(args, rank, local_rank, world):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    host_cache = {}
    line = measure_workload(args, args.config, rank, local_rank, world, host_cache, True)
    if args.config == "27b_b1" and not args.no_b16:
        # the metric names batch 1 and batch 16: the 27B batch-16 workload (confidence
        # head on) with the same steps, warm-up and timing rules
        sub = measure_workload(args, "27b_b16", rank, local_rank, world, host_cache, False)
        line["batch16"] = {kk: sub[kk] for kk in (
            "value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "drafted_tok_s",
            "accepted_tok_s", "mean_acceptance_length", "per_position_acceptance", "roofline",
            "step_roofline", "graph", "timing", "timed_reps", "serial", "uncaptured", "stage_ms",
            "gpu_launches", "e2e", "clocks")}
    if args.config == "27b_b1" and not args.no_backbone:
        # the same batch-1 step with one drafter backbone layer (N1) over a 1024-token
        # context, same steps, warm-up and timing rules
        sub = measure_workload(args, "27b_b1_backbone", rank, local_rank, world, host_cache, False)
        line["backbone"] = {kk: sub[kk] for kk in (
            "value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "drafted_tok_s",
            "accepted_tok_s", "mean_acceptance_length", "step_roofline", "graph", "timing", "timed_reps",
            "serial", "stage_ms", "gpu_launches", "e2e", "clocks")}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------- sweep

SWEEP_B = (1, 2, 4, 8, 16, 32, 64)
SWEEP_K = (4, 6, 7)
SWEEP_R = (32, 128)
SWEEP_SIGMA = (0.5, 2.0)


def run_sweep(args):
    """27B shapes over B x k x r x sigma (84 cells), probabilistic verify, the same step
    pipeline as the headline (--verify, --q-stats).  Per cell: 3 input sets (taps, prev tokens, target = own draft logits + sigma * N(0, 1)), one
    CUDA graph per set, W = 3 warm-up and --sweep-steps timed replays rotating the sets
    (1.8-2.2 GB of weights stream from HBM every step).  Prints one JSON line per cell:
    steps/s, drafted tok/s, acceptance and the step's roofline fraction."""
    import torch

    import speculative_decoding_fc_gb300 as ds

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    H, T, V = 5120, 5, 151936
    peak_gbs, peak_tf, peak_src = measured_peaks()

    def d16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    base = syn.weights(H, T, V, 8, with_markov=False)
    fc_w, lm_w = d16(base["fc_w"]), d16(base["lm_w"])
    del base
    stream = torch.cuda.current_stream(device)
    nsets = 3
    for r in SWEEP_R:
        mk = syn.weights(8, 1, V, r, with_markov=True)
        w1, w2 = d16(mk["w1"]), d16(mk["w2"])
        del mk
        for B in SWEEP_B:
            for k in SWEEP_K:
                # unit-variance noise and taps per input set, shared by both sigmas
                raw = [syn.step_inputs(replica_step_seed(si, 0), B, k, H, T, V, ("const", 1.0))
                       for si in range(nsets)]
                cell = dict(B=B, k=k, H=H, T=T, V=V, r=r, conf=False)
                pipe = Pipeline(ds, torch, device, cell, 1,
                                {"fc_w": fc_w, "lm_w": lm_w, "w1": w1, "w2": w2, "conf_w": None}, args)
                hist = tuple(torch.zeros((B,), dtype=torch.int32, device=device) for _ in range(3))
                acc_o = hist[0]
                dev_sets = []
                for st in raw:
                    taps = [d16(t) for t in st["taps"]]
                    prev = torch.from_numpy(st["prev"]).to(device)
                    h = ds.fc_project(taps, fc_w)
                    lg = ds.lm_head(h, lm_w).view(B, k, V)
                    ds.greedy_sample(lg, w1, w2, prev, want_q_stats=False)
                    own = torch.cat([lg, lg[:, -1:]], dim=1)
                    dev_sets.append({"taps": taps, "prev": prev, "own": own,
                                     "noise": torch.from_numpy(st["noise"]).to(device)})
                del raw
                for sigma in SWEEP_SIGMA:
                    for st in dev_sets:
                        st["target"] = (st["own"] + st["noise"] * sigma).contiguous()

                    for st in dev_sets:        # eager warm-up (workspaces, first launches)
                        pipe.step(st, stream, hist, 0)
                    torch.cuda.synchronize()
                    cap = torch.cuda.Stream(device)
                    cap.wait_stream(stream)
                    graphs = []
                    for st in dev_sets:
                        g = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(g, stream=cap):
                            pipe.step(st, cap, hist, 0)
                        graphs.append(g)
                    stream.wait_stream(cap)
                    for i in range(3):
                        graphs[i % nsets].replay()
                    torch.cuda.synchronize()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    acc_sum = 0
                    e0.record(stream)
                    for i in range(args.sweep_steps):
                        graphs[i % nsets].replay()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    ms = e0.elapsed_time(e1) / args.sweep_steps
                    # acceptance of one step on each set (outside the timed loop)
                    for g in graphs:
                        g.replay()
                        torch.cuda.synchronize()
                        acc_sum += int(acc_o.sum().item())
                    cfg = dict(B=B, k=k, H=H, T=T, V=V, r=r)
                    sb = step_bytes(cfg, 1)
                    t_roof = max(sb["total"] / (peak_gbs * 1e9), step_flops(cfg) / (peak_tf * 1e12))
                    bound = "hbm" if sb["total"] / (peak_gbs * 1e9) >= step_flops(cfg) / (peak_tf * 1e12) \
                        else "tensor"
                    sps = 1000.0 / ms
                    print(json.dumps({
                        "sweep_cell": {"B": B, "k": k, "r": r, "sigma": sigma},
                        "steps_per_s": sps, "ms_per_step": ms, "drafted_tok_s": sps * B * k,
                        "mean_acceptance_length": acc_sum / (nsets * B) + 1.0,
                        "roofline": {"bound": bound, "t_roofline_ms": t_roof * 1000.0,
                                     "frac": t_roof * 1000.0 / ms, "peak_source": peak_src},
                        "steps": args.sweep_steps, "warmup": 3, "input_sets": nsets,
                        "dtype": "bf16", "data": "synthetic"}), flush=True)
                    del graphs
                del dev_sets, pipe
                torch.cuda.empty_cache()
        del w1, w2
    return 0


def main():
    args = parse_args()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.sweep:
        return run_sweep(args) if rank == 0 else 0
    return run_ours(args, rank, local_rank, world)


if __name__ == "__main__":
    sys.exit(main())
