#!/usr/bin/env python
"""Early-exit greedy decode benchmark (one GB300 per rank).

A step is one ee_decode_step: one early-exit decode of every sequence of the
batch through the whole hot path (embedding, per layer RMSNorm -> QKV + RoPE
+ shared-KV write -> paged attention -> O + residual -> RMSNorm -> gate/up +
SwiGLU -> down + residual, the checkpoint exit heads with their decisions and
sub-batch compaction, the final head).

Default workload: Llama-3.1-8B shape, batch 1, 2048-token prompt, greedy
decode with thresholds at the 40th percentile of the no-exit confidences of
the first 8 decode steps.  The same kernels are also timed as the forced
no-exit baseline.  Weights and prompts are seeded synthetic data.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
        python bench.py --impl reference ...   (the CPU oracle, bounded sample)
For N > 1 run under torchrun: every rank decodes its own batch (replicas, no
collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_WORKLOAD = "llama3.1-8b-b1"
B32_WORKLOAD = "llama3.1-8b-b32"
SMALL_WORKLOAD = "llama3.2-1b-b1"
LARGE_WORKLOAD = "codellama-34b-b8"
METRIC = "decoded tokens/s"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers

# ncu summary with the DRAM bytes per GEMV launch of the default workload
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "k_linear_dram_llama3.2-1b_b1.md")
GEMV_SOURCES = ("k_linear.cu", "ee_gemv.cuh", "ee_epilogue.cuh", "ee_head.cuh", "ee_common.cuh", "ee_kernels.cuh")


def _code_only(text):
    """Source text without comments and with whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def gemv_source_digest():
    """sha256 (16 hex digits) of the GEMV kernel's sources in a fixed order,
    comments and whitespace removed: edits to comments keep the digest."""
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(ROOT, "early_exit_decoding_layer_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic_ratio(workload, path=TRAFFIC_SUMMARY):
    """DRAM bytes (read + write) over algorithmic bytes of the GEMV launches in
    the committed ncu summary: its `key: value` lines give the workload the
    capture ran on, the workloads the ratio is applied to (`applies_to`, a
    comma list; the GEMV streams each weight byte once per launch at any
    shape, so the ratio carries over from a small capture), the sources'
    digest and the two per-launch figures.  None unless `workload` is covered
    and the GEMV sources are unchanged since the capture."""
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith(("|", "#", " ", "-")):
                k, v = line.split(":", 1)
                kv[k.strip().strip("`")] = v.strip().strip("`")
    try:
        covered = {kv["workload"]} | {x.strip() for x in kv.get("applies_to", "").split(",") if x.strip()}
        if workload not in covered or kv.get("gemv_sources_sha256") != gemv_source_digest():
            return None
        return float(kv["dram_bytes_per_launch"]) / float(kv["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError, ZeroDivisionError, OSError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def mat_list(sh):
    d, dq, dk, F = sh.d_model, sh.n_heads * sh.head_dim, sh.n_kv_heads * sh.head_dim, sh.ffn_dim
    return {"qkv": (dq + 2 * dk, d), "o": (d, dq), "gateup": (2 * F, d), "down": (d, F)}


def w_bytes(N, K, int4):
    if int4:
        return N * K // 2 + N * ((K + 127) // 128) * 2
    return N * K * 2


def launch_bytes(sh, ckpts, kind, layer, exits, ctxs, lists="both"):
    """Algorithmic bytes one launch must read: the weights of the sub-batches
    it serves (bf16 rows of sequences still on the backbone, int4 rows of
    exited ones; a tensor-core launch serves one list, `lists` "full" or
    "exit", the GEMV both), the head tensors, or the K/V history."""
    mats = mat_list(sh)
    if kind in mats:
        N, K = mats[kind]
        full = lists in ("both", "full") and any(e >= layer for e in exits)
        ex = lists in ("both", "exit") and any(e < layer for e in exits)
        return full * w_bytes(N, K, False) + ex * w_bytes(N, K, True)
    d, V = sh.d_model, sh.vocab
    if kind in ("head_t", "head_e"):
        # a checkpoint's head reads T and E only for sequences still on the
        # backbone there (e >= layer); after every sequence exited its lists
        # are empty and it reads nothing
        if not any(e >= layer for e in exits):
            return 0
        return d * d * 2 if kind == "head_t" else V * d * 2
    if kind == "final_head":
        return V * d * 2
    if kind == "attn":
        return sum(int(c) * 2 * sh.n_kv_heads * sh.head_dim * 2 for c in ctxs)
    return 0


def step_bytes(sh, ckpts, exits, ctxs, heads, criterion="maxprob", token_source="final"):
    """Bytes a step must read (the workload's roofline rule): for each layer the
    bf16 weights if any sequence runs it in bf16 and the int4 weights plus
    scales if any runs it on the exit copy; T and E for every head evaluated
    (the similarity criterion reads two d-vectors per sequence instead, which
    is negligible and not counted); E for the final head; every sequence's
    K/V history of every layer."""
    # With exit-head tokens an exited sequence's last layer reads only its QKV
    # rows, and the final head serves the sequences that never exited.
    head_tok = heads and criterion == "maxprob" and token_source == "exit_head"
    heads = heads and criterion == "maxprob"
    L = sh.n_layers
    total = 0
    for j in range(L):
        for kind in ("qkv", "o", "gateup", "down"):
            if head_tok and j == L - 1 and kind != "qkv":
                stay = [e for e in exits if e == L - 1]
                total += launch_bytes(sh, ckpts, kind, j, stay, ctxs) if stay else 0
            else:
                total += launch_bytes(sh, ckpts, kind, j, exits, ctxs)
        if head_tok and j == L - 1:
            total += launch_bytes(sh, ckpts, "attn", j, exits, [c for c, e in zip(ctxs, exits) if e == L - 1])
        else:
            total += launch_bytes(sh, ckpts, "attn", j, exits, ctxs)
    if heads:
        for l in ckpts:
            if any(e >= l for e in exits):
                total += launch_bytes(sh, ckpts, "head_t", l, exits, ctxs)
                total += launch_bytes(sh, ckpts, "head_e", l, exits, ctxs)
    if not head_tok or any(e == L - 1 for e in exits):
        total += launch_bytes(sh, ckpts, "final_head", -1, exits, ctxs)
    return total


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "200"]
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        first = vis.split(",")[0].strip() if vis else ""
        if first:
            cmd += ["-i", first]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(use_cuda: bool):
    rank, world, local = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if use_cuda:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if use_cuda else "gloo")
    return rank, world, local


def barrier(world, use_cuda):
    if world > 1:
        import torch.distributed as dist
        if use_cuda:
            import torch
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def reduce_max(x: float, world: int, use_cuda: bool) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, use_cuda: bool) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- the oracle (CPU)

def oracle_step_sample(w, layers=2, ctx=None, seed=99, timings=None):
    """Times the CPU oracle's own functions on a bounded sample of one decode
    step of workload w: `layers` decoder layers at context `ctx` (synthetic K/V
    history standing in for the prompt), one checkpoint exit head and the final
    head.  Weight generation and conversion are outside the timing.  Returns
    (seconds per decode step of one sequence extrapolated to all layers with
    one head, dict of the parts)."""
    import oracle
    sh = w.shape
    cfg = oracle.ModelConfig.from_shape(sh, w.checkpoints)
    ctx = ctx or (w.max_prompt() + w.steps // 2)
    t_layer = []
    for j in range(layers):
        Wt = oracle.Weights(cfg, lambda jj: synth.layer_weights(sh, w.seed, jj),
                            np.zeros((2, sh.d_model), np.uint16), synth.final_gain(sh), [],
                            cache_bytes=0)
        lw = Wt.layer(j, False)
        kh = synth.normal_f32(seed, 7 * j + 1, (ctx + 1, sh.n_kv_heads, sh.head_dim), 1.0).astype(np.float64)
        vh = synth.normal_f32(seed, 7 * j + 2, (ctx + 1, sh.n_kv_heads, sh.head_dim), 1.0).astype(np.float64)
        h = synth.normal_f32(seed, 7 * j + 3, (sh.d_model,), 1.0).astype(np.float64)
        t0 = time.perf_counter()
        oracle.layer_decode(cfg, lw, h, ctx, kh, vh)
        t_layer.append(time.perf_counter() - t0)
        del lw, kh, vh
    E = oracle.bf16_to_f64(synth.embedding(sh, w.seed))
    g = oracle.bf16_to_f64(synth.final_gain(sh))
    T = oracle.bf16_to_f64(synth.exit_transform(sh, w.seed, 0)) if w.checkpoints else None
    h = synth.normal_f32(seed, 5, (sh.d_model,), 1.0).astype(np.float64)
    t0 = time.perf_counter()
    oracle.max_softmax(oracle.head_logits(h, g, E, sh.rms_eps, T))
    t_head = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.argmax_lowest(oracle.head_logits(h, g, E, sh.rms_eps))
    t_final = time.perf_counter() - t0
    parts = {"layer_s": float(np.mean(t_layer)), "exit_head_s": t_head, "final_head_s": t_final,
             "ctx": ctx}
    return sh.n_layers * parts["layer_s"] + t_head + t_final, parts


def cpu_threads():
    return os.cpu_count() or 1


def run_reference(args):
    """The oracle, as it stands, on this host's cores: every step is one bounded
    sample (one decoder layer at the workload's mid context plus the exit and
    final heads), extrapolated to a whole decode step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    secs = []
    parts = None
    t_all = time.perf_counter()
    for i in range(args.warmup + args.steps):
        s, parts = oracle_step_sample(w, layers=1, seed=100 + i)
        if i >= args.warmup:
            secs.append(s)
    per_step = statistics.median(secs)
    value = w.batch / (w.batch * per_step)  # sequences are decoded one after another
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3 * w.batch, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": w.batch, "seq_len": w.max_prompt(),
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": "per step: 1 decoder layer at context %d + exit head + final head "
                                   "(numpy float64), extrapolated to %d layers; %s"
                                   % (parts["ctx"], w.shape.n_layers, json.dumps(parts))},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ours

def load_engine(ee, w, max_batch, max_seq_len, stream):
    sh = w.shape
    eng = ee.DecodeEngine(sh, w.checkpoints, max_batch, max_seq_len, stream=stream)
    for j in range(sh.n_layers):
        eng.load_layer(j, synth.layer_weights(sh, w.seed, j))
    eng.load_shared(synth.embedding(sh, w.seed), synth.final_gain(sh),
                    [synth.exit_transform(sh, w.seed, c) for c in range(len(w.checkpoints))])
    return eng


def oracle_gammas(name):
    """The workload's thresholds calibrated on the CPU oracle (a stored file,
    see tests/golden/make_oracle_gammas.py), or None."""
    path = os.path.join(ROOT, "tests", "golden", "oracle_gammas.json")
    if not os.path.exists(path):
        return None
    return json.load(open(path)).get(name)


def calibration_hist(conf, gamma, ckpts, n_layers):
    """Exit layers that thresholds gamma give on no-exit confidence samples
    [samples, checkpoints] (first checkpoint whose confidence is above gamma)."""
    hist = {}
    for row in np.asarray(conf):
        e = n_layers - 1
        for c, l in enumerate(ckpts):
            if row[c] > gamma[c]:
                e = l
                break
        hist[int(e)] = hist.get(int(e), 0) + 1
    return dict(sorted(hist.items()))


def calibrate(eng, w, prompts, steps, percentiles):
    """gamma_l = p-th percentile of the no-exit confidences at checkpoint l over
    the first `steps` decode steps (one sample per sequence and step)."""
    eng.set_exit_enabled(True)
    eng.set_thresholds([np.inf] * len(w.checkpoints))
    tok = eng.prefill(prompts)
    confs = []
    for _ in range(steps):
        tok, _ = eng.decode_step(tok)
        confs.append(eng.debug_conf())
    c = np.concatenate(confs, axis=0)
    return {p: np.percentile(c, p, axis=0) for p in percentiles}, c


def timed_run(eng, w, prompts, steps, warmup, heads, world, profile_steps=0, ncu_region=False):
    import torch
    eng.set_exit_enabled(heads)
    tok = eng.prefill(prompts)
    for _ in range(warmup):
        tok, _ = eng.decode_step(tok)
    ctx0 = np.array([eng.seq_pos(s) for s in range(len(prompts))])
    barrier(world, True)
    torch.cuda.synchronize()
    clocks = ClockSampler()
    dev_ms = []
    exits = []
    if ncu_region:  # a profiler started with --profile-from-start off captures only these steps
        torch.cuda.profiler.start()
    t0 = time.perf_counter()
    for _ in range(steps):
        tok, ex = eng.decode_step(tok)
        dev_ms.append(eng.last_step_ms())
        exits.append(ex.copy())
    wall = time.perf_counter() - t0
    torch.cuda.synchronize()
    if ncu_region:
        torch.cuda.profiler.stop()
    barrier(world, True)
    clk = clocks.stop()
    prof = []
    if profile_steps:
        eng.set_profile(True)
        for _ in range(profile_steps):
            ctx = np.array([eng.seq_pos(s) + 1 for s in range(len(prompts))])
            tok, ex = eng.decode_step(tok)
            prof.append((eng.profile_read(), ex.copy(), ctx))
        eng.set_profile(False)
    return {"dev_ms": dev_ms, "wall_s": wall, "exits": exits, "ctx0": ctx0, "clocks": clk,
            "profile": prof}


def kernel_roofline(sh, ckpts, prof, peak):
    """Achieved HBM bandwidth of the GEMV kernel (every projection, exit-head and
    LM-head launch) and of the attention kernel from the profiled launches.
    A launch's duration is its own (first CTA start to last CTA end) where the
    kernel records it (the GEMV and the tensor-core GEMM), else the event
    pair around it (which adds the launch gap); the shares use the event
    times throughout."""
    lin = ("qkv", "o", "gateup", "down", "head_t", "head_e", "final_head")
    acc = {"linear": [0, 0.0, 0], "attn": [0, 0.0, 0]}
    per_kind = {}
    own = [0, 0]  # projection and head launches timed by the kernel itself, all of them
    for recs, exits, ctx in prof:
        for kind, layer, ms, kms, lists in recs:
            b = launch_bytes(sh, ckpts, kind, layer, exits, ctx, lists)
            key = "linear" if kind in lin else ("attn" if kind == "attn" else None)
            pk = per_kind.setdefault(kind, [0, 0.0, 0])
            pk[0] += b
            pk[1] += ms
            pk[2] += 1
            if key:
                acc[key][0] += b
                acc[key][1] += kms if kms > 0 else ms
                acc[key][2] += 1
                if key == "linear":
                    own[0] += kms > 0
                    own[1] += 1
    out = {}
    for k, (b, ms, n) in acc.items():
        gbs = b / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
        out[k] = {"bytes_per_launch": b / max(n, 1), "ms_per_launch": ms / max(n, 1),
                  "achieved_gbs": gbs, "frac": gbs / peak}
    tot = sum(v[1] for v in per_kind.values())
    out["share"] = {k: round(v[1] / tot, 4) for k, v in sorted(per_kind.items(), key=lambda x: -x[1][1])}
    out["ms_per_step_profiled"] = tot / max(len(prof), 1)
    out["launches_with_own_time"] = "%d of %d" % tuple(own)
    return out


def run_workload(ee, w, args, st, rank, world, peak, steps, profile_steps):
    """Loads the workload's model, calibrates the thresholds, and times the exit
    runs (one per threshold percentile) and the forced no-exit run."""
    sh = w.shape
    B = w.batch
    max_seq = w.max_prompt() + args.warmup + steps + w.calib_steps + 16
    lens, prompts = synth.workload_inputs(w)
    if rank:  # replicas decode different sequences
        prompts = synth.prompts(sh, w.seed + 1000 * rank, lens)
    t_load = time.perf_counter()
    eng = load_engine(ee, w, B, max_seq, st)
    t_load = time.perf_counter() - t_load
    lib_gammas, calib = calibrate(eng, w, prompts, w.calib_steps, w.gamma_percentiles)
    # the thresholds: the oracle's percentiles where they were computed
    # (tests/golden/oracle_gammas.json, written from the CPU oracle alone),
    # else the library's own calibration on this run's prompts
    og = oracle_gammas(w.name)
    gammas = {p: np.asarray(og["gamma"]["p%g" % p]) for p in w.gamma_percentiles} if og else lib_gammas
    gamma_source = "oracle" if og else "library"

    runs = {}
    for pct in w.gamma_percentiles:
        eng.set_thresholds(gammas[pct])
        runs[pct] = timed_run(eng, w, prompts, steps, args.warmup, True, world,
                              profile_steps=profile_steps, ncu_region=args.ncu_region)
    base = timed_run(eng, w, prompts, steps, args.warmup, False, world,
                     profile_steps=profile_steps, ncu_region=args.ncu_region)
    # exit-head tokens (the exit head's argmax is emitted; the same thresholds)
    head_tok_run = None
    if args.exit_head_token:
        eng.set_token_source("exit_head")
        eng.set_thresholds(gammas[w.gamma_percentiles[0]])
        head_tok_run = timed_run(eng, w, prompts, steps, args.warmup, True, world,
                                 ncu_region=args.ncu_region)
        eng.set_token_source("final")
    # the state-transition-similarity criterion, thresholds at the library's
    # percentiles of the no-exit similarity scores
    # (per sequence; at batch > 1 also the batch-minimum rule, whose
    # thresholds are percentiles of the per-step batch minimum)
    sts_runs, taus = {}, {}
    if args.sts:
        modes = ("sts",) if B == 1 else ("sts", "sts_batch")
        for mode in modes:
            eng.set_exit_criterion(mode)
            tm, _ = calibrate(eng, w, prompts, w.calib_steps, w.gamma_percentiles)
            for pct in w.gamma_percentiles:
                key = "%s_p%g" % (mode, pct)
                taus[key] = tm[pct]
                eng.set_thresholds(tm[pct])
                sts_runs[key] = timed_run(eng, w, prompts, steps, args.warmup, True, world,
                                          ncu_region=args.ncu_region)
        eng.set_exit_criterion("maxprob")

    def summarize(r, heads, criterion="maxprob", token_source="final"):
        dev_s = sum(r["dev_ms"]) / 1e3
        max_dev = reduce_max(dev_s, world, True)
        max_wall = reduce_max(r["wall_s"], world, True)
        tokens = B * steps * world
        bytes_total = 0
        for k, ex in enumerate(r["exits"]):
            ctx = r["ctx0"] + k + 1
            bytes_total += step_bytes(sh, w.checkpoints, ex, ctx, heads, criterion, token_source)
        hist = {}
        for ex in r["exits"]:
            for e in ex:
                hist[int(e)] = hist.get(int(e), 0) + 1
        return {"value": tokens / max_dev, "e2e": tokens / max_wall, "ms_per_step": 1e3 * max_dev / steps,
                "bytes_per_step": bytes_total / steps,
                "step_roofline_frac_8tbs": bytes_total / dev_s / 8e12,
                "step_roofline_frac_measured": bytes_total / dev_s / (peak * 1e9),
                "exit_hist": dict(sorted(hist.items())), "clocks": r["clocks"]}

    main = summarize(runs[w.gamma_percentiles[0]], True)
    nox = summarize(base, False)
    prof_main = runs[w.gamma_percentiles[0]]["profile"]
    kr = kernel_roofline(sh, w.checkpoints, prof_main, peak) if prof_main else None
    kr_base = kernel_roofline(sh, w.checkpoints, base["profile"], peak) if base["profile"] else None
    others = {str(pct): dict(summarize(runs[pct], True), gamma=[float(x) for x in gammas[pct]])
              for pct in w.gamma_percentiles[1:]}
    sts = {key: dict(summarize(sts_runs[key], True, "sts"), tau=[float(x) for x in taus[key]])
           for key in sts_runs}
    head_tok = dict(summarize(head_tok_run, True, "maxprob", "exit_head")) if head_tok_run else None
    # exit depths the library's own thresholds give on its calibration samples
    lib_hist = calibration_hist(calib, lib_gammas[w.gamma_percentiles[0]], w.checkpoints, sh.n_layers)
    return {"eng": eng, "gammas": gammas, "main": main, "nox": nox, "runs": runs, "kr": kr, "kr_base": kr_base,
            "t_load": t_load, "others": others, "sts": sts, "head_tok": head_tok, "gamma_source": gamma_source,
            "lib_gammas": lib_gammas, "lib_hist": lib_hist}


def run_ours(args):
    import torch

    rank, world, local = dist_init(True)
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_layer_gb300 as ee

    w = synth.WORKLOADS[args.workload]
    sh = w.shape
    peak, peak_kind = peaks()
    B = w.batch
    st = torch.cuda.Stream()
    res = run_workload(ee, w, args, st, rank, world, peak, args.steps, args.profile_steps)
    eng, gammas, main, nox, runs, kr, kr_base, t_load = (res[k] for k in (
        "eng", "gammas", "main", "nox", "runs", "kr", "kr_base", "t_load"))
    h2d, d2h, launches = eng.step_io(B, True)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s_step, parts = oracle_step_sample(w, layers=args.cpu_layers)
        cpu = {"value": 1.0 / s_step, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": "%d decoder layers at context %d + exit head + final head of one sequence "
                         "(numpy float64, weights prepared outside the timing), extrapolated to %d "
                         "layers; parts %s" % (args.cpu_layers, parts["ctx"], sh.n_layers, json.dumps(parts))}

    if rank == 0:
        clk = main["clocks"]
        line = {
            "metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init weights N(0,0.02), uniform random prompts)",
            "config": {"workload": w.name, "model": sh.name, "global_batch": B * world,
                       "seq_len": w.max_prompt(), "parallelism": "replicas" if world > 1 else "single",
                       "gamma_percentile": w.gamma_percentiles[0],
                       "gamma": [float(x) for x in gammas[w.gamma_percentiles[0]]],
                       "l2": "inputs larger than L2 (weights %.1f GB/step streamed)" % (main["bytes_per_step"] / 1e9)},
            "e2e": {"value": main["e2e"], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps,
            "roofline": None,
            "cpu_baseline": cpu,
            "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"),
                       "reasons": clk.get("reasons")},
            "no_exit": {"value": nox["value"], "ms_per_step": nox["ms_per_step"], "e2e": nox["e2e"],
                        "bytes_per_step": nox["bytes_per_step"],
                        "step_roofline_frac_8tbs": nox["step_roofline_frac_8tbs"],
                        "step_roofline_frac_measured": nox["step_roofline_frac_measured"],
                        "clocks": nox["clocks"], "kernel": kr_base},
            "speedup_vs_no_exit": main["value"] / nox["value"],
            "step_roofline": {"bytes_per_step": main["bytes_per_step"],
                              "frac_8tbs": main["step_roofline_frac_8tbs"],
                              "frac_measured": main["step_roofline_frac_measured"]},
            "exit_hist": main["exit_hist"],
            "load_s": t_load,
        }
        line["config"]["gamma_source"] = res["gamma_source"]
        line["gamma_library"] = {"gamma": [float(x) for x in res["lib_gammas"][w.gamma_percentiles[0]]],
                                 "exit_hist_on_calibration_samples": res["lib_hist"]}
        if res["head_tok"]:
            v = res["head_tok"]
            line["exit_head_token"] = {"value": v["value"], "ms_per_step": v["ms_per_step"], "e2e": v["e2e"],
                                       "speedup_vs_no_exit": v["value"] / nox["value"],
                                       "step_roofline_frac_measured": v["step_roofline_frac_measured"],
                                       "bytes_per_step": v["bytes_per_step"], "exit_hist": v["exit_hist"]}
        if res["sts"]:
            line["sts"] = {k: {"value": v["value"], "ms_per_step": v["ms_per_step"], "e2e": v["e2e"],
                               "speedup_vs_no_exit": v["value"] / nox["value"],
                               "step_roofline_frac_measured": v["step_roofline_frac_measured"],
                               "bytes_per_step": v["bytes_per_step"], "exit_hist": v["exit_hist"],
                               "tau": v["tau"]} for k, v in res["sts"].items()}
        if kr:
            k = kr["linear"]
            line["roofline"] = {"bound": "hbm", "kernel": "k_linear (GEMV, all launches of a step)",
                                "timing": "kernel's own time per launch: globaltimer at its first CTA's start "
                                          "and last CTA's end, profiled steps",
                                "achieved": k["achieved_gbs"], "peak": peak,
                                "peak_kind": peak_kind, "unit": "GB/s", "frac": k["frac"],
                                "traffic": None, "bytes_per_launch": k["bytes_per_launch"],
                                "ms_per_launch": k["ms_per_launch"]}
            ratio = measured_traffic_ratio(w.name)
            if ratio is not None:
                line["roofline"]["traffic"] = ratio * k["bytes_per_launch"]
                line["roofline"]["traffic_note"] = (
                    "ncu dram__bytes_read.sum + dram__bytes_write.sum over the GEMV launches of one exit-run "
                    "and one no-exit step of the Llama-3.2-1B batch-1 workload (profiles/%s) = %.4f x their "
                    "algorithmic bytes; scaled to this run's algorithmic bytes per launch"
                    % (os.path.basename(TRAFFIC_SUMMARY), ratio))
            line["kernels"] = kr
        for pct, extra in res["others"].items():
            line.setdefault("other_gammas", {})[pct] = {
                "value": extra["value"], "ms_per_step": extra["ms_per_step"],
                "exit_hist": extra["exit_hist"], "gamma": extra["gamma"]}
    eng.close()
    if rank == 0 and world == 1 and args.b32_steps > 0 and w.name == DEFAULT_WORKLOAD:
        # the metric's second configuration: the same shape at batch 32
        # (ragged prompts, thresholds at the 40th and 70th percentiles)
        import gc
        del eng, res
        gc.collect()
        torch.cuda.empty_cache()
        w32 = synth.WORKLOADS[B32_WORKLOAD]
        r32 = run_workload(ee, w32, args, st, rank, world, peak, args.b32_steps, 1)
        m32, n32 = r32["main"], r32["nox"]
        line["b32"] = {
            "workload": w32.name, "steps": args.b32_steps, "warmup": args.warmup,
            "value": m32["value"], "unit": "tokens/s", "ms_per_step": m32["ms_per_step"],
            "e2e": m32["e2e"], "step_roofline_frac_measured": m32["step_roofline_frac_measured"],
            "bytes_per_step": m32["bytes_per_step"], "exit_hist": m32["exit_hist"],
            "gamma_percentile": w32.gamma_percentiles[0], "clocks": m32["clocks"],
            "other_gammas": {k: {"value": v["value"], "ms_per_step": v["ms_per_step"],
                                 "step_roofline_frac_measured": v["step_roofline_frac_measured"]}
                             for k, v in r32["others"].items()},
            "no_exit": {"value": n32["value"], "ms_per_step": n32["ms_per_step"],
                        "step_roofline_frac_measured": n32["step_roofline_frac_measured"],
                        "bytes_per_step": n32["bytes_per_step"]},
            "kernels": r32["kr"], "kernels_no_exit": r32["kr_base"],
            "gamma_source": r32["gamma_source"],
            "sts": {k: {"value": v["value"], "ms_per_step": v["ms_per_step"],
                        "speedup_vs_no_exit": v["value"] / n32["value"],
                        "step_roofline_frac_measured": v["step_roofline_frac_measured"],
                        "exit_hist": v["exit_hist"], "tau": v["tau"]} for k, v in r32["sts"].items()},
        }
        r32["eng"].close()
    if rank == 0 and world == 1 and args.also_1b and w.name == DEFAULT_WORKLOAD:
        # the Llama-3.2-1B shape at batch 1 (512-token prompt), same runs
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        w1 = synth.WORKLOADS[SMALL_WORKLOAD]
        r1 = run_workload(ee, w1, args, st, rank, world, peak, args.steps, 1)
        m1, n1 = r1["main"], r1["nox"]
        line["b1_" + w1.shape.name] = {
            "workload": w1.name, "steps": args.steps, "value": m1["value"], "unit": "tokens/s",
            "ms_per_step": m1["ms_per_step"], "e2e": m1["e2e"],
            "step_roofline_frac_measured": m1["step_roofline_frac_measured"],
            "bytes_per_step": m1["bytes_per_step"], "exit_hist": m1["exit_hist"],
            "gamma_source": r1["gamma_source"], "clocks": m1["clocks"],
            "no_exit": {"value": n1["value"], "ms_per_step": n1["ms_per_step"],
                        "step_roofline_frac_measured": n1["step_roofline_frac_measured"]},
            "speedup_vs_no_exit": m1["value"] / n1["value"],
            "exit_head_token": ({"value": r1["head_tok"]["value"],
                                 "speedup_vs_no_exit": r1["head_tok"]["value"] / n1["value"]}
                                if r1["head_tok"] else None),
            "sts": {k: {"value": v["value"], "speedup_vs_no_exit": v["value"] / n1["value"],
                        "exit_hist": v["exit_hist"]} for k, v in r1["sts"].items()},
            "kernels": r1["kr"],
        }
        r1["eng"].close()
    if rank == 0 and world == 1 and args.with_34b and w.name == DEFAULT_WORKLOAD:
        # the CodeLlama-34B shape at batch 8 (4096-token prompts): the exit run
        # and the forced no-exit run only (each run re-prefills 8 x 4096 tokens)
        import copy
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        w34 = synth.WORKLOADS[LARGE_WORKLOAD]
        a34 = copy.copy(args)
        a34.exit_head_token = False
        a34.sts = False
        r34 = run_workload(ee, w34, a34, st, rank, world, peak, args.steps_34b, 1)
        m34, n34 = r34["main"], r34["nox"]
        line["b8_" + w34.shape.name] = {
            "workload": w34.name, "steps": args.steps_34b, "value": m34["value"], "unit": "tokens/s",
            "ms_per_step": m34["ms_per_step"], "e2e": m34["e2e"],
            "step_roofline_frac_measured": m34["step_roofline_frac_measured"],
            "bytes_per_step": m34["bytes_per_step"], "exit_hist": m34["exit_hist"],
            "gamma_source": r34["gamma_source"], "clocks": m34["clocks"],
            "no_exit": {"value": n34["value"], "ms_per_step": n34["ms_per_step"],
                        "step_roofline_frac_measured": n34["step_roofline_frac_measured"],
                        "bytes_per_step": n34["bytes_per_step"]},
            "speedup_vs_no_exit": m34["value"] / n34["value"],
            "kernels": r34["kr"],
        }
        r34["eng"].close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ops(args):
    """Single-kernel timings at a workload's shapes (batch 1): each op entry
    point replayed from a CUDA graph of back-to-back launches that cycle over
    enough weight copies that every launch reads HBM (inputs > L2); prints one
    JSON line with the device time per launch, GB/s and the fraction of the
    measured copy bandwidth."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_layer_gb300 as ee

    w = synth.WORKLOADS[args.workload]
    sh = w.shape
    peak, peak_kind = peaks()
    d, F, dq, dk, V = sh.d_model, sh.ffn_dim, sh.n_heads * sh.head_dim, sh.n_kv_heads * sh.head_dim, sh.vocab
    dev = torch.device("cuda")
    st = torch.cuda.Stream()
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    iters = args.ops_iters

    def bf16_bits(n, k):
        return (torch.randn((n, k), device=dev, generator=gen) * 0.02).to(torch.bfloat16).view(torch.int16)

    def x16(m, k):
        return torch.randn((m, k), device=dev, generator=gen).to(torch.float16).view(torch.int16)

    def timed(make_call, nbytes):
        ncopy = max(2, int(math.ceil(3 * L2_BYTES / max(nbytes, 1))))
        calls = [make_call(i) for i in range(min(ncopy, iters))]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            for c in calls:  # warm-up (first launches, kernel attributes) outside the capture
                c()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st):
            for i in range(iters):
                calls[i % len(calls)]()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record()
            g.replay()
            e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / iters
        return {"us": us, "bytes": nbytes, "gbs": nbytes / us * 1e-3, "frac": nbytes / us * 1e-3 / peak,
                "copies": len(calls)}

    out = {}
    mats = [("qkv", dq + 2 * dk, d), ("o", d, dq), ("gateup", 2 * F, d), ("down", d, F)]
    for name, N, K in mats:
        ws = []
        x = x16(1, K)

        def mk_bf16(i, N=N, K=K, x=x, ws=ws):
            if i >= len(ws):
                ws.append(bf16_bits(N, K))
            wi = ws[i]
            return lambda: ee.linear_bf16(x, wi, stream=st)
        out["bf16_" + name] = timed(mk_bf16, N * K * 2)
        del ws[:]
        t4 = []

        def mk_int4(i, N=N, K=K, x=x, t4=t4):
            if i >= len(t4):
                t4.append(ee.quantize_int4(bf16_bits(N, K)))
            qi, si = t4[i]
            return lambda: ee.linear_int4(x, qi, si, stream=st)
        ng = (K + 127) // 128
        out["int4_" + name] = timed(mk_int4, N * K // 2 + N * ng * 2)
        del t4[:]
        torch.cuda.empty_cache()
    # paged attention at the workload's context, one sequence
    ctx = w.max_prompt() + 64
    hq, hkv, hd = sh.n_heads, sh.n_kv_heads, sh.head_dim
    nb = (ctx + 15) // 16
    kvs = []

    def mk_attn(i):
        if i >= len(kvs):
            kc = torch.randn((nb, hkv, 16, hd), device=dev, generator=gen).to(torch.float16).view(torch.int16)
            vc = torch.randn((nb, hkv, 16, hd), device=dev, generator=gen).to(torch.float16).view(torch.int16)
            kvs.append((kc, vc))
        kc, vc = kvs[i]
        q = torch.randn((1, hq * hd), device=dev, generator=gen)
        bt = torch.arange(nb, dtype=torch.int32, device=dev).view(1, nb)
        pos = torch.tensor([ctx - 1], dtype=torch.int32, device=dev)
        scratch = torch.zeros(ee.attention_scratch_bytes(1, hq, hkv, hd, ctx), dtype=torch.uint8, device=dev)
        return lambda: ee.attention(q, kc, vc, bt, pos, hq, hkv, hd, ctx, scratch=scratch, stream=st)
    out["attention_ctx%d" % ctx] = timed(mk_attn, 2 * ctx * hkv * hd * 2)
    del kvs[:]
    Es = []

    def mk_head(i):
        if i >= len(Es):
            Es.append(bf16_bits(V, d))
        Ei = Es[i]
        u = x16(1, d)
        scratch = torch.zeros(ee.head_scratch_bytes(1), dtype=torch.uint8, device=dev)
        return lambda: ee.vocab_head(u, Ei, scratch=scratch, stream=st)
    out["vocab_head"] = timed(mk_head, V * d * 2)
    print(json.dumps({"ops": out, "workload": w.name, "iters": iters, "peak": peak, "peak_kind": peak_kind,
                      "timing": "CUDA graph of back-to-back launches, events around one replay, device time "
                                "per launch (includes the gap between launches)"}), flush=True)


def run_dry_dist(args):
    """Multi-rank plumbing without a GPU (gloo): each rank reports made-up
    per-rank times; rank 0 prints the aggregate line."""
    rank, world, _ = dist_init(False)
    B, K = 4, args.steps
    my_time = 1.0 + 0.5 * rank
    barrier(world, False)
    t = reduce_max(my_time, world, False)
    tok = reduce_sum(B * K, world, False)
    if rank == 0:
        print(json.dumps({"metric": METRIC, "value": tok / t, "n_gpus": world, "max_time_s": t,
                          "tokens": tok, "scaling": "weak"}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--profile-steps", type=int, default=3)
    ap.add_argument("--cpu-layers", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--b32-steps", type=int, default=32,
                    help="timed steps of the batch-32 run added to the default workload's line (0: skip)")
    ap.add_argument("--ncu-region", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    ap.add_argument("--with-34b", action="store_true",
                    help="also time the CodeLlama-34B shape at batch 8 (4096-token prompts; several minutes)")
    ap.add_argument("--34b-steps", dest="steps_34b", type=int, default=32)
    ap.add_argument("--no-1b", dest="also_1b", action="store_false",
                    help="skip the Llama-3.2-1B batch-1 runs added to the default workload's line")
    ap.add_argument("--no-exit-head-token", dest="exit_head_token", action="store_false",
                    help="skip the run that emits the exit head's token")
    ap.add_argument("--no-sts", dest="sts", action="store_false",
                    help="skip the runs with the state-transition-similarity exit criterion")
    ap.add_argument("--ops", action="store_true",
                    help="time each kernel's op entry point at the workload's shapes (batch 1) and exit")
    ap.add_argument("--ops-iters", type=int, default=200)
    ap.add_argument("--dry-dist", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.dry_dist:
        return run_dry_dist(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.ops:
        return run_ops(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
