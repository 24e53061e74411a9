"""Write tests/golden/oracle_gammas.json: exit thresholds of the benchmark
workloads calibrated on the CPU oracle alone.

Rule (the workloads' way of fixing a per-layer threshold without trained
heads; one fixed threshold per exit layer, CALM article §2.2, used in the test
p > gamma of "大语言模型解码加速：自适应层并行机制解析" §2.2): run the oracle with
no exit (gamma = +inf) over the workload's seeded weights and prompts, collect
the confidence at each checkpoint for every sequence over decode steps
1..calib_steps, and take the p-th percentile per checkpoint
(oracle.calibrate_gammas).

Prompt shortening: the float64 oracle's prefill costs 2 * tokens * params
flops, so a workload may be calibrated on a prefix of each prompt
(``PREFIX`` below: prompt length // divisor, at least ``min_len`` tokens).
The record states the lengths used.

Run from the repository root (CPU only; tens of GB of host memory for the
8B shape):  python tests/golden/make_oracle_gammas.py llama3.1-8b-b1 ...
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_gammas.json")

# workload -> (divisor, min_len): calibrate on prompt[: max(min_len, len // divisor)]
PREFIX = {
    "tiny-b1": (1, 1),
    "llama3.2-1b-b1": (1, 1),
    "llama3.1-8b-b1": (1, 1),
    "llama3.1-8b-b32": (8, 32),
}


def calibrate(name: str, cache_gb: float) -> dict:
    w = synth.WORKLOADS[name]
    div, min_len = PREFIX[name]
    lens, prompts = synth.workload_inputs(w)
    used = [int(min(len(p), max(min_len, len(p) // div))) for p in prompts]
    prompts = [list(map(int, p[:n])) for p, n in zip(prompts, used)]
    # the KV history is sized for the calibration prompts, not the workload's
    o = oracle.build_oracle(w, cache_bytes=int(cache_gb * (1 << 30)),
                            max_seq_len=max(used) + w.calib_steps + 1)
    t0 = time.time()
    gam, S = oracle.calibrate_gammas(o, prompts, w.calib_steps, w.gamma_percentiles)
    secs = time.time() - t0
    rec = {
        "workload": w.name, "seed": w.seed, "checkpoints": list(w.checkpoints),
        "workload_prompt_lens": [int(x) for x in lens],
        "calibration_prompt_lens": used,
        "prompt_rule": ("full prompts" if div == 1 else
                        "prefix of each prompt: max(%d, len // %d) tokens" % (min_len, div)),
        "calib_steps": w.calib_steps,
        "gamma": {("p%g" % p): [float(x) for x in gam[p]] for p in w.gamma_percentiles},
        "conf_samples": S.tolist(),   # [steps, batch, checkpoints]
        "oracle_seconds": round(secs, 1),
    }
    return rec


def main(argv):
    cache_gb = float(os.environ.get("ORACLE_CACHE_GB", "36"))
    names = argv or list(PREFIX)
    db = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for n in names:
        print("calibrating", n, flush=True)
        db[n] = calibrate(n, cache_gb)
        print(n, db[n]["gamma"], "%.0f s" % db[n]["oracle_seconds"], flush=True)
        with open(OUT, "w") as f:
            json.dump(db, f, indent=1)
    print("wrote", OUT)


if __name__ == "__main__":
    main(sys.argv[1:])
