"""Write tests/golden/tiny_oracle_trace.json from the CPU oracle alone.

The tiny workload (4 layers, d=256, batch 1, 32 prompt tokens, 16 greedy
decode steps, checkpoints at layers 1 and 2): gamma_l is the 40th percentile
of the oracle's no-exit confidences at layer l over decode steps 1..8; the
trace is the oracle's tokens, exit layers and confidences with those gammas.
Run from the repository root:  python tests/golden/make_tiny_trace.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    w = synth.WORKLOADS["tiny-b1"]
    lens, prompts = synth.workload_inputs(w)
    o = oracle.build_oracle(w)
    gam, samples = oracle.calibrate_gammas(o, prompts, w.calib_steps, w.gamma_percentiles)
    g = gam[w.gamma_percentiles[0]]
    o.set_thresholds(g)
    tok = o.prefill(prompts)
    trace = {"first_tokens": tok.tolist(), "tokens": [], "exit_layers": [], "conf": [],
             "margins": []}
    for _ in range(w.steps):
        r = o.decode_step(tok)
        trace["tokens"].append(r.next_tokens.tolist())
        trace["exit_layers"].append(r.exit_layers.tolist())
        trace["conf"].append([[None if np.isnan(c) else float(c) for c in row] for row in r.conf])
        trace["margins"].append(r.margins.tolist())
        tok = r.next_tokens
    out = {
        "workload": w.name, "seed": w.seed, "prompt_lens": lens.tolist(),
        "checkpoints": list(w.checkpoints), "gamma_percentile": w.gamma_percentiles[0],
        "gamma": [float(x) for x in g],
        "calibration_conf": samples.tolist(),
        "trace": trace,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_trace.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
