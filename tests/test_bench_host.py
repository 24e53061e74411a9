"""Host logic of bench.py: the roofline byte model against the workload's
stated per-step figures, and the multi-rank replica path over gloo (CPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench
import synth
from tests.conftest import ROOT


def test_step_bytes_8b_b1_no_exit():
    w = synth.WORKLOADS["llama3.1-8b-b1"]
    sh = w.shape
    L = sh.n_layers
    # bf16 layer: QKV 6144x4096 + O 4096x4096 + gate/up 28672x4096 + down 4096x14336, 2 B each
    assert sum(bench.w_bytes(N, K, False) for N, K in bench.mat_list(sh).values()) == 436207616
    ctx = 2048 + 128
    b = bench.step_bytes(sh, w.checkpoints, [L - 1], [ctx], heads=False)
    expect = 32 * 436207616 + 128256 * 4096 * 2 + 32 * ctx * 2 * 8 * 128 * 2
    assert b == expect
    assert 15.2e9 < b < 15.4e9       # the workload's 15.3 GB no-exit figure


def test_step_bytes_exit_at_first_checkpoint():
    w = synth.WORKLOADS["llama3.1-8b-b1"]
    sh = w.shape
    ctx = 2176
    b = bench.step_bytes(sh, w.checkpoints, [4], [ctx], heads=True)
    bf16 = 436207616
    int4 = sum(bench.w_bytes(N, K, True) for N, K in bench.mat_list(sh).values())
    assert int4 == 112459776
    E, T = 128256 * 4096 * 2, 4096 * 4096 * 2
    assert b == 5 * bf16 + 27 * int4 + (T + E) + E + 32 * ctx * 4096
    assert 7.5e9 < b < 7.8e9         # the workload's 7.64 GB bound


def test_launch_bytes_heads_after_every_exit_read_nothing():
    """A checkpoint head after all sequences exited runs on empty lists: no
    algorithmic bytes; before (or at) the exit layer it reads T and E."""
    w = synth.WORKLOADS["llama3.1-8b-b1"]
    sh = w.shape
    E, T = 128256 * 4096 * 2, 4096 * 4096 * 2
    assert bench.launch_bytes(sh, w.checkpoints, "head_t", 4, [4], [100]) == T
    assert bench.launch_bytes(sh, w.checkpoints, "head_e", 4, [4], [100]) == E
    assert bench.launch_bytes(sh, w.checkpoints, "head_t", 8, [4], [100]) == 0
    assert bench.launch_bytes(sh, w.checkpoints, "head_e", 8, [4], [100]) == 0
    assert bench.launch_bytes(sh, w.checkpoints, "head_e", 8, [4, 31], [100, 100]) == E
    assert bench.launch_bytes(sh, w.checkpoints, "final_head", -1, [4], [100]) == E
    # a layer with sequences on both paths: the GEMV reads both copies, each
    # tensor-core launch only its own list's
    bf16 = bench.w_bytes(*bench.mat_list(sh)["gateup"], False)
    q4 = bench.w_bytes(*bench.mat_list(sh)["gateup"], True)
    assert bench.launch_bytes(sh, w.checkpoints, "gateup", 10, [4, 31], [100, 100]) == bf16 + q4
    assert bench.launch_bytes(sh, w.checkpoints, "gateup", 10, [4, 31], [100, 100], "full") == bf16
    assert bench.launch_bytes(sh, w.checkpoints, "gateup", 10, [4, 31], [100, 100], "exit") == q4


def test_step_bytes_mixed_batch_reads_each_matrix_once():
    w = synth.WORKLOADS["llama3.1-8b-b32"]
    sh = w.shape
    # one sequence never exits, one exits at 4: every layer reads bf16, layers 5.. also int4
    b = bench.step_bytes(sh, w.checkpoints, [31, 4], [100, 100], heads=True)
    bf16 = 436207616
    int4 = 112459776
    E, T = 128256 * 4096 * 2, 4096 * 4096 * 2
    heads = 7 * (T + E)   # the non-exiting sequence is scored at every checkpoint
    kv = 2 * 32 * 100 * 4096
    assert b == 32 * bf16 + 27 * int4 + heads + E + kv


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.timeout(300)
def test_replicas_world_size_2_gloo():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--dry-dist", "--gpus", "2", "--steps", "10",
           "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1   # rank 0 alone prints
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2
    assert out["max_time_s"] == 1.5          # the slower rank sets the time
    assert out["value"] == pytest.approx(2 * 4 * 10 / 1.5)


def test_measured_traffic_only_for_unchanged_sources(tmp_path):
    """The ncu traffic ratio is used only for its workload and while the GEMV
    sources hash to the digest recorded beside it."""
    digest = bench.gemv_source_digest()
    p = tmp_path / "summary.md"
    body = "# title\n\n| a | b |\n|---|---|\nworkload: `llama3.1-8b-b1`\ngemv_sources_sha256: `%s`\n" \
           "dram_bytes_per_launch: `1002`\nalgorithmic_bytes_per_launch: `1000`\n"
    p.write_text(body % digest)
    assert bench.measured_traffic_ratio("llama3.1-8b-b1", str(p)) == 1.002
    assert bench.measured_traffic_ratio("llama3.1-8b-b32", str(p)) is None
    p.write_text(body % ("0" * 16))
    assert bench.measured_traffic_ratio("llama3.1-8b-b1", str(p)) is None
    assert bench.measured_traffic_ratio("llama3.1-8b-b1", str(tmp_path / "missing.md")) is None
    # a capture on a small workload applies to the workloads it names
    p.write_text((body % digest).replace("llama3.1-8b-b1", "llama3.2-1b-b1")
                 + "applies_to: `llama3.1-8b-b1, llama3.2-1b-b1`\n")
    assert bench.measured_traffic_ratio("llama3.1-8b-b1", str(p)) == 1.002
    assert bench.measured_traffic_ratio("llama3.2-1b-b1", str(p)) == 1.002
    assert bench.measured_traffic_ratio("llama3.1-8b-b32", str(p)) is None


def test_source_digest_ignores_comments_only():
    a = "int f(int x) { // the sum\n  return x + 1; /* one */ }\n"
    b = "int f(int x) {\n  return x + 1;\n}\n// a note\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_similarity_criterion_reads_no_head_bytes():
    sh = synth.SHAPES["llama3.1-8b"]
    ck = synth.WORKLOADS["llama3.1-8b-b1"].checkpoints
    ctx = [2100]
    # a sequence still on the backbone at every checkpoint: the max-prob heads read T and E each time
    full = bench.step_bytes(sh, ck, [31], ctx, True)
    sts = bench.step_bytes(sh, ck, [31], ctx, True, "sts")
    nox = bench.step_bytes(sh, ck, [31], ctx, False)
    assert sts == nox
    assert full - sts == len(ck) * (sh.d_model * sh.d_model * 2 + sh.vocab * sh.d_model * 2)


def test_calibration_histogram_first_checkpoint_above_threshold():
    conf = [[0.5, 0.9], [0.1, 0.2], [0.6, 0.1], [0.3, 0.8]]
    assert bench.calibration_hist(conf, [0.4, 0.7], (4, 8), 32) == {4: 2, 8: 1, 31: 1}
    # strict: equal to the threshold stays
    assert bench.calibration_hist([[0.4, 0.7]], [0.4, 0.7], (4, 8), 32) == {31: 1}


def test_exit_head_token_byte_model():
    sh = synth.SHAPES["llama3.1-8b"]
    ck = synth.WORKLOADS["llama3.1-8b-b1"].checkpoints
    ctx = [2100]
    final = bench.step_bytes(sh, ck, [4], ctx, True)
    tok = bench.step_bytes(sh, ck, [4], ctx, True, "maxprob", "exit_head")
    m = bench.mat_list(sh)
    dead = sum(bench.w_bytes(*m[k], True) for k in ("o", "gateup", "down"))
    kv = 2100 * 2 * sh.n_kv_heads * sh.head_dim * 2
    assert final - tok == dead + kv + sh.vocab * sh.d_model * 2
    # a sequence that never exits reads the same either way
    assert bench.step_bytes(sh, ck, [31], ctx, True, "maxprob", "exit_head") == bench.step_bytes(sh, ck, [31], ctx, True)


def test_reference_arm_contract():
    """--impl reference times the oracle on the host and prints the base
    contract's line with impl, cpu_baseline and e2e (no host-device copies);
    under a multi-rank launch only rank 0 works and prints."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny-b1",
           "--steps", "1", "--warmup", "3"]
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=root, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["metric"] == bench.METRIC and line["config"]["workload"] == "tiny-b1"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    env1 = dict(env, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out1 = subprocess.run(cmd, capture_output=True, text=True, env=env1, cwd=root, timeout=300)
    assert out1.returncode == 0 and "{" not in out1.stdout, (out1.stdout, out1.stderr[-2000:])
