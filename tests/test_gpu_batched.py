"""Parity of the decode step at batch sizes above the GEMV's staging limit,
where the projections and heads run on the tensor-core GEMM (tcgen05, fp32
accumulators in tensor memory): the tiny model at batch 12 with mixed exit
depths every step, and the Llama-3.2-1B shape (128256-row vocabulary head)
at batch 10 on a short workload."""
import numpy as np
import pytest

import synth
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import early_exit_decoding_layer_gb300 as ee  # noqa: E402

TINY = synth.WORKLOADS["tiny-b1"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_launches_per_step_count_both_sub_batches():
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=48)
    L, nck = TINY.shape.n_layers, len(TINY.checkpoints)
    _, _, n1 = eng.step_io(1, True)
    _, _, n12 = eng.step_io(12, True)
    assert n1 == 1 + 5 * L + 2 * nck + 1          # GEMV path: norms applied while staging
    # norm kernels; one tensor-core launch serves both sub-batch lists
    assert n12 == 1 + (1 + 4 + 2) * L + 3 * nck + 2
    _, _, n12_off = eng.step_io(12, False)
    assert n12_off == 1 + (1 + 4 + 2) * L + 2
    eng.close()


def test_tiny_batch12_mixed_exits():
    """12 ragged sequences; per-step thresholds of -inf/+inf per checkpoint so
    that the full and exit sub-batches change every step (both GEMM modes,
    list compaction by the tensor-core head)."""
    B = 12
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=16, max_seq_len=64)
    lens = [5, 16, 17, 31, 9, 12, 20, 3, 33, 15, 8, 26]
    pr = synth.prompts(TINY.shape, 41, lens)
    rng = np.random.default_rng(3)
    gps = [[rng.choice([-np.inf, np.inf], p=[0.3, 0.7]) for _ in TINY.checkpoints] for _ in range(10)]
    st = parity.drive(eng, orc, pr, gps[0], 10, gamma_per_step=gps)
    seen = set(int(x) for e in st.gpu_exits for x in e)
    assert len(st.gpu_exits[0]) == B
    assert seen >= {1, 3}
    print("tiny b=12 parity:", st)
    parity.check_kv(eng, orc)
    eng.close()


def test_tiny_batch12_calibrated_thresholds():
    """Thresholds between the confidences, so some sequences of a step exit
    and others do not (decisions inside the window are excused)."""
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=16, max_seq_len=64)
    pr = synth.prompts(TINY.shape, 43, [10 + 2 * i for i in range(12)])
    # confidences of the oracle at gamma = +inf over 2 steps: thresholds at their median
    o2 = parity.build_oracle(TINY, max_batch=16, max_seq_len=64)
    o2.set_thresholds(np.full(len(TINY.checkpoints), np.inf))
    tok = o2.prefill(pr)
    confs = []
    for _ in range(2):
        r = o2.decode_step(tok)
        confs.append(r.conf)
        tok = r.next_tokens
    gamma = np.median(np.concatenate(confs, axis=0), axis=0)
    st = parity.drive(eng, orc, pr, gamma, 8)
    print("tiny b=12 calibrated:", st)
    eng.close()


def test_llama1b_shape_batch10():
    """Llama-3.2-1B shape at batch 10: 24- to 60-token prompts, 3 steps, exits
    forced at the first checkpoint for half of the steps."""
    w = synth.WORKLOADS["llama3.2-1b-b1"]
    eng = parity.load_engine(w, max_batch=10, max_seq_len=72)
    orc = parity.build_oracle(w, max_batch=10, max_seq_len=72, cache_bytes=16 << 30)
    pr = synth.prompts(w.shape, w.seed + 5, [24 + 4 * i for i in range(10)])
    inf = np.inf
    gps = [[-inf, inf, inf], [inf, inf, inf], [inf, -inf, inf]]
    st = parity.drive(eng, orc, pr, gps[0], 3, gamma_per_step=gps)
    assert [sorted(set(int(x) for x in e)) for e in st.gpu_exits] == [[4], [15], [8]]
    print("1B b=10 parity:", st)
    eng.close()


def test_tiny_batch40_wide_b_tile():
    """40 ragged sequences: lists of more than 32 sequences take the wide B
    tile of the tensor-core GEMM (64 hi + 64 lo rows, three stages) for the
    full sub-batch, and 40 exit rows on the int4 path when all exit early."""
    B = 40
    eng = parity.load_engine(TINY, max_batch=64, max_seq_len=48)
    orc = parity.build_oracle(TINY, max_batch=64, max_seq_len=48)
    lens = [3 + (7 * i) % 29 for i in range(B)]
    pr = synth.prompts(TINY.shape, 47, lens)
    inf = np.inf
    ck = len(TINY.checkpoints)
    gps = [[inf] * ck, [-inf] + [inf] * (ck - 1), [inf] * ck, [inf] + [-inf] * (ck - 1)]
    st = parity.drive(eng, orc, pr, gps[0], len(gps), gamma_per_step=gps)
    assert len(st.gpu_exits[0]) == B
    assert [sorted(set(int(x) for x in e)) for e in st.gpu_exits] == [
        [TINY.shape.n_layers - 1], [TINY.checkpoints[0]], [TINY.shape.n_layers - 1], [TINY.checkpoints[1]]]
    print("tiny b=40 parity:", st)
    parity.check_kv(eng, orc)
    eng.close()


def test_profiled_step_records_own_times_and_lists():
    """A profiled step at batch 12: every projection and head launch carries
    its own kernel time (globaltimer stamps, no launch gap), the tensor-core
    GEMM launches name the lists they serve (the full list alone up to the
    first checkpoint, both lists after it), the step launches as many
    kernels as ee_step_io states, and the profiled step's tokens and exits
    equal those of the graph-replayed step."""
    B = 12
    lens = [5, 16, 17, 31, 9, 12, 20, 3, 33, 15, 8, 26]
    pr = synth.prompts(TINY.shape, 41, lens)
    gamma = [-np.inf, np.inf]   # everyone leaves at the first checkpoint
    runs = []
    for profile in (False, True):
        eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
        eng.set_thresholds(np.asarray(gamma))
        tok = eng.prefill(pr)
        tok, ex = eng.decode_step(tok)
        eng.set_profile(profile)
        tok2, ex2 = eng.decode_step(tok)
        runs.append((tok2.copy(), ex2.copy(), eng.profile_read() if profile else None, eng.step_io(B, True)[2]))
        eng.close()
    assert np.array_equal(runs[0][0], runs[1][0]) and np.array_equal(runs[0][1], runs[1][1])
    recs = runs[1][2]
    assert len(recs) == runs[1][3], (len(recs), runs[1][3])
    proj = [r for r in recs if r[0] in ("qkv", "o", "gateup", "down", "head_t", "head_e", "final_head")]
    assert proj and all(r[3] > 0 for r in proj), [r for r in proj if r[3] <= 0][:4]
    assert all(r[3] <= r[2] * 1.5 + 0.05 for r in proj)     # own time within the event pair (loose)
    ck = TINY.checkpoints[0]
    # after the first checkpoint one launch serves both lists (bf16 units, then int4 units)
    late = [r for r in proj if r[0] in ("qkv", "o", "gateup", "down") and r[1] > ck]
    assert late and {r[4] for r in late} == {"both"}, late[:4]
    early = [r for r in proj if r[0] in ("qkv", "o", "gateup", "down") and r[1] <= ck]
    assert early and {r[4] for r in early} == {"full"}, early[:4]
    assert all(r[4] == "both" for r in recs if r[0] in ("attn", "begin", "norm"))
