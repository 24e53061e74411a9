"""End-to-end parity of the early-exit decode step (C ABI) against the CPU
oracle: the tiny workload as configured, the no-exit and all-exit limits,
KV-slot coverage and bookkeeping, batch independence, graph replay, and the
Llama-3.2-1B shape on a truncated workload."""
import json

import numpy as np
import pytest

import oracle
import synth
from tests import parity
from tests.conftest import golden_path

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import early_exit_decoding_layer_gb300 as ee  # noqa: E402

TINY = synth.WORKLOADS["tiny-b1"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module")
def tiny_engine():
    eng = parity.load_engine(TINY, max_batch=4, max_seq_len=80)
    yield eng
    eng.close()


def tiny_gamma():
    return json.load(open(golden_path("tiny_oracle_trace.json")))["gamma"]


def test_int4_copies_bit_exact(tiny_engine):
    for j in range(TINY.shape.n_layers):
        lw = synth.layer_weights(TINY.shape, TINY.seed, j)
        for m in synth.MATS:
            q, s = oracle.quantize_int4_group(lw[m], 128)
            gp, gs = tiny_engine.debug_int4(j, m)
            assert np.array_equal(gp, oracle.pack_int4(q)), (j, m)
            assert np.array_equal(gs, s), (j, m)


def test_tiny_workload_parity(tiny_engine):
    """The configured tiny workload: 32-token prompt, 16 steps, gamma at the
    oracle's 40th percentile."""
    lens, prompts = synth.workload_inputs(TINY)
    orc = parity.build_oracle(TINY, max_batch=4, max_seq_len=80)
    st = parity.drive(tiny_engine, orc, prompts, tiny_gamma(), TINY.steps)
    ref = json.load(open(golden_path("tiny_oracle_trace.json")))["trace"]
    # the GPU's trace equals the stored oracle trace except at excused steps
    diff = sum(int(a != b) for a, b in zip(np.concatenate(st.gpu_exits), np.ravel(ref["exit_layers"])))
    assert diff == st.exit_mismatch
    assert st.token_mismatch == 0 or st.token_mismatch <= 1
    print("tiny parity:", st)
    parity.check_kv(tiny_engine, orc)


def test_no_exit_and_exit_disabled(tiny_engine):
    lens, prompts = synth.workload_inputs(TINY)
    orc = parity.build_oracle(TINY, max_batch=4, max_seq_len=80)
    inf = [np.inf] * len(TINY.checkpoints)
    st = parity.drive(tiny_engine, orc, prompts, inf, 10)
    assert all((e == TINY.shape.n_layers - 1).all() for e in st.gpu_exits)
    # the forced no-exit baseline (no head evaluated) emits the same tokens and states
    tiny_engine.set_exit_enabled(False)
    first = tiny_engine.prefill(prompts)
    tok = first
    for k in range(10):
        n, e = tiny_engine.decode_step(tok)
        assert np.array_equal(n, st.gpu_tokens[k]) and (e == TINY.shape.n_layers - 1).all()
        assert np.isnan(tiny_engine.debug_conf()).all()
        tok = n
    tiny_engine.set_exit_enabled(True)


def test_exit_at_layer0_all_int4():
    """gamma = -inf with one checkpoint at layer 0: layers 1..L-1 always run on
    the int4 copies."""
    eng = parity.load_engine(TINY, max_batch=2, max_seq_len=64, checkpoints=(0,))
    orc = parity.build_oracle(TINY, max_batch=2, max_seq_len=64, checkpoints=(0,))
    pr = synth.prompts(TINY.shape, 3, [20, 9])
    st = parity.drive(eng, orc, pr, [-np.inf], 8)
    assert all((e == 0).all() for e in st.gpu_exits)
    parity.check_kv(eng, orc)
    eng.close()


def test_kv_coverage_mixed_exits():
    """Ragged prompts across block boundaries and per-step thresholds that force
    a different exit pattern every step: every slot is written, by bf16 or int4
    layers, and the block tables match the oracle's bookkeeping."""
    eng = parity.load_engine(TINY, max_batch=3, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=3, max_seq_len=64)
    pr = synth.prompts(TINY.shape, 11, [15, 16, 17])
    rng = np.random.default_rng(0)
    gps = [[rng.choice([-np.inf, np.inf]) for _ in TINY.checkpoints] for _ in range(20)]
    st = parity.drive(eng, orc, pr, gps[0], 20, gamma_per_step=gps)
    seen = set(int(x) for e in st.gpu_exits for x in e)
    assert seen >= {1, 2, 3}
    parity.check_kv(eng, orc)
    eng.close()


def test_batch_independence(tiny_engine):
    pr = synth.prompts(TINY.shape, 21, [9, 30, 17])
    g = tiny_gamma()
    tiny_engine.set_thresholds(g)
    tb = tiny_engine.prefill(pr)
    seqs_b = [[] for _ in pr]
    tok = tb
    for _ in range(6):
        n, e = tiny_engine.decode_step(tok)
        for s in range(len(pr)):
            seqs_b[s].append((int(n[s]), int(e[s])))
        tok = n
    for s in range(len(pr)):
        t1 = tiny_engine.prefill([pr[s]])
        assert t1[0] == tb[s]
        for k in range(6):
            n, e = tiny_engine.decode_step(t1)
            assert (int(n[0]), int(e[0])) == seqs_b[s][k], (s, k)
            t1 = n


def test_graph_and_eager_identical(tiny_engine):
    lens, prompts = synth.workload_inputs(TINY)
    tiny_engine.set_thresholds(tiny_gamma())
    out = []
    for use_graph in (True, False):
        tiny_engine.set_use_graph(use_graph)
        tiny_engine.set_debug(True)
        tok = tiny_engine.prefill(prompts)
        trace = []
        for _ in range(6):
            n, e = tiny_engine.decode_step(tok)
            trace.append((n.copy(), e.copy(), tiny_engine.debug_hidden(3).copy()))
            tok = n
        out.append(trace)
    tiny_engine.set_use_graph(True)
    for a, b in zip(*out):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        assert np.array_equal(a[2], b[2])


def test_prepacked_int4_equals_library_quantiser(tiny_engine):
    eng2 = parity.load_engine(TINY, max_batch=4, max_seq_len=80, int4_from_oracle=True)
    lens, prompts = synth.workload_inputs(TINY)
    g = [-np.inf, np.inf]  # every step exits at layer 1 -> layers 2, 3 on int4
    res = []
    for e in (tiny_engine, eng2):
        e.set_thresholds(g)
        e.set_debug(True)
        tok = e.prefill(prompts)
        tr = []
        for _ in range(4):
            n, x = e.decode_step(tok)
            tr.append((n.copy(), x.copy(), e.debug_hidden(3).copy()))
            tok = n
        res.append(tr)
    for a, b in zip(*res):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    eng2.close()


def test_host_validation_errors(tiny_engine):
    with pytest.raises(ee.EEError) as ex:
        tiny_engine.prefill([[TINY.shape.vocab]])
    assert ex.value.status == 1
    with pytest.raises(ee.EEError) as ex:
        tiny_engine.prefill([[1] * 80])
    assert ex.value.status == 3
    with pytest.raises(ee.EEError) as ex:
        tiny_engine.prefill([[1]] * 5)
    assert ex.value.status == 3
    tiny_engine.reset()
    with pytest.raises(ee.EEError) as ex:
        tiny_engine.decode_step([])
    # capacity: decoding past max_seq_len fails cleanly and leaves the context usable
    tok = tiny_engine.prefill([[5] * 78])
    n, e = tiny_engine.decode_step(tok)
    n, e = tiny_engine.decode_step(n)
    with pytest.raises(ee.EEError) as ex:
        tiny_engine.decode_step(n)
    assert ex.value.status == 3
    tiny_engine.prefill([[1, 2, 3]])


def test_llama1b_shape_truncated():
    """Llama-3.2-1B shape (16 layers, d=2048, 32/8 heads, hd 64, F=8192,
    V=128256): 64-token prompt, 6 steps; an exit forced at the second
    checkpoint (layer 8) on some steps so both weight paths run."""
    w = synth.WORKLOADS["llama3.2-1b-b1"]
    eng = parity.load_engine(w, max_batch=1, max_seq_len=80)
    orc = parity.build_oracle(w, max_batch=1, max_seq_len=80, cache_bytes=16 << 30)
    pr = synth.prompts(w.shape, w.seed, [64])
    inf = np.inf
    gps = [[inf, -inf, inf], [inf, inf, inf], [-inf, inf, inf], [inf, inf, inf], [inf, inf, -inf],
           [inf, -inf, inf]]
    st = parity.drive(eng, orc, pr, gps[0], 6, gamma_per_step=gps)
    assert [int(e[0]) for e in st.gpu_exits] == [8, 15, 4, 15, 12, 8]
    print("1B parity:", st)
    eng.close()
