"""Parity of the state-transition-similarity exit criterion ("River-LLM 深度解析"
§5.1-5.3: a token leaves the full-precision path at a checkpoint layer when
the cosine between that layer's input and output states is above the layer's
threshold) through the C ABI against the CPU oracle: the tiny workload with
thresholds at the oracle's 40th percentile, batch 12 on the tensor-core path
with mixed thresholds, and the Llama-3.2-1B shape on a short workload."""
import numpy as np
import pytest

import oracle
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


def oracle_taus(w, prompts, pcts, max_batch, max_seq_len, steps=8, cache_bytes=4 << 30):
    """tau_l = percentiles of the oracle's no-exit similarity scores at layer l."""
    o = parity.build_oracle(w, max_batch=max_batch, max_seq_len=max_seq_len, criterion="sts",
                            cache_bytes=cache_bytes)
    gam, S = oracle.calibrate_gammas(o, prompts, steps, pcts)
    return gam, S


def test_launches_per_step_similarity_criterion():
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=48)
    L, nck = TINY.shape.n_layers, len(TINY.checkpoints)
    eng.set_exit_criterion("sts")
    _, _, n1 = eng.step_io(1, True)
    assert n1 == 1 + 5 * L + nck + 1        # one decision launch per checkpoint, no head
    eng.set_exit_criterion("maxprob")
    _, _, n1h = eng.step_io(1, True)
    assert n1h == 1 + 5 * L + 2 * nck + 1
    eng.close()


def test_tiny_similarity_criterion_calibrated():
    lens, prompts = synth.workload_inputs(TINY)
    gam, S = oracle_taus(TINY, prompts, (40.0,), 4, 80)
    assert np.all(np.abs(S) <= 1.0 + 1e-12)
    eng = parity.load_engine(TINY, max_batch=4, max_seq_len=80)
    orc = parity.build_oracle(TINY, max_batch=4, max_seq_len=80, criterion="sts")
    st = parity.drive(eng, orc, prompts, gam[40.0], TINY.steps)
    exits = [int(e[0]) for e in st.gpu_exits]
    assert len(set(exits)) >= 2, exits          # thresholds at P40 give exits at several depths
    print("tiny sts parity:", st, "exits", exits)
    parity.check_kv(eng, orc)
    eng.close()


def test_tiny_batch12_similarity_mixed_thresholds():
    """Batch 12 (tensor-core projections): thresholds at the 40th and 70th
    percentiles and forced limits, so the sub-batches change every step."""
    B = 12
    lens = [5, 16, 17, 31, 9, 12, 20, 3, 33, 15, 8, 26]
    pr = synth.prompts(TINY.shape, 43, lens)
    gam, _ = oracle_taus(TINY, pr, (40.0, 70.0), 16, 64, steps=4)
    inf = np.inf
    gps = [gam[40.0], gam[70.0], [-inf, inf], gam[40.0], [inf, -inf], gam[70.0]]
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=16, max_seq_len=64, criterion="sts")
    st = parity.drive(eng, orc, pr, gps[0], len(gps), gamma_per_step=gps)
    seen = set(int(x) for e in st.gpu_exits for x in e)
    assert len(st.gpu_exits[0]) == B and seen >= {1, 2, 3}, seen
    print("tiny b=12 sts parity:", st)
    parity.check_kv(eng, orc)
    eng.close()


def test_llama1b_shape_similarity_criterion():
    w = synth.WORKLOADS["llama3.2-1b-b1"]
    pr = synth.prompts(w.shape, w.seed, [48])
    gam, S = oracle_taus(w, pr, (40.0,), 1, 64, steps=4, cache_bytes=16 << 30)
    eng = parity.load_engine(w, max_batch=1, max_seq_len=64)
    orc = parity.build_oracle(w, max_batch=1, max_seq_len=64, criterion="sts", cache_bytes=16 << 30)
    inf = np.inf
    gps = [gam[40.0], [inf, -inf, inf], gam[40.0], [-inf, inf, inf], gam[40.0]]
    st = parity.drive(eng, orc, pr, gps[0], len(gps), gamma_per_step=gps)
    ex = [int(e[0]) for e in st.gpu_exits]
    assert ex[1] == 8 and ex[3] == 4, ex
    print("1B sts parity:", st, "exits", ex, "scores", S.mean(axis=(0, 1)))
    eng.close()


def test_tiny_batch12_similarity_batch_rule():
    """The batch rule (River-LLM §5.2): the sequences on the full path exit
    together on the minimum score; thresholds at percentiles of the batch
    minimum, so the batch exits at several depths over the steps."""
    lens = [5, 16, 17, 31, 9, 12, 20, 3, 33, 15, 8, 26]
    pr = synth.prompts(TINY.shape, 47, lens)
    o = parity.build_oracle(TINY, max_batch=16, max_seq_len=64, criterion="sts_batch")
    gam, S = oracle.calibrate_gammas(o, pr, 4, (30.0, 60.0))
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=16, max_seq_len=64, criterion="sts_batch")
    gps = [gam[30.0], gam[60.0], gam[30.0], gam[60.0], gam[30.0]]
    st = parity.drive(eng, orc, pr, gps[0], len(gps), gamma_per_step=gps)
    for e in st.gpu_exits:
        assert len(set(int(x) for x in e)) == 1, e    # the batch exits together
    print("tiny b=12 sts batch-rule parity:", st, [int(e[0]) for e in st.gpu_exits])
    eng.close()
