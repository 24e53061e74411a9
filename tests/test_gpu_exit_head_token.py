"""Parity of the exit-head token source (the CALM article §3.1: an exited
token is the exit head's prediction; its remaining layers still write their
K/V, in the last layer through the QKV projection only) through the C ABI
against the CPU oracle: the tiny workload at batch 1 and at batch 12 on the
tensor-core path, with every K/V slot checked."""
import json

import numpy as np
import pytest

import synth
from tests import parity
from tests.conftest import golden_path

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny-b1"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_tiny_exit_head_tokens():
    lens, prompts = synth.workload_inputs(TINY)
    gamma = json.load(open(golden_path("tiny_oracle_trace.json")))["gamma"]
    eng = parity.load_engine(TINY, max_batch=4, max_seq_len=80)
    orc = parity.build_oracle(TINY, max_batch=4, max_seq_len=80, token_source="exit_head")
    inf = np.inf
    gps = [gamma] * 6 + [[-inf, inf], [inf, -inf], [inf, inf], gamma]
    st = parity.drive(eng, orc, prompts, gps[0], len(gps), gamma_per_step=gps)
    exits = [int(e[0]) for e in st.gpu_exits]
    assert exits[6] == 1 and exits[7] == 2 and exits[8] == 3, exits
    print("tiny exit-head tokens:", st)
    parity.check_kv(eng, orc)
    # the engine leaves the mode when asked
    eng.set_token_source("final")
    eng.close()


def test_tiny_batch12_exit_head_tokens():
    lens = [5, 16, 17, 31, 9, 12, 20, 3, 33, 15, 8, 26]
    pr = synth.prompts(TINY.shape, 51, lens)
    rng = np.random.default_rng(9)
    gps = [[rng.choice([-np.inf, np.inf], p=[0.35, 0.65]) for _ in TINY.checkpoints] for _ in range(6)]
    eng = parity.load_engine(TINY, max_batch=16, max_seq_len=64)
    orc = parity.build_oracle(TINY, max_batch=16, max_seq_len=64, token_source="exit_head")
    st = parity.drive(eng, orc, pr, gps[0], len(gps), gamma_per_step=gps)
    seen = set(int(x) for e in st.gpu_exits for x in e)
    assert seen >= {1, 3}, seen
    print("tiny b=12 exit-head tokens:", st)
    parity.check_kv(eng, orc)
    eng.close()


def test_exit_head_tokens_need_the_exit_head_criterion():
    import early_exit_decoding_layer_gb300 as ee
    eng = parity.load_engine(TINY, max_batch=1, max_seq_len=40)
    eng.set_token_source("exit_head")
    eng.set_exit_criterion("sts")
    tok = eng.prefill([[1, 2, 3]])
    with pytest.raises(ee.EEError) as e:
        eng.decode_step(tok)
    assert e.value.status == 2   # EE_ERR_STATE
    eng.set_exit_criterion("maxprob")
    eng.decode_step(tok)
    eng.close()
