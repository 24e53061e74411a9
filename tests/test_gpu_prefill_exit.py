"""Parity of sequence-level exit in prefill ("River-LLM 深度解析" §6.1: all
tokens of a prompt leave the full-precision path at one checkpoint, the one
where the minimum of their state transition similarities first clears the
threshold; the later layers run on the int4 copies and fill the K/V cache)
through the C ABI against the CPU oracle: prompts that exit at different
layers or not at all, every K/V slot compared, then decode steps."""
import numpy as np
import pytest

import synth
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny-b1"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_tiny_prefill_sequence_level_exit():
    lens = [9, 23, 16, 31]
    pr = synth.prompts(TINY.shape, 61, lens)
    # the oracle's per-prompt minima with no exit fix thresholds that split the batch
    probe = parity.build_oracle(TINY, max_batch=4, max_seq_len=64)
    probe.prefill(pr, exit_tau=[np.inf, np.inf])
    lo = probe.prefill_scores            # [prompt, checkpoint]
    assert np.all(np.isfinite(lo))
    tau0 = float(np.median(lo[:, 0]))    # about half the prompts leave at layer 1
    taus = [[tau0, -np.inf],             # the rest leave at layer 2
            [-np.inf, np.inf],           # every prompt leaves at layer 1
            [np.inf, np.inf]]            # none: the plain prefill
    for tau in taus:
        eng = parity.load_engine(TINY, max_batch=4, max_seq_len=64)
        orc = parity.build_oracle(TINY, max_batch=4, max_seq_len=64)
        gamma = [np.inf, np.inf]
        st = parity.drive(eng, orc, pr, gamma, 3, prefill_tau=tau)
        ex = eng.prefill_exit_layers()
        print("prefill exit", tau, ex.tolist(), st)
        if tau[0] == tau0:
            assert set(ex.tolist()) == {1, 2}
        parity.check_kv(eng, orc)
        eng.close()
