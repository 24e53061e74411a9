"""End-to-end parity of the whole Llama-3.1-8B-shape model (32 layers, d=4096,
32 query / 8 KV heads, hd 128, F=14336, V=128256, checkpoints at layers
4, 8, ..., 28) through the C ABI against the CPU oracle, on the seeded
weights of the 8B workloads.

* batch 1 (the GEMV path): a 160-token prompt and 8 decode steps that mix
  the oracle-calibrated thresholds with forced exits at the first and the
  last checkpoint (layers 4 and 28) and a no-exit step;
* batch 32 (the tensor-core GEMM path, N = 28672 and K = 14336, narrow B
  tile): ragged prompts of 13..47 tokens whose decode positions cross
  16-token block boundaries, 4 steps at the oracle's 40th and 70th
  percentile thresholds (sequences exit at mixed depths).

Every step compares the residual stream after every layer (relative L2
<= 1e-2), the exit layers and tokens (identical outside the stated windows)
and the confidences; the K/V slots and block tables are checked at the end.
The oracle (float64) keeps its converted layers in host memory, about 110 GB
at this shape."""
import gc
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

W1 = synth.WORKLOADS["llama3.1-8b-b1"]
W32 = synth.WORKLOADS["llama3.1-8b-b32"]
SHAPE = W1.shape
CK = W1.checkpoints
MAX_SEQ = 192


def oracle_gamma(name, p):
    return json.load(open(golden_path("oracle_gammas.json")))[name]["gamma"]["p%g" % p]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


class Model:
    """The engine and the oracle over one workload's seeded weights; the bf16
    layers are drawn once and serve both.  close() frees the host copies."""

    def __init__(self, w, int4_from):
        self.layers = [synth.layer_weights(SHAPE, w.seed, j) for j in range(SHAPE.n_layers)]
        self.eng = ee.DecodeEngine(SHAPE, CK, w.batch, MAX_SEQ)
        for j in range(SHAPE.n_layers):
            self.eng.load_layer(j, self.layers[j])
        E = synth.embedding(SHAPE, w.seed)
        T = [synth.exit_transform(SHAPE, w.seed, c) for c in range(len(CK))]
        self.eng.load_shared(E, synth.final_gain(SHAPE), T)
        self.cfg = oracle.ModelConfig.from_shape(SHAPE, CK)
        L = self.layers
        self.W = oracle.Weights(self.cfg, lambda j: L[j], E, synth.final_gain(SHAPE), T,
                                cache_bytes=160 << 30)
        keys = [(j, False) for j in range(SHAPE.n_layers)]
        keys += [(j, True) for j in range(int4_from, SHAPE.n_layers)]
        self.W.warm(keys, workers=16)
        self.orc = oracle.Oracle(self.cfg, self.W, w.batch, MAX_SEQ)

    def close(self):
        self.eng.close()
        self.orc = self.W = None
        self.layers.clear()
        gc.collect()


def test_llama8b_batch1_mixed_exits():
    m = Model(W1, CK[0] + 1)
    try:
        lens, prompts = synth.workload_inputs(W1)
        pr = [list(map(int, prompts[0][:160]))]
        g40 = oracle_gamma(W1.name, 40)
        inf = np.inf
        first_only = [-inf] + [inf] * (len(CK) - 1)       # exit at layer 4
        last_only = [inf] * (len(CK) - 1) + [-inf]        # exit at layer 28
        gps = [g40, first_only, g40, last_only, [inf] * len(CK), g40, first_only, g40]
        st = parity.drive(m.eng, m.orc, pr, gps[0], len(gps), gamma_per_step=gps)
        ex = [int(e[0]) for e in st.gpu_exits]
        assert ex[1] == 4 and ex[6] == 4 and ex[3] == 28 and ex[4] == SHAPE.n_layers - 1, ex
        print("8B b=1:", st)
        parity.check_kv(m.eng, m.orc)
    finally:
        m.close()


def test_llama8b_batch32_tensor_core_mixed_exits():
    m = Model(W32, CK[0] + 1)
    try:
        lens = [13 + (s * 11) % 35 for s in range(W32.batch)]     # 13..47, ragged
        pr = synth.prompts(SHAPE, W32.seed, lens)
        gps = [oracle_gamma(W32.name, 40), oracle_gamma(W32.name, 70),
               oracle_gamma(W32.name, 40), oracle_gamma(W32.name, 70)]
        st = parity.drive(m.eng, m.orc, pr, gps[0], len(gps), gamma_per_step=gps)
        depths = set(int(x) for e in st.gpu_exits for x in e)
        assert len(depths) >= 3, depths       # mixed exit depths across the batch
        print("8B b=32:", st, "exit depths", sorted(depths))
        parity.check_kv(m.eng, m.orc)
    finally:
        m.close()
