"""Parity at the CodeLlama-34B layer shape (d=8192, 64 query / 8 KV heads,
hd 128, F=22016, V=32016), truncated to two layers so that the fp64 oracle
stays small: batch 1 on the GEMV (activation rows of up to 22016 values
staged in shared memory, grouped-query attention with 8 query heads per KV
head), and batches 8 and 10 on the tensor-core GEMM with K=22016 (eight rows
of 8192 values no longer fit the GEMV's staging area, so a batch-8 step
runs there too, with RMSNorm kernels)."""
import numpy as np
import pytest

import synth
from tests import parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPE = synth.Shape("codellama-34b-2-layers", 2, 8192, 64, 8, 128, 22016, 32016)
W34 = synth.Workload("codellama-34b-2-layers", SHAPE, (0,), 8, 12, 2, 1238)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("batch", [1, 8, 10])
def test_codellama34b_layer_shape(batch):
    eng = parity.load_engine(W34, max_batch=batch, max_seq_len=32)
    orc = parity.build_oracle(W34, max_batch=batch, max_seq_len=32, cache_bytes=24 << 30)
    pr = synth.prompts(SHAPE, 77 + batch, [6 + i for i in range(batch)])
    _, _, n = eng.step_io(batch, True)
    assert n == 1 + (7 if batch > 1 else 5) * SHAPE.n_layers + (3 if batch > 1 else 2) + (2 if batch > 1 else 1)
    # step 0 exits every sequence at layer 0 (layer 1 on the int4 copy), step 1 none
    gps = [[-np.inf], [np.inf]]
    st = parity.drive(eng, orc, pr, gps[0], 2, gamma_per_step=gps)
    assert [sorted(set(int(x) for x in e)) for e in st.gpu_exits] == [[0], [1]]
    print("34B shape b=%d parity:" % batch, st)
    parity.check_kv(eng, orc)
    eng.close()
