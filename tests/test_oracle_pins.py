"""Pins of the CPU oracle against facts fixed outside it: hand-worked examples
(tests/golden), closed forms, textbook reductions, independent library
routines and brute force on tiny inputs.  CPU only."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth
from oracle import model as om
from tests.conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------- int4 exit copies

def f32_bits_to_bf16(vals):
    """bf16 patterns of values that are exactly representable in bf16."""
    a = np.asarray(vals, dtype=np.float32)
    u = a.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def test_quantiser_hand_worked_example():
    g = read_golden("int4_quant_example.txt")
    w = f32_bits_to_bf16(g["w"])[None, :]
    q, s = oracle.quantize_int4_group(w, group=g["group"][0])
    assert q[0].tolist() == g["q"]
    assert s[0].tolist() == g["scale_bits"]
    assert oracle.bf16_to_f32(s[0]).tolist() == g["scale"]
    packed = oracle.pack_int4(q)
    assert packed[0].tolist() == g["packed"]
    deq = oracle.dequant_int4(q, s, group=g["group"][0])
    assert deq[0].tolist() == g["dequant"]


def test_nibble_roundtrip_all_values():
    vals = np.arange(-8, 8, dtype=np.int8)
    q = np.stack([vals, vals[::-1]])  # every value in both nibble positions
    p = oracle.pack_int4(q)
    assert p.shape == (2, 8)
    assert np.array_equal(oracle.unpack_int4(p, 16), q)
    # low nibble is the even column: column 0 = -8 -> 0x8, column 1 = -7 -> 0x9
    assert p[0, 0] == 0x98


def test_nibble_roundtrip_random():
    rng = np.random.default_rng(0)
    q = rng.integers(-8, 8, size=(33, 704)).astype(np.int8)
    assert np.array_equal(oracle.unpack_int4(oracle.pack_int4(q), 704), q)


def test_exactly_representable_weights_dequantise_exactly():
    # rows whose groups hold k * s with |k| <= 7 and amax = 7 s: scale is s exactly
    s_vals = np.array([2.0 ** -7, 2.0 ** -5, 0.25], dtype=np.float32)
    rng = np.random.default_rng(1)
    rows = []
    for s in s_vals:
        k = rng.integers(-7, 8, size=256).astype(np.float32)
        k[0], k[128] = 7, -7
        rows.append(k * s)
    w = f32_bits_to_bf16(np.stack(rows))
    q, sb = oracle.quantize_int4_group(w, 128)
    deq = oracle.dequant_int4(q, sb, 128)
    assert np.array_equal(deq, oracle.bf16_to_f64(w))


def test_partial_last_group_and_zero_group():
    # in = 704 = 5*128 + 64 (the tiny model's down projection)
    rng = np.random.default_rng(2)
    w32 = (rng.standard_normal((3, 704)) * 0.02).astype(np.float32)
    w32[1, 128:256] = 0.0
    w = om.f32_to_bf16_bits(w32)
    q, s = oracle.quantize_int4_group(w, 128)
    assert s.shape == (3, 6)
    assert s[1, 1] == 0 and np.all(q[1, 128:256] == 0)
    # the partial group's scale only sees its own 64 columns
    wf = oracle.bf16_to_f32(w)
    amax = np.max(np.abs(wf[:, 640:]), axis=1)
    expect = om.f32_to_bf16_bits((amax / np.float32(7)).astype(np.float32))
    assert np.array_equal(s[:, 5], expect)
    # every code within range and every error within half a scale step (+clamp slack)
    deq = oracle.dequant_int4(q, s, 128)
    sc = oracle.bf16_to_f64(s)[:, np.arange(704) // 128]
    assert q.min() >= -8 and q.max() <= 7
    assert np.all(np.abs(deq - wf) <= 0.5 * sc * (1 + 2 ** -7) + 1e-30)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1.0078125 -> even (1.0)
    # 1 + 3*2^-8 is halfway between 1.0078125 and 1.015625 -> even (1.015625)
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    b = om.f32_to_bf16_bits(x)
    assert b.tolist() == [0x3F80, 0x3F82, 0x3F81]


def test_w4a16_size_matches_page():
    g = read_golden("w4a16_size.txt")
    sh = synth.SHAPES["llama3.1-8b"]
    mats = [(sh.n_heads * sh.head_dim + 2 * sh.n_kv_heads * sh.head_dim, sh.d_model),
            (sh.d_model, sh.n_heads * sh.head_dim), (2 * sh.ffn_dim, sh.d_model),
            (sh.d_model, sh.ffn_dim)]
    bf = sum(n * k * 2 for n, k in mats)
    rng = np.random.default_rng(3)
    # packed bytes from the oracle's own packer on one row per matrix, scaled by rows
    q4 = 0
    for n, k in mats:
        q = rng.integers(-8, 8, size=(1, k)).astype(np.int8)
        _, s = oracle.quantize_int4_group(np.zeros((1, k), np.uint16), 128)
        q4 += n * (oracle.pack_int4(q).nbytes + s.nbytes)
    assert bf == g["bf16_layer_bytes"][0] and q4 == g["int4_layer_bytes"][0]
    pct = 100 * (1 - q4 / bf)
    assert g["percent_smaller_min"][0] <= pct <= g["percent_smaller_max"][0]


# --------------------------------------------------------------- layer pieces

def test_linear_matches_torch_functional_linear():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5))
    W = rng.standard_normal((7, 5))
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(W)).numpy()
    assert np.allclose(oracle.linear(x, W), ref, rtol=1e-14, atol=1e-14)
    # orientation on a square matrix: W[i, j] = 1 maps input j to output i
    W = np.zeros((4, 4))
    W[1, 3] = 1.0
    assert oracle.linear(np.array([0, 0, 0, 5.0]), W).tolist() == [0, 5.0, 0, 0]


def test_rmsnorm_constant_vector_closed_form():
    eps = 1e-5
    g = np.array([1.0, 2.0, -0.5, 3.0])
    for c in (0.3, -2.0, 1e-3):
        out = oracle.rmsnorm(np.full(4, c), g, eps)
        expect = math.copysign(1.0, c) * g / math.sqrt(1 + eps / (c * c))
        assert np.allclose(out, expect, rtol=1e-14)


def test_rmsnorm_unit_rms():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((4, 256)) * 7
    n = oracle.rmsnorm(h, np.ones(256), 0.0)
    assert np.allclose(np.sqrt(np.mean(n * n, axis=-1)), 1.0, rtol=1e-14)


def test_rope_identity_at_zero_and_rotation_sign():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 64))
    assert np.array_equal(oracle.rope(x, 0, 1e4), x)
    # head_dim 2: the pair (x0, x1) rotates counter-clockwise by pos * theta^0
    for p in (1, 5, 1000):
        out = oracle.rope(np.array([1.0, 0.0]), p, 1e4)
        assert np.allclose(out, [math.cos(p), math.sin(p)], atol=1e-12)
        out = oracle.rope(np.array([0.0, 1.0]), p, 1e4)
        assert np.allclose(out, [-math.sin(p), math.cos(p)], atol=1e-12)


def test_rope_pairs_and_frequencies():
    # head_dim 8: element i pairs with i + 4 and turns by pos * 10000^(-2i/8)
    hd, pos = 8, 3
    for i in range(4):
        x = np.zeros(hd)
        x[i] = 1.0
        out = oracle.rope(x, pos, 1e4)
        ang = pos * 1e4 ** (-2 * i / hd)
        expect = np.zeros(hd)
        expect[i], expect[i + 4] = math.cos(ang), math.sin(ang)
        assert np.allclose(out, expect, atol=1e-13)


def test_rope_relative_position_invariance():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    a = oracle.rope(q, 17, 1e4) @ oracle.rope(k, 5, 1e4)
    b = oracle.rope(q, 17 + 300, 1e4) @ oracle.rope(k, 5 + 300, 1e4)
    assert abs(a - b) < 1e-9 * (1 + abs(a))
    assert np.isclose(np.linalg.norm(oracle.rope(q, 999, 1e4)), np.linalg.norm(q), rtol=1e-13)


def test_attention_hand_worked_example():
    g = read_golden("attention_example.txt")
    q = np.array(g["q"])[None, :]
    K = np.array([g["k0"], g["k1"]])[:, None, :]
    V = np.array([g["v0"], g["v1"]])[:, None, :]
    o = oracle.attention_decode(q, K, V)
    assert np.allclose(o[0], g["o"], rtol=1e-14, atol=1e-14)


def test_attention_single_token_returns_value_of_group():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((1, 2, 16))
    V = rng.standard_normal((1, 2, 16))
    o = oracle.attention_decode(q, K, V)
    # Hq=4, Hkv=2: heads 0,1 read kv head 0; heads 2,3 read kv head 1
    assert np.allclose(o, V[0][[0, 0, 1, 1]], rtol=1e-15)


def test_attention_against_torch_sdpa_and_mha_reduction():
    rng = np.random.default_rng(9)
    hq, hkv, hd, ctx = 8, 2, 32, 37
    q = rng.standard_normal((hq, hd))
    K = rng.standard_normal((ctx, hkv, hd))
    V = rng.standard_normal((ctx, hkv, hd))
    o = oracle.attention_decode(q, K, V)
    kk = torch.from_numpy(np.repeat(K, hq // hkv, axis=1)).permute(1, 0, 2)
    vv = torch.from_numpy(np.repeat(V, hq // hkv, axis=1)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], kk, vv)[:, 0, :].numpy()
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
    # Hkv = Hq is plain multi-head attention: head h reads kv head h
    K2 = rng.standard_normal((ctx, hq, hd))
    V2 = rng.standard_normal((ctx, hq, hd))
    o2 = oracle.attention_decode(q, K2, V2)
    for h in range(hq):
        s = K2[:, h] @ q[h] / math.sqrt(hd)
        p = np.exp(s - s.max())
        assert np.allclose(o2[h], (p / p.sum()) @ V2[:, h], rtol=1e-12)


def test_swiglu_values():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert math.isclose(oracle.silu(np.array([1.0]))[0], 0.7310585786300049, rel_tol=1e-15)
    g = np.array([1.0, -2.0, 30.0])
    u = np.array([2.0, 3.0, 0.5])
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    assert np.allclose(oracle.swiglu(g, u), ref, rtol=1e-14)


# --------------------------------------------------------------- exit head

def test_lowrank_head_parameter_count():
    g = read_golden("lowrank_head_params.txt")
    V, d = g["vocab"][0], g["d_model"][0]
    # the exit transform is d x d (u = n T); the full head would be V x d
    T = synth.exit_transform(synth.Shape("t", 1, 8, 1, 1, 8, 8, 8), 1, 0)
    assert T.shape == (8, 8)
    assert d * d == g["transform_params"][0]
    assert V * d == g["full_head_params"][0]
    assert (V * d) // (d * d) == g["ratio_floor"][0]


def test_confidence_all_equal_logits_is_one_over_vocab():
    for V in (7, 2048):
        assert oracle.max_softmax(np.full(V, 3.25)) == pytest.approx(1.0 / V, rel=1e-15)


def test_confidence_matches_logsumexp_and_bounds():
    rng = np.random.default_rng(10)
    for scale in (0.01, 1.0, 30.0):
        z = rng.standard_normal(5000) * scale
        c = oracle.max_softmax(z)
        ref = math.exp(z.max() - scipy.special.logsumexp(z))
        assert c == pytest.approx(ref, rel=1e-12)
        assert 1.0 / z.size < c <= 1.0


def test_exit_head_brute_force_and_transform_orientation():
    rng = np.random.default_rng(11)
    d, V = 16, 50
    h = rng.standard_normal(d)
    g = rng.standard_normal(d)
    E = rng.standard_normal((V, d))
    T = rng.standard_normal((d, d))
    z = oracle.head_logits(h, g, E, 1e-5, T)
    n = h / math.sqrt(sum(x * x for x in h) / d + 1e-5) * g
    for v in range(V):
        u = [sum(n[r] * T[r, c] for r in range(d)) for c in range(d)]   # u = n T
        assert z[v] == pytest.approx(sum(u[c] * E[v, c] for c in range(d)), rel=1e-10, abs=1e-10)
    # T = I is the model's own LM head (logit lens)
    assert np.allclose(oracle.head_logits(h, g, E, 1e-5, np.eye(d)),
                       oracle.head_logits(h, g, E, 1e-5), rtol=1e-14)


def test_argmax_ties_lowest_index_and_margin():
    z = np.array([1.0, 3.0, 0.5, 3.0])
    assert oracle.argmax_lowest(z) == 1
    assert oracle.top2_margin(z) == 0.0
    assert oracle.top2_margin(np.array([1.0, 4.0, 2.5])) == 1.5


def test_percentile_reading():
    g = read_golden("percentile_example.txt")
    s = np.array(g["samples"])
    assert np.percentile(s, 40) == pytest.approx(g["p40"][0], rel=1e-15)
    assert np.percentile(s, 70) == pytest.approx(g["p70"][0], rel=1e-15)


class _ScriptedOracle:
    """Stands in for the oracle inside calibrate_gammas: it replays fixed
    confidences and checks how it is driven (thresholds, token flow, calls)."""

    def __init__(self, conf_steps, checkpoints):
        self.cfg = type("Cfg", (), {"checkpoints": tuple(checkpoints)})()
        self.conf_steps = conf_steps
        self.gamma = None
        self.calls = []
        self.expect_tok = None

    def set_thresholds(self, g):
        self.gamma = np.asarray(g, dtype=np.float64)

    def prefill(self, prompts):
        self.calls.append("prefill")
        self.expect_tok = np.arange(len(prompts), dtype=np.int32) + 7
        return self.expect_tok.copy()

    def decode_step(self, tok, forced_exit=None, eval_heads=True):
        assert self.calls and self.calls[0] == "prefill"
        assert np.all(np.isposinf(self.gamma)), "calibration must run with exits disabled"
        assert forced_exit is None and eval_heads
        assert np.array_equal(np.asarray(tok), self.expect_tok), "tokens must flow step to step"
        k = sum(c == "step" for c in self.calls)
        self.calls.append("step")
        B = len(tok)
        self.expect_tok = self.expect_tok + 100
        return oracle.StepResult(self.expect_tok.copy(), np.zeros(B, np.int32),
                                 np.asarray(self.conf_steps[k], dtype=np.float64).reshape(B, -1),
                                 np.zeros((1, B, 1)), np.zeros((B, 2)), np.ones(B))


def test_calibrate_gammas_hand_worked():
    """oracle.calibrate_gammas against a hand-worked case: samples come from
    decode steps 1..N only, with gamma = +inf, per checkpoint, percentiles by
    linear interpolation (CALM article §2.2: one threshold per layer)."""
    g = read_golden("gamma_calibration_example.txt")
    n = int(g["steps"][0])
    conf = [g["step%d" % (k + 1)] for k in range(n + 1)]
    fake = _ScriptedOracle(conf, (4, 8))
    gam, S = oracle.calibrate_gammas(fake, [[1, 2], [3]], n, (40, 70))
    assert fake.calls == ["prefill"] + ["step"] * n
    assert S.shape == (n, 2, 2)
    assert np.allclose(gam[40], g["p40"], rtol=1e-12, atol=0)
    assert np.allclose(gam[70], g["p70"], rtol=1e-12, atol=0)


# --------------------------------------------------------------- whole model

@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["tiny-b1"]
    lens, prompts = synth.workload_inputs(w)
    return w, prompts


def test_no_exit_decode_equals_uncached_recompute(tiny):
    """gamma = +inf: KV-cached decode == full causal recompute of every token
    (page 1 §2.2 loop), which pins the cache, the RoPE positions and causality."""
    w, prompts = tiny
    o = oracle.build_oracle(w)
    o.set_thresholds([np.inf] * len(w.checkpoints))
    toks = list(prompts[0][:20])
    first = o.prefill([toks])
    seq = toks + [int(first[0])]
    for _ in range(6):
        r = o.decode_step([seq[-1]])
        hs, logits = oracle.forward_full(o.cfg, o.W, seq)
        assert np.allclose(r.hidden[:, 0], hs[:, -1], rtol=1e-10, atol=1e-12)
        assert int(r.next_tokens[0]) == oracle.argmax_lowest(logits)
        assert np.all(r.exit_layers == w.shape.n_layers - 1)
        seq.append(int(r.next_tokens[0]))


def test_exit_at_layer0_equals_all_int4_model(tiny):
    """gamma = -inf with a single checkpoint at layer 0: every decoded token ran
    layer 0 in bf16 and layers 1..L-1 on the int4 copies; equal to a plain model
    built that way (uncached, per-position weight choice)."""
    w, prompts = tiny
    o = oracle.build_oracle(w)
    o.cfg.checkpoints = (0,)
    o.W.T = [o.W.T[0]]
    o.gamma = np.array([-np.inf])
    toks = list(prompts[0][:12])
    first = o.prefill([toks])
    seq = toks + [int(first[0])]
    for _ in range(5):
        r = o.decode_step([seq[-1]])
        assert r.exit_layers[0] == 0
        int4_after = [None] * len(toks) + [0] * (len(seq) - len(toks))
        hs, logits = oracle.forward_full(o.cfg, o.W, seq, int4_after=int4_after)
        assert np.allclose(r.hidden[:, 0], hs[:, -1], rtol=1e-10, atol=1e-12)
        assert int(r.next_tokens[0]) == oracle.argmax_lowest(logits)
        seq.append(int(r.next_tokens[0]))
    # and the int4 layers really differ from the bf16 ones
    hs_bf16, _ = oracle.forward_full(o.cfg, o.W, seq)
    assert not np.allclose(hs_bf16[-1, -1], hs[-1, -1], rtol=1e-6)


def test_kv_coverage_and_block_bookkeeping(tiny):
    """Every (layer, position) slot of every sequence is written whatever the
    exit pattern; blocks are handed out in ascending order."""
    w, _ = tiny
    o = oracle.build_oracle(w, max_batch=3, max_seq_len=64)
    pr = synth.prompts(w.shape, 99, [15, 16, 17])
    first = o.prefill(pr)
    assert [s.blocks for s in o.seqs] == [[0], [1], [2, 3]]
    rng = np.random.default_rng(12)
    tok = first
    for step in range(20):
        forced = [int(rng.choice([-1] + list(w.checkpoints))) for _ in range(3)]
        r = o.decode_step(tok, forced_exit=forced)
        for s in range(3):
            expect = forced[s] if forced[s] >= 0 else w.shape.n_layers - 1
            assert r.exit_layers[s] == expect
            P = o.seqs[s].pos
            assert not np.isnan(o.K[s][:, :P]).any() and not np.isnan(o.V[s][:, :P]).any()
            assert np.isnan(o.K[s][:, P:]).all()
        tok = r.next_tokens
    # sequence 1 starts at position 16 -> needs a block at its first decode step;
    # then every 16 positions; allocation order follows sequence order per step
    ids = sorted(b for s in o.seqs for b in s.blocks)
    assert ids == list(range(len(ids)))
    assert o.slot(2, 17) == (o.seqs[2].blocks[1], 1)


def test_batch_independence(tiny):
    w, _ = tiny
    pr = synth.prompts(w.shape, 7, [9, 14, 11])
    ob = oracle.build_oracle(w, max_batch=3, max_seq_len=40)
    g = np.array([0.0025, 0.0021])
    ob.set_thresholds(g)
    tb = ob.prefill(pr)
    outs_b = []
    for _ in range(5):
        r = ob.decode_step(tb)
        outs_b.append((r.next_tokens.copy(), r.exit_layers.copy()))
        tb = r.next_tokens
    for s in range(3):
        o1 = oracle.build_oracle(w, max_batch=1, max_seq_len=40)
        o1.set_thresholds(g)
        t1 = o1.prefill([pr[s]])
        for k in range(5):
            r = o1.decode_step(t1)
            assert r.next_tokens[0] == outs_b[k][0][s] and r.exit_layers[0] == outs_b[k][1][s]
            t1 = r.next_tokens


def test_exit_decision_is_strict_and_first_checkpoint_wins(tiny):
    w, prompts = tiny
    o = oracle.build_oracle(w)
    o.set_thresholds([np.inf, np.inf])
    t = o.prefill([prompts[0]])
    snap = o.snapshot()
    r0 = o.decode_step(t)
    c1, c2 = r0.conf[0]
    # gamma equal to the confidence: strict '>' means no exit there
    o.restore(snap)
    o.set_thresholds([c1, -np.inf])
    r = o.decode_step(t)
    assert r.exit_layers[0] == w.checkpoints[1]
    o.restore(snap)
    o.set_thresholds([np.nextafter(c1, 0), -np.inf])
    r = o.decode_step(t)
    assert r.exit_layers[0] == w.checkpoints[0]
    assert np.isnan(r.conf[0, 1])      # no head after the exit
    o.restore(snap)
    r = o.decode_step(t, eval_heads=False)
    assert np.isnan(r.conf).all() and r.exit_layers[0] == w.shape.n_layers - 1


def test_tiny_trace_reproduces(tiny):
    """The stored tiny trace (tests/golden/make_tiny_trace.py) still matches the
    oracle: guards against silent drift of the oracle or the generator."""
    import json
    from tests.conftest import golden_path
    ref = json.load(open(golden_path("tiny_oracle_trace.json")))
    w, prompts = tiny
    o = oracle.build_oracle(w)
    o.set_thresholds(ref["gamma"])
    tok = o.prefill(prompts)
    assert tok.tolist() == ref["trace"]["first_tokens"]
    for k in range(w.steps):
        r = o.decode_step(tok)
        assert r.next_tokens.tolist() == ref["trace"]["tokens"][k]
        assert r.exit_layers.tolist() == ref["trace"]["exit_layers"][k]
        tok = r.next_tokens


# ---------------------------------------------------- state transition similarity

def test_sts_hand_worked_examples():
    """River-LLM §5.1: cosine of the unit-normalised input and output states."""
    g = read_golden("sts_example.txt")
    for k in "abcde":
        got = oracle.state_transition_similarity(np.array(g[k + "_in"], float), np.array(g[k + "_out"], float))
        assert got == pytest.approx(g[k + "_sts"][0], abs=1e-15), k
    rng = np.random.default_rng(3)
    x = rng.standard_normal(64)
    assert oracle.state_transition_similarity(x, 3.5 * x) == pytest.approx(1.0, abs=1e-14)   # scale invariant
    y = rng.standard_normal(64)
    assert oracle.state_transition_similarity(x, y) == pytest.approx(
        oracle.state_transition_similarity(y, x), abs=1e-15)                                 # symmetric
    assert -1.0 - 1e-12 <= oracle.state_transition_similarity(x, y) <= 1.0 + 1e-12


def _tiny_sts_oracle(gamma=None, T_nan=False):
    w = synth.WORKLOADS["tiny-b1"]
    o = oracle.build_oracle(w, criterion="sts")
    if T_nan:
        o.W.T = [np.full_like(t, np.nan) for t in o.W.T]
    o.set_thresholds(np.full(len(w.checkpoints), np.inf) if gamma is None else gamma)
    lens, prompts = synth.workload_inputs(w)
    return w, o, [list(prompts[0][:20])]


def test_sts_scores_the_checkpoint_layers_input_and_output():
    """At checkpoint j the score compares the state entering layer j (the
    output of layer j-1) with the state leaving it, read back from the
    per-layer residual streams the step returns."""
    w, o, pr = _tiny_sts_oracle()
    tok = o.prefill(pr)
    r = o.decode_step(tok)
    for c, j in enumerate(w.checkpoints):
        assert j >= 1
        want = oracle.state_transition_similarity(r.hidden[j - 1, 0], r.hidden[j, 0])
        assert r.conf[0, c] == pytest.approx(want, abs=1e-15)
        # a different pair of states (one layer later) gives a different score
        other = oracle.state_transition_similarity(r.hidden[j, 0], r.hidden[j + 1, 0])
        assert abs(other - r.conf[0, c]) > 1e-6


def test_sts_reads_no_vocabulary_or_exit_transform():
    """§5.3: the decision is O(d); with the exit transforms replaced by NaN
    the similarity-criterion decode is unchanged (they are never read)."""
    w, o1, pr = _tiny_sts_oracle(gamma=[0.5, 0.5])
    _, o2, _ = _tiny_sts_oracle(gamma=[0.5, 0.5], T_nan=True)
    t1, t2 = o1.prefill(pr), o2.prefill(pr)
    for _ in range(3):
        r1, r2 = o1.decode_step(t1), o2.decode_step(t2)
        assert np.array_equal(r1.next_tokens, r2.next_tokens)
        assert np.array_equal(r1.exit_layers, r2.exit_layers)
        assert np.allclose(r1.conf, r2.conf, equal_nan=True)
        t1, t2 = r1.next_tokens, r2.next_tokens


def test_sts_threshold_is_strict():
    """A token exits at the first checkpoint whose score is strictly above tau."""
    w, o, pr = _tiny_sts_oracle()
    tok = o.prefill(pr)
    snap = o.snapshot()
    r = o.decode_step(tok)
    s0 = r.conf[0, 0]
    o.restore(snap)
    o.set_thresholds([s0, -np.inf])              # equal to the score: no exit at layer 1
    r = o.decode_step(tok)
    assert r.exit_layers[0] == w.checkpoints[1]
    o.restore(snap)
    o.set_thresholds([np.nextafter(s0, -np.inf), np.inf])   # just below: exits at layer 1
    r = o.decode_step(tok)
    assert r.exit_layers[0] == w.checkpoints[0]


def test_sts_batch_rule_exits_together_on_the_minimum():
    """River-LLM §5.2: with the batch rule every sequence still on the
    full-precision path exits when the minimum of their scores clears tau,
    and none does otherwise; with one sequence it is the per-token rule."""
    w = synth.WORKLOADS["tiny-b1"]
    lens = [7, 12, 19]
    pr = synth.prompts(w.shape, 5, lens)
    per = oracle.build_oracle(w, max_batch=3, criterion="sts")
    bat = oracle.build_oracle(w, max_batch=3, criterion="sts_batch")
    for o in (per, bat):
        o.set_thresholds([np.inf, np.inf])
    tp, tb = per.prefill(pr), bat.prefill(pr)
    sp, sb = per.snapshot(), bat.snapshot()
    rp = per.decode_step(tp)
    s0 = rp.conf[:, 0]                                  # per-sequence scores at layer 1
    lo, hi = float(s0.min()), float(s0.max())
    assert hi > lo
    # tau between the minimum and the maximum: some sequences exit per token, none in the batch rule
    tau = 0.5 * (lo + hi)
    per.restore(sp)
    per.set_thresholds([tau, np.inf])
    assert 0 < int((per.decode_step(tp).exit_layers == 1).sum()) < 3
    bat.restore(sb)
    bat.set_thresholds([tau, np.inf])
    rb = bat.decode_step(tb)
    assert np.all(rb.exit_layers == w.shape.n_layers - 1)
    assert np.allclose(rb.conf[:, 0], lo, rtol=0, atol=1e-15)   # every sequence records the minimum
    # tau just below the minimum: the whole batch exits at layer 1
    bat.restore(sb)
    bat.set_thresholds([np.nextafter(lo, -np.inf), np.inf])
    assert np.all(bat.decode_step(tb).exit_layers == 1)
    # batch of one: identical to the per-token rule
    one_p = oracle.build_oracle(w, max_batch=1, criterion="sts")
    one_b = oracle.build_oracle(w, max_batch=1, criterion="sts_batch")
    for o in (one_p, one_b):
        o.set_thresholds([tau, tau])
        t = o.prefill(pr[:1])
        o._r = o.decode_step(t)
    assert np.array_equal(one_p._r.exit_layers, one_b._r.exit_layers)
    assert np.allclose(one_p._r.conf, one_b._r.conf, equal_nan=True)


# ---------------------------------------------------- exit-head token

def test_exit_head_token_is_the_exit_heads_argmax():
    """With the exit-head token source an exited sequence emits the argmax of
    the head that let it leave (CALM article §3.1); a sequence that never
    exits emits the final head's argmax, as with the default source."""
    w = synth.WORKLOADS["tiny-b1"]
    lens, prompts = synth.workload_inputs(w)
    pr = [list(prompts[0][:20])]
    fin = oracle.build_oracle(w)
    ex = oracle.build_oracle(w, token_source="exit_head")
    for o in (fin, ex):
        o.set_thresholds([-np.inf, np.inf])          # exit at the first checkpoint (layer 1)
    tf, te = fin.prefill(pr), ex.prefill(pr)
    assert np.array_equal(tf, te)
    rf, re_ = fin.decode_step(tf), ex.decode_step(te)
    assert re_.exit_layers[0] == 1 and rf.exit_layers[0] == 1
    # the exit head of checkpoint 0 on the state after layer 1
    z = oracle.head_logits(re_.hidden[1, 0], ex.W.g_final, ex.W.E, w.shape.rms_eps, ex.W.T[0])
    assert re_.next_tokens[0] == oracle.argmax_lowest(z)
    assert re_.margins[0] == pytest.approx(oracle.top2_margin(z))
    # the state after the last layer is the same either way (the int4 layers still run)
    assert np.allclose(re_.hidden, rf.hidden, rtol=0, atol=0)
    # no exit: both sources agree exactly
    for o in (fin, ex):
        o.set_thresholds([np.inf, np.inf])
    a, b = fin.decode_step(rf.next_tokens), ex.decode_step(rf.next_tokens)
    assert np.array_equal(a.next_tokens, b.next_tokens)


def test_exit_head_token_needs_the_exit_head():
    w = synth.WORKLOADS["tiny-b1"]
    with pytest.raises(AssertionError):
        oracle.build_oracle(w, criterion="sts", token_source="exit_head")


# ---------------------------------------------------- sequence-level exit in prefill

def test_prefill_sequence_exit_limits_and_minimum_rule():
    """River-LLM §6.1: in prefill all tokens of a prompt exit at one layer.
    tau = +inf is the plain prefill; tau = -inf exits every prompt at the
    first checkpoint, which equals the plain causal forward with every
    position on the int4 copies after it (checked through forward_full,
    the uncached route); the decision uses the minimum over the tokens."""
    w = synth.WORKLOADS["tiny-b1"]
    pr = synth.prompts(w.shape, 8, [9, 14])
    ck = w.checkpoints
    plain = oracle.build_oracle(w, max_batch=2)
    t0 = plain.prefill(pr)
    o = oracle.build_oracle(w, max_batch=2)
    assert np.array_equal(o.prefill(pr, exit_tau=[np.inf] * len(ck)), t0)
    assert np.all(o.prefill_exits == w.shape.n_layers - 1)
    for s in range(2):
        assert np.allclose(o.K[s][:, :len(pr[s])], plain.K[s][:, :len(pr[s])], rtol=0, atol=0)
    scores = o.prefill_scores.copy()
    # every prompt exits at the first checkpoint
    first = o.prefill(pr, exit_tau=[-np.inf] * len(ck))
    assert np.all(o.prefill_exits == ck[0])
    for s in range(2):
        hs, logits, Ks, Vs = oracle.forward_full(o.cfg, o.W, pr[s], int4_after=[ck[0]] * len(pr[s]),
                                                 return_kv=True)
        assert first[s] == oracle.argmax_lowest(logits)
        assert np.allclose(o.K[s][:, :len(pr[s])], Ks, rtol=1e-12, atol=1e-14)
        assert np.allclose(o.V[s][:, :len(pr[s])], Vs, rtol=1e-12, atol=1e-14)
    # the minimum over the tokens decides: tau between the two prompts' minima
    a, b = scores[0, 0], scores[1, 0]
    tau = 0.5 * (a + b)
    o.prefill(pr, exit_tau=[tau, np.inf])
    want = [ck[0] if sc > tau else w.shape.n_layers - 1 for sc in (a, b)]
    assert o.prefill_exits.tolist() == want and len(set(want)) == 2
    # the minimum itself: a prompt whose minimum equals tau does not exit (strict)
    o.prefill(pr, exit_tau=[a, np.inf])
    assert o.prefill_exits[0] == w.shape.n_layers - 1
