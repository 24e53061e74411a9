"""Single-kernel parity: each CUDA kernel through the C ABI against the CPU
oracle's routine on the same seeded inputs, at small ragged sizes and at the
Llama-3.1-8B shapes."""
import math

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import early_exit_decoding_layer_gb300 as ee  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_bits(x64, rng=None):
    return oracle.f32_to_bf16_bits(np.asarray(x64, dtype=np.float32))


def half_pair_order(x16):
    """fp16 activations in the kernels' pair order: within each run of 8
    columns the order is 0,4,1,5,2,6,3,7 (written here by scattering)."""
    M, K = x16.shape
    idx = np.arange(K)
    j = idx % 8
    slot = (idx - j) + np.where(j < 4, 2 * j, 2 * (j - 4) + 1)
    out = np.empty_like(x16)
    out[:, slot] = x16
    assert np.array_equal(ee.pair_order(x16), out)   # the binding's gather agrees
    return out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    assert torch.cuda.is_available()


# ------------------------------------------------------------------ quantiser

@pytest.mark.parametrize("rows,cols", [(3, 704), (64, 256), (130, 4096), (8, 14336)])
def test_quantize_bit_exact(rows, cols):
    w = synth.normal_bf16(77, rows * 131 + cols, (rows, cols), 0.02)
    w[0, :128] = 0  # an all-zero group
    q_ref, s_ref = oracle.quantize_int4_group(w, 128)
    packed, scales = ee.quantize_int4(dev(w.view(np.int16)))
    torch.cuda.synchronize()
    ng = (cols + 127) // 128
    assert np.array_equal(packed.cpu().numpy(), oracle.pack_int4(q_ref))
    assert np.array_equal(scales.cpu().numpy().view(np.uint16)[:, :ng], s_ref)


# ------------------------------------------------------------------ GEMV

@pytest.mark.parametrize("M,N,K", [(1, 34, 256), (3, 256, 704), (8, 6144, 4096), (11, 96, 2048),
                                   (1, 4096, 14336), (2, 28672, 4096)])
def test_linear_bf16(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K)
    W = synth.normal_bf16(5, N * 7 + K, (N, K), 0.02)
    x16 = rng.standard_normal((M, K)).astype(np.float16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = ee.linear_bf16(dev(half_pair_order(x16).view(np.int16)), dev(W.view(np.int16)), err=err).cpu().numpy()
    xf, Wf = x16.astype(np.float64), oracle.bf16_to_f64(W)
    ref = oracle.linear(xf, Wf)
    bound = 1e-5 * (np.abs(xf) @ np.abs(Wf).T) + 1e-7   # fp32 accumulation of exact products
    assert np.all(np.abs(y - ref) <= bound)
    assert err.item() == 0


@pytest.mark.parametrize("M,N,K", [(1, 34, 256), (3, 256, 704), (8, 6144, 4096), (9, 64, 2048),
                                   (1, 4096, 14336), (1, 28672, 4096)])
def test_linear_int4(M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K + 1)
    W = synth.normal_bf16(6, N * 7 + K, (N, K), 0.02)
    q, s = oracle.quantize_int4_group(W, 128)
    packed = oracle.pack_int4(q)
    ss = (K + 127) // 128 + (3 if M == 9 else 0)   # padded rows take the scale-gather path
    spad = np.zeros((N, ss), dtype=np.uint16)
    spad[:, : s.shape[1]] = s
    x16 = rng.standard_normal((M, K)).astype(np.float16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = ee.linear_int4(dev(half_pair_order(x16).view(np.int16)), dev(packed),
                       dev(spad.view(np.int16)), err=err).cpu().numpy()
    Wd = oracle.dequant_int4(q, s, 128)
    xf = x16.astype(np.float64)
    ref = oracle.linear(xf, Wd)
    # products accumulate in fp16 over 16 terms per half lane before fp32:
    # each partial carries at most ~16 roundings of 2^-11 relative
    bound = 4e-3 * (np.abs(xf) @ np.abs(Wd).T) + 1e-6
    assert np.all(np.abs(y - ref) <= bound)
    assert err.item() == 0
    # and the typical error is far below the bound
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) < 2e-3


# ------------------------------------------------------------------ attention

def paged(rng, B, ctxs, hkv, hd, nblocks_extra=5):
    """Random fp16 K/V histories scattered over shuffled 16-slot blocks."""
    bps = max((c + 15) // 16 for c in ctxs)
    nblocks = B * bps + nblocks_extra
    order = rng.permutation(nblocks)
    bt = np.zeros((B, bps), dtype=np.int32)
    kc = np.full((nblocks, hkv, 16, hd), 0xFFFF, dtype=np.uint16)
    vc = kc.copy()
    K, V = [], []
    n = 0
    for b in range(B):
        Kb = rng.standard_normal((ctxs[b], hkv, hd)).astype(np.float16).view(np.uint16)
        Vb = rng.standard_normal((ctxs[b], hkv, hd)).astype(np.float16).view(np.uint16)
        for i in range((ctxs[b] + 15) // 16):
            bt[b, i] = order[n]
            n += 1
        for t in range(ctxs[b]):
            kc[bt[b, t // 16], :, t % 16] = Kb[t]
            vc[bt[b, t // 16], :, t % 16] = Vb[t]
        K.append(Kb)
        V.append(Vb)
    return kc, vc, bt, K, V


@pytest.mark.parametrize("B,hq,hkv,hd,ctxs", [
    (1, 4, 2, 64, [1]), (1, 4, 2, 64, [15]), (1, 4, 2, 64, [16]), (1, 4, 2, 64, [17]),
    (3, 32, 8, 64, [300, 1, 47]), (1, 32, 8, 128, [2304]), (2, 64, 8, 128, [4100, 33]),
    (4, 8, 8, 128, [5, 64, 129, 1000]), (2, 16, 16, 64, [700, 16]), (1, 64, 8, 128, [1]),
    # grids of several waves of CTAs, ragged contexts
    (8, 32, 8, 128, [3000, 17, 1500, 800, 2047, 64, 1201, 2500]),
    (6, 32, 8, 64, [2000, 900, 31, 1777, 1200, 640]),
])
def test_attention(B, hq, hkv, hd, ctxs):
    rng = np.random.default_rng(B * 7 + hq + hd + sum(ctxs))
    kc, vc, bt, K, V = paged(rng, B, ctxs, hkv, hd)
    q = rng.standard_normal((B, hq * hd)).astype(np.float32)
    pos = np.array(ctxs, dtype=np.int32) - 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_ctx = max(ctxs) + 37
    scratch = torch.zeros(ee.attention_scratch_bytes(B, hq, hkv, hd, max_ctx), dtype=torch.uint8, device="cuda")
    for rep in range(2):  # the second call checks that the counters were left at zero
        o = ee.attention(dev(q), dev(kc.view(np.int16)), dev(vc.view(np.int16)), dev(bt), dev(pos),
                         hq, hkv, hd, max_ctx, scratch=scratch, err=err).cpu().numpy()
        for b in range(B):
            ref = oracle.attention_decode(q[b].astype(np.float64).reshape(hq, hd),
                                          K[b].view(np.float16).astype(np.float64),
                                          V[b].view(np.float16).astype(np.float64))
            assert np.allclose(o[b].reshape(hq, hd), ref, rtol=1e-4, atol=1e-5), (rep, b)
    assert err.item() == 0


# ------------------------------------------------------------------ vocabulary head

@pytest.mark.parametrize("M,V,d", [(1, 2048, 256), (3, 1002, 704), (1, 128256, 4096), (5, 32016, 256)])
def test_vocab_head(M, V, d):
    rng = np.random.default_rng(M + V + d)
    E = synth.normal_bf16(9, V + d, (V, d), 0.02)
    u16 = rng.standard_normal((M, d)).astype(np.float16)
    conf, arg = ee.vocab_head(dev(half_pair_order(u16).view(np.int16)), dev(E.view(np.int16)))
    conf, arg = conf.cpu().numpy(), arg.cpu().numpy()
    z = oracle.linear(u16.astype(np.float64), oracle.bf16_to_f64(E))
    for m in range(M):
        c_ref = oracle.max_softmax(z[m])
        assert abs(conf[m] - c_ref) <= 1e-4 * c_ref
        a = oracle.argmax_lowest(z[m])
        if arg[m] != a:   # only a near-tie may differ
            assert z[m, a] - z[m, arg[m]] < 1e-5 * np.abs(z[m]).max()
    # a planted winner is found, ties go to the lowest index
    E2 = np.zeros((64, 32), dtype=np.uint16)
    E2[[5, 9, 40], 0] = 0x3F80  # 1.0
    u2 = np.zeros((1, 32), dtype=np.uint16)
    u2[0, 0] = 0x4000  # fp16 2.0 (column 0 stays first in pair order)
    conf, arg = ee.vocab_head(dev(u2.view(np.int16)), dev(E2.view(np.int16)))
    assert arg.item() == 5
    expect = 1.0 / (3 + 61 * math.exp(-2.0))
    assert abs(conf.item() - expect) < 1e-6
