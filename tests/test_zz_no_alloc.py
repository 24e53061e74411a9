"""ee_op_attention_noalloc (attention with the library's fixed scratch array,
for callers that cannot allocate device memory) against ee_op_attention with a
caller buffer and against the CPU oracle's attention, on the same seeded
inputs; and a check that a call allocates no device memory.  Collected last so
that it also runs after every other test in the same process; it passes alone
as well."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import early_exit_decoding_layer_gb300 as ee  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    ee.load_library()


def paged_inputs(seed, B, ctxs, hq, hkv, hd):
    """fp16 K/V histories scattered over shuffled 16-slot blocks, fp32 queries."""
    rng = np.random.default_rng(seed)
    bps = max((c + 15) // 16 for c in ctxs)
    nblocks = B * bps + 3
    order = rng.permutation(nblocks).astype(np.int32)
    bt = order[:B * bps].reshape(B, bps).copy()
    kc = rng.standard_normal((nblocks, hkv, 16, hd)).astype(np.float16)
    vc = rng.standard_normal((nblocks, hkv, 16, hd)).astype(np.float16)
    q = rng.standard_normal((B, hq * hd)).astype(np.float32)
    pos = np.array(ctxs, dtype=np.int32) - 1
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    return d(q), d(kc.view(np.int16)), d(vc.view(np.int16)), d(bt), d(pos)


# (B, Hq, Hkv, hd, ctxs, max_ctx): the Llama-3.1-8B head layout at a long
# context, a ragged small batch, and a shape whose merge counters land where
# the previous case's partial results were.
CASES = [
    (1, 32, 8, 128, [2047], 2300),
    (3, 8, 2, 64, [1, 33, 300], 320),
    (2, 16, 16, 128, [17, 900], 1000),
]


def oracle_attention(q, kc, vc, bt, pos, hq, hkv, hd):
    """The oracle's decode attention per sequence over its gathered history."""
    q, kc, vc = q.cpu().numpy(), kc.cpu().numpy().view(np.float16), vc.cpu().numpy().view(np.float16)
    bt, pos = bt.cpu().numpy(), pos.cpu().numpy()
    out = np.empty((q.shape[0], hq * hd))
    for b in range(q.shape[0]):
        ctx = int(pos[b]) + 1
        slots = [(bt[b, t // 16], t % 16) for t in range(ctx)]
        K = np.stack([kc[blk, :, off, :] for blk, off in slots]).astype(np.float64)
        V = np.stack([vc[blk, :, off, :] for blk, off in slots]).astype(np.float64)
        out[b] = oracle.attention_decode(q[b].astype(np.float64).reshape(hq, hd), K, V).reshape(-1)
    return out


def test_noalloc_matches_attention_two_calls_in_a_row():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i, (B, hq, hkv, hd, ctxs, max_ctx) in enumerate(CASES):
        assert ee.attention_scratch_bytes(B, hq, hkv, hd, max_ctx) <= ee.ATTN_STATIC_SCRATCH_BYTES
        q, kc, vc, bt, pos = paged_inputs(100 + i, B, ctxs, hq, hkv, hd)
        ref = ee.attention(q, kc, vc, bt, pos, hq, hkv, hd, max_ctx, err=err)
        want = oracle_attention(q, kc, vc, bt, pos, hq, hkv, hd)
        out = torch.empty_like(ref)
        for rep in range(2):
            out.fill_(float("nan"))
            ee.attention_noalloc(q, kc, vc, bt, pos, hq, hkv, hd, max_ctx, out=out, err=err)
            torch.cuda.synchronize()
            assert torch.allclose(out, ref, rtol=1e-4, atol=1e-5), (i, rep)
            # the same tolerance as the attention kernel's own oracle parity test
            assert np.allclose(out.cpu().numpy(), want, rtol=1e-4, atol=1e-5), (i, rep)
    assert err.item() == 0


def test_noalloc_call_allocates_no_device_memory():
    B, hq, hkv, hd, ctxs, max_ctx = CASES[0]
    q, kc, vc, bt, pos = paged_inputs(7, B, ctxs, hq, hkv, hd)
    out = torch.empty(B, hq * hd, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ee.attention_noalloc(q, kc, vc, bt, pos, hq, hkv, hd, max_ctx, out=out, err=err)  # warm-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(3):
        ee.attention_noalloc(q, kc, vc, bt, pos, hq, hkv, hd, max_ctx, out=out, err=err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0                      # nothing taken from the device (cudaMemGetInfo)
    for k in ("allocation.all.allocated", "reserved_bytes.all.current", "allocated_bytes.all.current"):
        assert stats1.get(k, 0) == stats0.get(k, 0), k   # nor from torch's caching allocator
    assert err.item() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # B = 16 at max_ctx 2048 with the Llama-3.1-8B heads needs more than the
    # fixed array holds: EE_ERR_CAPACITY, and nothing is launched.
    assert ee.attention_scratch_bytes(16, 32, 8, 128, 2048) > ee.ATTN_STATIC_SCRATCH_BYTES
    z = torch.zeros(16, 32 * 128, dtype=torch.float32, device="cuda")
    bt = torch.zeros(16, 128, dtype=torch.int32, device="cuda")
    pos = torch.zeros(16, dtype=torch.int32, device="cuda")
    kv = torch.zeros(8, 16, 128, dtype=torch.int16, device="cuda")
    with pytest.raises(ee.EEError) as e:
        ee.attention_noalloc(z, kv, kv, bt, pos, 32, 8, 128, 2048, out=z)
    assert e.value.status == 3  # EE_ERR_CAPACITY
    with pytest.raises(ee.EEError) as e:
        ee.attention_noalloc(z, kv, kv, bt, pos, 32, 8, 96, 2048, out=z)   # head_dim 96
    assert e.value.status == 1  # EE_ERR_INVALID_ARG
