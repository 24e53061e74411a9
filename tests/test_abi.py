"""The C ABI library: it loads, exports every symbol include/ee.h declares,
and validates configurations on the host before any CUDA call.  CPU only
(no compute call is made)."""
import ctypes
import os
import re

import pytest

import early_exit_decoding_layer_gb300 as ee
import synth
from tests.conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from early_exit_decoding_layer_gb300 import build
    build.build()
    return ee.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "ee.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ee_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(ee.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_arena_bytes_and_host_validation(lib):
    sh = synth.SHAPES["tiny"]
    cfg = ee.make_config(sh, (1, 2), 1, 64)
    n = lib.ee_arena_bytes(ctypes.byref(cfg))
    assert n > 0
    # the arena grows with the KV capacity
    assert lib.ee_arena_bytes(ctypes.byref(ee.make_config(sh, (1, 2), 4, 64))) > n
    bad = [
        ee.make_config(sh, (2, 1), 1, 64),             # checkpoints not ascending
        ee.make_config(sh, (3,), 1, 64),               # checkpoint at the last layer
        ee.make_config(sh, (1,), 0, 64),               # empty batch
        ee.make_config(sh, (1,), ee.EE_MAX_BATCH + 1, 64),
        ee.make_config(synth.Shape("x", 2, 100, 4, 2, 64, 704, 2048), (0,), 1, 64),  # d % 32
        ee.make_config(synth.Shape("x", 2, 256, 4, 3, 64, 704, 2048), (0,), 1, 64),  # Hq % Hkv
        ee.make_config(synth.Shape("x", 2, 256, 4, 2, 96, 704, 2048), (0,), 1, 64),  # head_dim
        ee.make_config(synth.Shape("x", 2, 256, 4, 2, 64, 704, 2049), (0,), 1, 64),  # odd vocab
    ]
    for b in bad:
        assert lib.ee_arena_bytes(ctypes.byref(b)) == 0
        ctx = ctypes.c_void_p()
        assert lib.ee_create(ctypes.byref(b), 256, 1 << 30, None, ctypes.byref(ctx)) == 1
        assert not ctx.value
    # a valid config with a too-small arena is refused before any device work
    ctx = ctypes.c_void_p()
    assert lib.ee_create(ctypes.byref(cfg), 256, n - 1, None, ctypes.byref(ctx)) == 4
    # an unaligned arena is refused
    assert lib.ee_create(ctypes.byref(cfg), 257, n, None, ctypes.byref(ctx)) == 1


def test_op_argument_validation(lib):
    # shape errors are reported before any launch
    assert lib.ee_op_linear_bf16(0, 8, 64, 16, 16, 16, None, None) == 1
    assert lib.ee_op_linear_bf16(1, 7, 64, 16, 16, 16, None, None) == 1
    assert lib.ee_op_linear_bf16(1, 8, 40, 16, 16, 16, None, None) == 1
    assert lib.ee_op_linear_int4(1, 8, 256, 16, 16, 16, 1, 16, None, None) == 1
    assert lib.ee_op_attention(1, 4, 3, 64, 100, 16, 16, 16, 16, 1, 16, 16, 16, None, None) == 1
    assert lib.ee_op_attention(1, 4, 2, 64, 1 << 20, 16, 16, 16, 16, 1, 16, 16, 16, None, None) == 1
    assert lib.ee_op_vocab_head(1, 7, 64, 16, 16, 16, 16, 16, None, None) == 1
    assert lib.ee_op_quantize_int4(16, 4, 40, 16, 16, 2, None) == 1
    assert lib.ee_attention_scratch_bytes(0, 4, 2, 64, 100) == 0
    assert lib.ee_attention_scratch_bytes(1, 4, 2, 64, 100) > 0
    assert lib.ee_head_scratch_bytes(1) > 0
    # the fixed-scratch attention checks its arguments before it touches the
    # device: bad shapes and NULL pointers are refused with no CUDA call
    assert lib.ee_op_attention_noalloc(1, 4, 3, 64, 100, 16, 16, 16, 16, 1, 16, 16, None, None) == 1
    assert lib.ee_op_attention_noalloc(1, 4, 2, 96, 100, 16, 16, 16, 16, 1, 16, 16, None, None) == 1
    assert lib.ee_op_attention_noalloc(1, 4, 2, 64, 100, None, 16, 16, 16, 1, 16, 16, None, None) == 1
    assert lib.ee_op_attention_noalloc(1, 4, 2, 64, 100, 16, 16, 16, 16, 0, 16, 16, None, None) == 1


def test_static_scratch_size_matches_header():
    src = open(os.path.join(ROOT, "include", "ee.h")).read()
    m = re.search(r"#define\s+EE_ATTN_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "EE_ATTN_STATIC_SCRATCH_BYTES not found in ee.h"
    assert ee.ATTN_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
