"""Seeded synthetic inputs shared by the CPU oracle and the CUDA library.

This module draws the random-init weights, exit-head transforms and prompts
of the early-exit decode workloads.  It holds none of the decode method's
arithmetic (no norm, projection, attention, quantiser or exit rule): it only
produces the inputs both sides consume, so that the oracle and the CUDA path
see bit-identical data.

The generator is defined in ``synth.c`` (SplitMix64 counter streams and
Box-Muller normals with platform-independent series for ln/sin/cos); this
file compiles it on first use with the host C compiler and wraps it with
ctypes.  Weights are returned as bf16 bit patterns in ``numpy.uint16``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import (  # noqa: F401  (re-exported)
    Shape,
    Workload,
    SHAPES,
    WORKLOADS,
    checkpoints_every,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib = None

BF16_ONE = 0x3F80

# tensor ids inside one weight seed
MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
_MAT_ID = {m: i + 1 for i, m in enumerate(MATS)}
TID_EMBED = 1 << 20
TID_T_BASE = (1 << 20) + 1
TID_PROMPT_BASE = 1 << 24
TID_PROMPT_LENS = (1 << 24) - 1
PROMPT_SEED_XOR = 0x5EED5EED5EED5EED


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so (host C, no GPU needed)."""
    with _lock:
        if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
            cc = os.environ.get("CC", "cc")
            tmp = _SO + ".%d.tmp" % os.getpid()
            subprocess.check_call([
                cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                "-pthread", "-o", tmp, _SRC, "-lm",
            ])
            os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, dbl, i64, dbl, vp, ctypes.c_int]
        lib.synth_normal_bf16.restype = None
        lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, dbl, dbl, vp, ctypes.c_int]
        lib.synth_normal_f32.restype = None
        lib.synth_uniform_int.argtypes = [u64, u64, u64, i64, i64, vp]
        lib.synth_uniform_int.restype = None
        lib.synth_raw_u64.argtypes = [u64, u64, u64, vp]
        lib.synth_raw_u64.restype = None
        lib.synth_mix64.argtypes = [u64]
        lib.synth_mix64.restype = u64
        lib.synth_series_log.argtypes = [dbl]
        lib.synth_series_log.restype = dbl
        lib.synth_series_sincos.argtypes = [dbl, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]
        lib.synth_series_sincos.restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, tid: int, shape, std: float, base: float = 0.0,
                diag_add: float = 0.0, offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bit patterns of base + std*N(0,1) (+ diag_add on the diagonal of a 2-D shape)."""
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags.c_contiguous and out.size == n
    ncols = shape[-1] if (diag_add != 0.0 and len(shape) == 2) else 0
    _load().synth_normal_bf16(seed, tid, offset, n, base, std, ncols, diag_add,
                              out.ctypes.data, _threads())
    return out


def normal_f32(seed: int, tid: int, shape, std: float, base: float = 0.0) -> np.ndarray:
    shape = tuple(int(s) for s in np.atleast_1d(shape))
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, 0, out.size, base, std, out.ctypes.data, _threads())
    return out


def uniform_int(seed: int, tid: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int32)
    _load().synth_uniform_int(seed, tid, int(n), int(lo), int(hi), out.ctypes.data)
    return out


def raw_u64(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(int(n), dtype=np.uint64)
    _load().synth_raw_u64(seed, tid, int(n), out.ctypes.data)
    return out


def mix64(z: int) -> int:
    return int(_load().synth_mix64(z))


def series_log(x: float) -> float:
    return float(_load().synth_series_log(x))


def series_sincos(x: float):
    s, c = ctypes.c_double(), ctypes.c_double()
    _load().synth_series_sincos(x, ctypes.byref(s), ctypes.byref(c))
    return s.value, c.value


# ---------------------------------------------------------------------------
# model tensors of one workload

def mat_shape(shape: Shape, name: str):
    d, hq, hkv, hd, f = shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim
    return {
        "wq": (hq * hd, d), "wk": (hkv * hd, d), "wv": (hkv * hd, d), "wo": (d, hq * hd),
        "wg": (f, d), "wu": (f, d), "wd": (d, f),
    }[name]


def layer_weights(shape: Shape, seed: int, layer: int, std: float = 0.02) -> dict:
    """bf16 bit patterns of one layer's seven matrices ([out, in] row-major) and its gains."""
    out = {}
    for m in MATS:
        out[m] = normal_bf16(seed, layer * 16 + _MAT_ID[m], mat_shape(shape, m), std)
    out["g_attn"] = np.full(shape.d_model, BF16_ONE, dtype=np.uint16)
    out["g_ffn"] = np.full(shape.d_model, BF16_ONE, dtype=np.uint16)
    return out


def embedding(shape: Shape, seed: int, std: float = 0.02) -> np.ndarray:
    """E [V, d] bf16 bits (tied input embedding and LM head)."""
    return normal_bf16(seed, TID_EMBED, (shape.vocab, shape.d_model), std)


def exit_transform(shape: Shape, seed: int, ckpt_index: int, std: float = 0.01) -> np.ndarray:
    """T_c [d, d] bf16 bits, T = I + N(0, std) (row-vector convention u = n T)."""
    d = shape.d_model
    return normal_bf16(seed, TID_T_BASE + ckpt_index, (d, d), std, diag_add=1.0)


def final_gain(shape: Shape) -> np.ndarray:
    return np.full(shape.d_model, BF16_ONE, dtype=np.uint16)


def prompts(shape: Shape, seed: int, lens) -> list:
    """Uniform random prompt token ids in [0, V) per sequence."""
    pseed = seed ^ PROMPT_SEED_XOR
    return [uniform_int(pseed, TID_PROMPT_BASE + s, int(n), 0, shape.vocab - 1)
            for s, n in enumerate(lens)]


def prompt_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    return uniform_int(seed ^ PROMPT_SEED_XOR, TID_PROMPT_LENS, batch, lo, hi)


def workload_inputs(w: Workload):
    """(prompt_lens, prompts) of a workload, from its prompt seed."""
    if w.prompt_len_range is not None:
        lens = prompt_lengths(w.seed, w.batch, *w.prompt_len_range)
    else:
        lens = np.full(w.batch, w.prompt_len, dtype=np.int32)
    return lens, prompts(w.shape, w.seed, lens)
