"""Python binding of libee.so, the GB300 early-exit decoding library.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI of ``include/ee.h``.  PyTorch provides device
memory (the arena and op buffers) and streams.  There is no CPU fallback:
importing works without a GPU, but every call needs the built library and
a CUDA device and raises otherwise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libee.so")

EE_MAX_BATCH = 64
EE_MAX_CHECKPOINTS = 32
MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")

STATUS = {0: "EE_OK", 1: "EE_ERR_INVALID_ARG", 2: "EE_ERR_STATE", 3: "EE_ERR_CAPACITY",
          4: "EE_ERR_OOM_ARENA", 5: "EE_ERR_CUDA", 6: "EE_ERR_DEVICE_TIMEOUT",
          7: "EE_ERR_UNSUPPORTED"}

# every symbol include/ee.h declares
EXPORTS = (
    "ee_arena_bytes", "ee_create", "ee_destroy", "ee_last_error", "ee_load_weights",
    "ee_load_layer", "ee_load_shared", "ee_set_thresholds", "ee_set_exit_enabled",
    "ee_set_use_graph", "ee_prefill", "ee_decode_step", "ee_reset", "ee_seq_info",
    "ee_set_debug", "ee_debug_hidden", "ee_debug_conf", "ee_debug_kv", "ee_debug_block_table",
    "ee_debug_int4", "ee_op_quantize_int4", "ee_op_linear_bf16", "ee_op_linear_int4",
    "ee_attention_scratch_bytes", "ee_op_attention", "ee_head_scratch_bytes",
    "ee_op_vocab_head", "ee_step_io", "ee_set_profile", "ee_profile_read", "ee_last_step_ms",
    "ee_op_attention_noalloc", "ee_set_exit_criterion", "ee_set_token_source",
    "ee_set_prefill_exit", "ee_prefill_exit_layers",
)

LISTS = ("both", "full")  # EE_LISTS_*
KINDS = ("begin", "norm", "qkv", "attn", "o", "gateup", "down", "head_norm", "head_t", "head_e",
         "final_norm", "final_head", "exit_sts")


class EEError(RuntimeError):
    def __init__(self, status: int, msg: str = ""):
        self.status = status
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))


c_i32, c_f32, c_vp, c_sz = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
P = ctypes.POINTER


class EEConfig(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("d_model", c_i32), ("n_heads", c_i32), ("n_kv_heads", c_i32),
                ("head_dim", c_i32), ("ffn_dim", c_i32), ("vocab", c_i32), ("rms_eps", c_f32),
                ("rope_theta", c_f32), ("quant_group", c_i32), ("kv_block", c_i32),
                ("max_batch", c_i32), ("max_seq_len", c_i32), ("n_checkpoints", c_i32),
                ("checkpoint_layers", P(c_i32))]


class EELayerWeights(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "wg", "wu", "wd")] + \
               [("q4", c_vp * 7), ("s4", c_vp * 7)]


class EESharedWeights(ctypes.Structure):
    _fields_ = [("embed", c_vp), ("g_final", c_vp), ("exit_T", P(c_vp))]


class EELaunchRecord(ctypes.Structure):
    _fields_ = [("kind", c_i32), ("layer", c_i32), ("ms", c_f32), ("kernel_ms", c_f32), ("lists", c_i32)]


class EEWeights(ctypes.Structure):
    _fields_ = [("layers", P(EELayerWeights)), ("shared", EESharedWeights)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libee.so; raises if it has not been built (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libee.so not built: run `python -m early_exit_decoding_layer_gb300.build` "
                           "(or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    i32 = c_i32
    sig = {
        "ee_arena_bytes": (c_sz, [P(EEConfig)]),
        "ee_create": (i32, [P(EEConfig), c_vp, c_sz, c_vp, P(c_vp)]),
        "ee_destroy": (None, [c_vp]),
        "ee_last_error": (ctypes.c_char_p, [c_vp]),
        "ee_load_weights": (i32, [c_vp, P(EEWeights)]),
        "ee_load_layer": (i32, [c_vp, i32, P(EELayerWeights)]),
        "ee_load_shared": (i32, [c_vp, P(EESharedWeights)]),
        "ee_set_thresholds": (i32, [c_vp, P(c_f32)]),
        "ee_set_exit_enabled": (i32, [c_vp, i32]),
        "ee_set_exit_criterion": (i32, [c_vp, i32]),
        "ee_set_token_source": (i32, [c_vp, i32]),
        "ee_set_prefill_exit": (i32, [c_vp, P(c_f32)]),
        "ee_prefill_exit_layers": (i32, [c_vp, P(i32)]),
        "ee_set_use_graph": (i32, [c_vp, i32]),
        "ee_prefill": (i32, [c_vp, i32, P(i32), P(i32), P(i32)]),
        "ee_decode_step": (i32, [c_vp, P(i32), P(i32), P(i32)]),
        "ee_reset": (i32, [c_vp]),
        "ee_seq_info": (i32, [c_vp, P(i32), i32, P(i32)]),
        "ee_set_debug": (i32, [c_vp, i32]),
        "ee_debug_hidden": (i32, [c_vp, i32, P(c_f32)]),
        "ee_debug_conf": (i32, [c_vp, P(c_f32)]),
        "ee_debug_kv": (i32, [c_vp, i32, i32, i32, c_vp, c_vp]),
        "ee_debug_block_table": (i32, [c_vp, i32, P(i32), i32, P(i32)]),
        "ee_debug_int4": (i32, [c_vp, i32, i32, c_vp, c_vp]),
        "ee_op_quantize_int4": (i32, [c_vp, i32, i32, c_vp, c_vp, i32, c_vp]),
        "ee_op_linear_bf16": (i32, [i32, i32, i32, c_vp, c_vp, c_vp, c_vp, c_vp]),
        "ee_op_linear_int4": (i32, [i32, i32, i32, c_vp, c_vp, c_vp, i32, c_vp, c_vp, c_vp]),
        "ee_attention_scratch_bytes": (c_sz, [i32, i32, i32, i32, i32]),
        "ee_op_attention": (i32, [i32, i32, i32, i32, i32, c_vp, c_vp, c_vp, c_vp, i32, c_vp, c_vp,
                                  c_vp, c_vp, c_vp]),
        "ee_head_scratch_bytes": (c_sz, [i32]),
        "ee_op_vocab_head": (i32, [i32, i32, i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
        "ee_step_io": (i32, [c_vp, i32, i32, P(c_sz), P(c_sz), P(i32)]),
        "ee_set_profile": (i32, [c_vp, i32]),
        "ee_profile_read": (i32, [c_vp, P(EELaunchRecord), i32, P(i32)]),
        "ee_last_step_ms": (i32, [c_vp, P(c_f32)]),
        "ee_op_attention_noalloc": (i32, [i32, i32, i32, i32, i32, c_vp, c_vp, c_vp, c_vp, i32, c_vp,
                                          c_vp, c_vp, c_vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(a) -> int:
    """Address of a numpy array (host) or torch tensor (host or device)."""
    if a is None:
        return 0
    if isinstance(a, np.ndarray):
        assert a.flags.c_contiguous
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        assert a.is_contiguous()
        return a.data_ptr()
    raise TypeError(type(a))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def make_config(shape, checkpoints: Sequence[int], max_batch: int, max_seq_len: int) -> EEConfig:
    ck = (c_i32 * max(1, len(checkpoints)))(*checkpoints)
    cfg = EEConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                   shape.ffn_dim, shape.vocab, shape.rms_eps, shape.rope_theta, shape.quant_group,
                   shape.kv_block, max_batch, max_seq_len, len(checkpoints),
                   ctypes.cast(ck, P(c_i32)))
    cfg._ck = ck  # keep alive
    return cfg


def arena_bytes(shape, checkpoints, max_batch, max_seq_len) -> int:
    return int(load_library().ee_arena_bytes(ctypes.byref(make_config(shape, checkpoints, max_batch,
                                                                      max_seq_len))))


class DecodeEngine:
    """One early-exit decoding context on one GPU (see include/ee.h)."""

    def __init__(self, shape, checkpoints: Sequence[int], max_batch: int, max_seq_len: int,
                 device: int = 0, stream=None):
        """stream: a torch.cuda.Stream to queue all work on (default: the
        current stream if it is not the legacy default stream, else a stream
        the library creates)."""
        import torch

        self.lib = load_library()
        if not torch.cuda.is_available():
            raise RuntimeError("DecodeEngine needs a CUDA device")
        self.shape = shape
        self.checkpoints = tuple(int(c) for c in checkpoints)
        self.max_batch = max_batch
        self.max_seq_len = max_seq_len
        self.device = torch.device("cuda", device)
        self.cfg = make_config(shape, self.checkpoints, max_batch, max_seq_len)
        nbytes = int(self.lib.ee_arena_bytes(ctypes.byref(self.cfg)))
        if nbytes == 0:
            raise EEError(1, "invalid model configuration")
        self.arena_nbytes = nbytes
        with torch.cuda.device(self.device):
            self._arena = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
            base = (self._arena.data_ptr() + 255) // 256 * 256
            if stream is None:
                stream = torch.cuda.current_stream(self.device)
            self.stream = stream
            stream = stream.cuda_stream
            ctx = c_vp()
            st = self.lib.ee_create(ctypes.byref(self.cfg), base, nbytes, stream, ctypes.byref(ctx))
        if st != 0:
            raise EEError(st, "ee_create failed")
        self.ctx = ctx
        self.batch = 0

    # -- plumbing ------------------------------------------------------------
    def _check(self, st: int):
        if st != 0:
            msg = self.lib.ee_last_error(self.ctx)
            raise EEError(st, msg.decode() if msg else "")

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.ee_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- weights -------------------------------------------------------------
    def load_layer(self, layer: int, w: dict, int4: Optional[dict] = None):
        """w: bf16 bit patterns (uint16 numpy arrays or tensors) named g_attn, wq, wk,
        wv, wo, g_ffn, wg, wu, wd; int4: optional {mat: (packed uint8, scales uint16)}."""
        lw = EELayerWeights()
        keep = []
        for n in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "wg", "wu", "wd"):
            a = w[n] if not isinstance(w[n], np.ndarray) else np.ascontiguousarray(w[n])
            keep.append(a)
            setattr(lw, n, _ptr(a))
        if int4 is not None:
            for k, m in enumerate(MATS):
                q, s = int4[m]
                q = np.ascontiguousarray(q) if isinstance(q, np.ndarray) else q
                s = np.ascontiguousarray(s) if isinstance(s, np.ndarray) else s
                keep += [q, s]
                lw.q4[k] = _ptr(q)
                lw.s4[k] = _ptr(s)
        self._check(self.lib.ee_load_layer(self.ctx, layer, ctypes.byref(lw)))

    def load_shared(self, embed, g_final, exit_T: Sequence):
        keep = [np.ascontiguousarray(a) if isinstance(a, np.ndarray) else a
                for a in [embed, g_final] + list(exit_T)]
        arr = (c_vp * max(1, len(exit_T)))(*[_ptr(t) for t in keep[2:]])
        sw = EESharedWeights(_ptr(keep[0]), _ptr(keep[1]), ctypes.cast(arr, P(c_vp)))
        self._check(self.lib.ee_load_shared(self.ctx, ctypes.byref(sw)))

    # -- settings ------------------------------------------------------------
    def set_thresholds(self, gamma: Sequence[float]):
        g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float32))
        assert g.shape == (len(self.checkpoints),)
        self._check(self.lib.ee_set_thresholds(self.ctx, g.ctypes.data_as(P(c_f32))))

    def set_exit_enabled(self, enabled: bool):
        self._check(self.lib.ee_set_exit_enabled(self.ctx, 1 if enabled else 0))

    CRITERIA = {"maxprob": 0, "sts": 1, "sts_batch": 2}

    def set_exit_criterion(self, criterion: str):
        """'maxprob' (exit-head confidence, default), 'sts' (state transition
        similarity, per sequence) or 'sts_batch' (its batch-minimum rule)."""
        self._check(self.lib.ee_set_exit_criterion(self.ctx, self.CRITERIA[criterion]))

    def set_prefill_exit(self, tau):
        """Sequence-level exit in prefill with thresholds tau (None: off)."""
        if tau is None:
            self._check(self.lib.ee_set_prefill_exit(self.ctx, None))
            return
        t = np.asarray(tau, dtype=np.float32)
        self._check(self.lib.ee_set_prefill_exit(self.ctx, t.ctypes.data_as(P(c_f32))))

    def prefill_exit_layers(self) -> np.ndarray:
        out = np.empty(max(self.batch, 1), dtype=np.int32)
        self._check(self.lib.ee_prefill_exit_layers(self.ctx, out.ctypes.data_as(P(ctypes.c_int32))))
        return out[: self.batch]

    TOKEN_SOURCES = {"final": 0, "exit_head": 1}

    def set_token_source(self, source: str):
        """'final' (final head after the int4 layers, default) or 'exit_head'."""
        self._check(self.lib.ee_set_token_source(self.ctx, self.TOKEN_SOURCES[source]))

    def set_use_graph(self, use_graph: bool):
        self._check(self.lib.ee_set_use_graph(self.ctx, 1 if use_graph else 0))

    def set_debug(self, debug: bool):
        self._check(self.lib.ee_set_debug(self.ctx, 1 if debug else 0))

    # -- decoding ------------------------------------------------------------
    def prefill(self, prompts: Sequence[Sequence[int]]) -> np.ndarray:
        lens = _i32([len(p) for p in prompts])
        toks = _i32(np.concatenate([np.asarray(p, dtype=np.int32) for p in prompts]))
        out = np.zeros(len(prompts), dtype=np.int32)
        self._check(self.lib.ee_prefill(self.ctx, len(prompts), lens.ctypes.data_as(P(c_i32)),
                                        toks.ctypes.data_as(P(c_i32)), out.ctypes.data_as(P(c_i32))))
        self.batch = len(prompts)
        return out

    def decode_step(self, tokens: Sequence[int]):
        t = _i32(tokens)
        assert t.shape == (self.batch,)
        nxt = np.zeros(self.batch, dtype=np.int32)
        ex = np.zeros(self.batch, dtype=np.int32)
        self._check(self.lib.ee_decode_step(self.ctx, t.ctypes.data_as(P(c_i32)),
                                            nxt.ctypes.data_as(P(c_i32)), ex.ctypes.data_as(P(c_i32))))
        return nxt, ex

    def reset(self):
        self._check(self.lib.ee_reset(self.ctx))
        self.batch = 0

    def seq_pos(self, seq: int) -> int:
        b, p = c_i32(), c_i32()
        self._check(self.lib.ee_seq_info(self.ctx, ctypes.byref(b), seq, ctypes.byref(p)))
        return p.value

    def step_io(self, batch: int, heads: bool):
        """(h2d bytes, d2h bytes, kernel launches) of one decode step."""
        h, d, n = c_sz(), c_sz(), c_i32()
        self._check(self.lib.ee_step_io(self.ctx, batch, 1 if heads else 0, ctypes.byref(h),
                                        ctypes.byref(d), ctypes.byref(n)))
        return h.value, d.value, n.value

    def last_step_ms(self) -> float:
        ms = c_f32()
        self._check(self.lib.ee_last_step_ms(self.ctx, ctypes.byref(ms)))
        return ms.value

    def set_profile(self, profile: bool):
        self._check(self.lib.ee_set_profile(self.ctx, 1 if profile else 0))

    def profile_read(self):
        """[(kind name, layer, ms, kernel_ms, lists)] of the last profiled
        step's launches (kernel_ms: the GEMV's or tensor-core GEMM's own time,
        else 0; lists: "both" or "full", the sub-batch lists the launch
        serves)."""
        n = c_i32()
        self._check(self.lib.ee_profile_read(self.ctx, None, 0, ctypes.byref(n)))
        recs = (EELaunchRecord * max(1, n.value))()
        self._check(self.lib.ee_profile_read(self.ctx, recs, n.value, ctypes.byref(n)))
        return [(KINDS[r.kind], r.layer, r.ms, r.kernel_ms, LISTS[r.lists]) for r in recs[: n.value]]

    # -- inspection ----------------------------------------------------------
    def debug_hidden(self, layer: int) -> np.ndarray:
        out = np.zeros((self.batch, self.shape.d_model), dtype=np.float32)
        self._check(self.lib.ee_debug_hidden(self.ctx, layer, out.ctypes.data_as(P(c_f32))))
        return out

    def debug_conf(self) -> np.ndarray:
        out = np.zeros((self.batch, len(self.checkpoints)), dtype=np.float32)
        self._check(self.lib.ee_debug_conf(self.ctx, out.ctypes.data_as(P(c_f32))))
        return out

    def debug_kv(self, seq: int, layer: int, pos: int):
        n = self.shape.n_kv_heads * self.shape.head_dim
        k = np.zeros(n, dtype=np.uint16)
        v = np.zeros(n, dtype=np.uint16)
        self._check(self.lib.ee_debug_kv(self.ctx, seq, layer, pos, k.ctypes.data, v.ctypes.data))
        return k, v

    def debug_block_table(self, seq: int) -> np.ndarray:
        cap = (self.max_seq_len + 15) // 16
        out = np.zeros(cap, dtype=np.int32)
        n = c_i32()
        self._check(self.lib.ee_debug_block_table(self.ctx, seq, out.ctypes.data_as(P(c_i32)), cap,
                                                  ctypes.byref(n)))
        return out[: n.value]

    def debug_int4(self, layer: int, mat: str):
        sh = self.shape
        dq, dk = sh.n_heads * sh.head_dim, sh.n_kv_heads * sh.head_dim
        rows, cols = {"wq": (dq, sh.d_model), "wk": (dk, sh.d_model), "wv": (dk, sh.d_model),
                      "wo": (sh.d_model, dq), "wg": (sh.ffn_dim, sh.d_model),
                      "wu": (sh.ffn_dim, sh.d_model), "wd": (sh.d_model, sh.ffn_dim)}[mat]
        packed = np.zeros((rows, cols // 2), dtype=np.uint8)
        scales = np.zeros((rows, (cols + 127) // 128), dtype=np.uint16)
        self._check(self.lib.ee_debug_int4(self.ctx, layer, MATS.index(mat), packed.ctypes.data,
                                           scales.ctypes.data))
        return packed, scales


# ---------------------------------------------------------------- single kernels

def pair_order(x):
    """Columns of x [..., K] (K % 8 == 0) rearranged into the kernels' activation
    pair order: within each run of 8 the order is 0,4,1,5,2,6,3,7."""
    K = x.shape[-1]
    idx = np.arange(K)
    j = idx % 8
    src = (idx - j) + np.where(j % 2 == 0, j // 2, 4 + j // 2)
    return x[..., src]


def _stream(stream=None) -> int:
    import torch
    return (stream or torch.cuda.current_stream()).cuda_stream


def _raise(st: int, what: str):
    if st != 0:
        raise EEError(st, what)


def quantize_int4(w, stream=None):
    """w: bf16 bits [rows, cols] (torch.int16/uint16 CUDA tensor) -> (packed uint8, scales int16)."""
    import torch
    rows, cols = w.shape
    sstride = (cols + 127) // 128
    packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device=w.device)
    scales = torch.zeros((rows, sstride), dtype=torch.int16, device=w.device)
    _raise(load_library().ee_op_quantize_int4(_ptr(w), rows, cols, _ptr(packed), _ptr(scales), sstride,
                                              _stream(stream)), "ee_op_quantize_int4")
    return packed, scales


def linear_bf16(x_f16, w, err=None, stream=None):
    """x_f16 [M, K] fp16 bits in pair order, w [N, K] bf16 bits -> y [M, N] fp32."""
    import torch
    x = x_f16
    M, K = x.shape
    N = w.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _raise(load_library().ee_op_linear_bf16(M, N, K, _ptr(x), _ptr(w), _ptr(y), _ptr(err),
                                            _stream(stream)), "ee_op_linear_bf16")
    return y


def linear_int4(x_f16, packed, scales, err=None, stream=None):
    """x_f16 [M, K] fp16 bits in pair order, packed [N, K/2], scales [N, S] -> y fp32."""
    import torch
    M, K = x_f16.shape
    N = packed.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x_f16.device)
    _raise(load_library().ee_op_linear_int4(M, N, K, _ptr(x_f16), _ptr(packed), _ptr(scales),
                                            scales.shape[1], _ptr(y), _ptr(err), _stream(stream)),
           "ee_op_linear_int4")
    return y


def attention_scratch_bytes(B, n_heads, n_kv_heads, head_dim, max_ctx) -> int:
    return int(load_library().ee_attention_scratch_bytes(B, n_heads, n_kv_heads, head_dim, max_ctx))


def attention(q, kcache, vcache, block_table, pos, n_heads, n_kv_heads, head_dim, max_ctx,
              scratch=None, err=None, stream=None):
    """q [B, Hq*hd] fp32; caches [blocks, Hkv, 16, hd] fp16 bits; block_table [B, W] int32;
    pos [B] int32.  Returns o [B, Hq*hd] fp32."""
    import torch
    B = q.shape[0]
    if scratch is None:
        scratch = torch.zeros(attention_scratch_bytes(B, n_heads, n_kv_heads, head_dim, max_ctx),
                              dtype=torch.uint8, device=q.device)
    o = torch.empty((B, n_heads * head_dim), dtype=torch.float32, device=q.device)
    _raise(load_library().ee_op_attention(B, n_heads, n_kv_heads, head_dim, max_ctx, _ptr(q), _ptr(kcache),
                                          _ptr(vcache), _ptr(block_table), block_table.shape[1],
                                          _ptr(pos), _ptr(o), _ptr(scratch), _ptr(err),
                                          _stream(stream)), "ee_op_attention")
    return o


ATTN_STATIC_SCRATCH_BYTES = 4 << 20  # EE_ATTN_STATIC_SCRATCH_BYTES


def attention_noalloc(q, kcache, vcache, block_table, pos, n_heads, n_kv_heads, head_dim, max_ctx,
                      out=None, err=None, stream=None):
    """ee_op_attention_noalloc: attention() with the library's fixed scratch array
    instead of a caller buffer.  The C call allocates nothing; pass `out`
    ([B, Hq*hd] fp32) to keep this wrapper from allocating the result either."""
    import torch
    B = q.shape[0]
    o = out if out is not None else torch.empty((B, n_heads * head_dim), dtype=torch.float32,
                                                device=q.device)
    _raise(load_library().ee_op_attention_noalloc(B, n_heads, n_kv_heads, head_dim, max_ctx, _ptr(q),
                                                  _ptr(kcache), _ptr(vcache), _ptr(block_table),
                                                  block_table.shape[1], _ptr(pos), _ptr(o), _ptr(err),
                                                  _stream(stream)), "ee_op_attention_noalloc")
    return o


def head_scratch_bytes(M) -> int:
    return int(load_library().ee_head_scratch_bytes(M))


def vocab_head(u, E, scratch=None, err=None, stream=None):
    """u [M, d] fp16 bits in pair order, E [V, d] bf16 bits -> (conf [M] fp32, argmax [M] int32)."""
    import torch
    M, d = u.shape
    V = E.shape[0]
    if scratch is None:
        scratch = torch.zeros(head_scratch_bytes(M), dtype=torch.uint8, device=u.device)
    conf = torch.empty(M, dtype=torch.float32, device=u.device)
    arg = torch.empty(M, dtype=torch.int32, device=u.device)
    _raise(load_library().ee_op_vocab_head(M, V, d, _ptr(u), _ptr(E), _ptr(conf), _ptr(arg),
                                           _ptr(scratch), _ptr(err), _stream(stream)),
           "ee_op_vocab_head")
    return conf, arg
