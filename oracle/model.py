"""CPU oracle of the early-exit decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import or run anything under ``oracle/``.  The CUDA
library never calls it and it never calls the CUDA library; the two share
only the seeded inputs of the ``synth`` module.

What it computes (plain, slow, in numpy float64 unless a step fixes another
precision), following the three pages on early-exit decoding:

* "River-LLM 深度解析" (page 1): exit layers are parameter copies of each
  backbone layer quantised to W4A16 (§4.1-4.2 and the ``ExitLayer`` code of
  §8.1: scale = max|w|/7, q = clamp(round(w/scale), -8, 7), dequant q*scale);
  they write K/V into the same cache slots as the backbone layers (§4.3,
  §8.2 ``SharedKVCache``); a KV-cached decoder attends over the history
  (§3.1 ``CachedAttention``) and the uncached generation loop of §2.2
  recomputes every position (used here as an independent check).
* the CALM article (page 2): the decode loop of §3.1 (embed, run a layer,
  update the KV cache, score confidence, exit once the score clears the
  layer's threshold, otherwise finish with the LM head); a sharp softmax is
  a confident one (§2.1); one fixed threshold per layer (§2.2).
* "大语言模型解码加速：自适应层并行机制解析" (page 3): the low-rank exit head
  softmax(h^(l) T^(l) E^T) with T in R^{d x d} (§2.1) and the test
  p(t|h^(l)) > gamma (§2.2).

Readings where the pages are silent (each also listed in the design notes):
* the exit rule is max softmax(RMSNorm_final(h_l) T_l E^T) > gamma_l, strict;
  heads are evaluated in increasing layer order while a sequence is still
  on the full-precision path; the first one that clears wins;
* after an exit at checkpoint l the layers l+1..L-1 run on the int4 copies
  and the token emitted is the final head's argmax (lowest index on ties);
* int4 groups are 128 consecutive input columns of one output row with a
  bf16 scale (a final partial group when in % 128 != 0); the quantiser runs
  in float32 (scale = bf16_rne(amax/7), q = clamp(rint_half_even(w/s), -8, 7));
* Llama layer: RMSNorm (eps 1e-5), rotate-half RoPE (theta 1e4), GQA with
  head h reading kv head floor(h*Hkv/Hq), SwiGLU FFN, no biases, tied E;
* prefill is the plain bf16 stack over all prompt positions with no exit;
* the KV cache is paged in 16-token blocks allocated in ascending id order
  from a free list (prefill: sequences in order; decode: a new block for a
  sequence whose position is a multiple of 16, sequences in order).

Parity status: the pieces are pinned by the ``-m "not gpu"`` tests (int4
round trips and a hand-worked quantisation, closed forms of RMSNorm, RoPE,
attention and the exit head, the uncached recompute, the all-int4 model, KV
coverage, batch independence).  The whole-model token and exit traces have
no printed worked example on the pages: beyond those pins they are
"parity unpinned".
"""
from __future__ import annotations

import copy
import math
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

import numpy as np

# ---------------------------------------------------------------------------
# bf16 helpers (IEEE-754 binary32 with the low 16 mantissa bits removed)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16, ties to even (IEEE roundTiesToEven
    on the 8-bit significand).  NaN is not expected here."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# int4 exit-layer weights (page 1 §4.2 and §8.1 `_quantize_int4`, grouped)


def quantize_int4_group(w_bits: np.ndarray, group: int = 128):
    """Group-wise symmetric int4 quantisation of a bf16 matrix [out, in].

    Page 1 §8.1 quantises a whole tensor with scale = max|w| / 7 and
    q = clamp(round(w / scale), -8, 7) (torch.round: half to even).  The
    exit stack here applies the same rule to each group of ``group``
    consecutive input columns of one output row, with the scale stored in
    bf16.  Arithmetic in float32 (the precision the GPU library takes the
    same integer decisions in): amax is exact, amax/7 is one correctly
    rounded float32 division, rounded again to bf16 (nearest even); w/s is
    one correctly rounded float32 division, rounded half to even.  amax = 0
    gives s = 0 and q = 0.

    Returns (q int8 [out, in], scale bf16 bits uint16 [out, ceil(in/group)]).
    """
    w = bf16_to_f32(w_bits)
    out_dim, in_dim = w.shape
    ng = (in_dim + group - 1) // group
    q = np.zeros((out_dim, in_dim), dtype=np.int8)
    s_bits = np.zeros((out_dim, ng), dtype=np.uint16)
    for gi in range(ng):
        c0, c1 = gi * group, min(in_dim, (gi + 1) * group)
        blk = w[:, c0:c1]
        amax = np.max(np.abs(blk), axis=1).astype(np.float32)
        s32 = (amax / np.float32(7.0)).astype(np.float32)
        sb = f32_to_bf16_bits(s32)
        s = bf16_to_f32(sb)
        s_bits[:, gi] = sb
        safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        ratio = (blk / safe[:, None]).astype(np.float32)
        qq = np.clip(np.rint(ratio), -8, 7)
        qq = np.where(s[:, None] == 0, 0, qq)
        q[:, c0:c1] = qq.astype(np.int8)
    return q, s_bits


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Two's-complement nibbles, two per byte: byte j of a row holds column
    2j in its low nibble and column 2j+1 in its high nibble."""
    q = np.asarray(q, dtype=np.int8)
    assert q.shape[1] % 2 == 0
    nib = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed: np.ndarray, in_dim: int) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    out = np.empty((p.shape[0], in_dim), dtype=np.int16)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    out = np.where(out >= 8, out - 16, out)
    return out.astype(np.int8)


def dequant_int4(q: np.ndarray, s_bits: np.ndarray, group: int = 128) -> np.ndarray:
    """W4A16 dequantisation q * s (page 1 §8.1 forward: quantized.float() * scale).
    Exact: |q| <= 8 and s has an 8-bit significand, so q*s fits float32."""
    s = bf16_to_f64(s_bits)
    cols = np.arange(q.shape[1]) // group
    return q.astype(np.float64) * s[:, cols]


# ---------------------------------------------------------------------------
# Llama decoder pieces


def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T with W stored [out, in] (the F.linear call of page 1 §8.1)."""
    return x @ W.T


def rmsnorm(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis (Llama RMSNorm)."""
    h = np.asarray(h, dtype=np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    return h / np.sqrt(ms + eps) * g


def rope_angles(pos: int, head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return pos * inv_freq


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of x [..., head_dim] at absolute position pos:
    pairs (i, i + hd/2) rotate by pos * theta^(-2i/hd)."""
    hd = x.shape[-1]
    half = hd // 2
    a = rope_angles(pos, hd, theta)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(z: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(z, axis=axis, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention_decode(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """One query position against its KV history (page 1 §3.1):
    softmax(q K^T / sqrt(d_k)) V per query head; q [Hq, hd], K/V [ctx, Hkv, hd].
    Query head h reads kv head floor(h * Hkv / Hq)."""
    hq, hd = q.shape
    hkv = K.shape[1]
    out = np.empty((hq, hd), dtype=np.float64)
    for h in range(hq):
        g = (h * hkv) // hq
        scores = K[:, g, :] @ q[h] / math.sqrt(hd)
        p = softmax(scores)
        out[h] = p @ V[:, g, :]
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    return silu(gate) * up


def head_logits(h: np.ndarray, g_final: np.ndarray, E: np.ndarray, eps: float,
                T: Optional[np.ndarray] = None) -> np.ndarray:
    """Logits of the LM head (T None) or of a checkpoint exit head:
    RMSNorm_final(h) [T] E^T (page 3 §2.1: softmax(h^(l) T^(l) E^T))."""
    n = rmsnorm(h, g_final, eps)
    u = n @ T if T is not None else n     # row-vector convention u = n T
    return linear(u, E)


def max_softmax(z: np.ndarray) -> float:
    """Confidence = largest softmax probability = 1 / sum_v exp(z_v - z_max)
    (page 2 §2.1: a sharp distribution is a confident one)."""
    m = np.max(z)
    return float(1.0 / np.sum(np.exp(z - m)))


def state_transition_similarity(h_in: np.ndarray, h_out: np.ndarray, eps: float = 1e-12) -> float:
    """River-LLM §5.1 (compute_sts): the cosine between a layer's input and
    output states, each first scaled to unit L2 norm (F.normalize: x divided
    by max(||x||, eps)), then their dot product.  A high value means the layer
    barely changed the token's state.  O(d); no vocabulary read (§5.3)."""
    a = np.asarray(h_in, dtype=np.float64)
    b = np.asarray(h_out, dtype=np.float64)
    a = a / max(float(np.linalg.norm(a)), eps)
    b = b / max(float(np.linalg.norm(b)), eps)
    return float(np.dot(a, b))


def argmax_lowest(z: np.ndarray) -> int:
    """Greedy token: argmax with ties to the lowest index (np.argmax's rule)."""
    return int(np.argmax(z))


def top2_margin(z: np.ndarray) -> float:
    if z.size < 2:
        return float("inf")
    part = np.partition(z, -2)
    return float(part[-1] - part[-2])


# ---------------------------------------------------------------------------
# weights


@dataclass
class ModelConfig:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    quant_group: int = 128
    kv_block: int = 16
    checkpoints: tuple = ()

    @classmethod
    def from_shape(cls, shape, checkpoints):
        return cls(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads,
                   shape.head_dim, shape.ffn_dim, shape.vocab, shape.rms_eps,
                   shape.rope_theta, shape.quant_group, shape.kv_block, tuple(checkpoints))


MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


class Weights:
    """bf16 backbone weights (bit patterns), their int4 copies and the head
    tensors, served as float64 arrays.

    ``layer_src(j)`` returns a dict with the seven bf16 matrices and two
    gains of layer j as uint16 bit patterns (e.g. from ``synth``); the int4
    copy of each matrix is made here with ``quantize_int4_group`` unless
    ``int4_src`` supplies (packed, scales) pairs.  Converted layers are
    cached while the cache stays under ``cache_bytes``.
    """

    def __init__(self, cfg: ModelConfig, layer_src: Callable[[int], dict], E_bits: np.ndarray,
                 g_final_bits: np.ndarray, T_bits: Sequence[np.ndarray],
                 int4_src: Optional[Callable[[int], dict]] = None, cache_bytes: int = 4 << 30):
        self.cfg = cfg
        self._layer_src = layer_src
        self._int4_src = int4_src
        self.E = bf16_to_f64(E_bits)
        self.E_bits = E_bits
        self.g_final = bf16_to_f64(g_final_bits)
        self.T = [bf16_to_f64(t) for t in T_bits]
        self._cache: Dict[tuple, dict] = {}
        self._cache_bytes = cache_bytes
        self._cached = 0

    def int4_layer(self, j: int) -> dict:
        """{mat: (packed uint8 [out, in/2], scale bits [out, ngroups])}."""
        if self._int4_src is not None:
            return self._int4_src(j)
        src = self._layer_src(j)
        out = {}
        for m in MATS:
            q, s = quantize_int4_group(src[m], self.cfg.quant_group)
            out[m] = (pack_int4(q), s)
        return out

    def layer(self, j: int, int4: bool) -> dict:
        key = (j, bool(int4))
        if key in self._cache:
            return self._cache[key]
        lw = self._convert(j, bool(int4))
        self._keep(key, lw)
        return lw

    def _keep(self, key, lw: dict):
        nbytes = sum(v.nbytes for v in lw.values())
        if self._cached + nbytes <= self._cache_bytes:
            self._cache[key] = lw
            self._cached += nbytes

    def warm(self, keys, workers: int = 8):
        """Converts the (layer, int4) entries ``keys`` ahead of use on a few
        host threads (the conversions are independent numpy passes) and keeps
        them within the cache budget.  No arithmetic differs from ``layer``."""
        from concurrent.futures import ThreadPoolExecutor

        todo = [(int(j), bool(q)) for j, q in keys if (int(j), bool(q)) not in self._cache]
        with ThreadPoolExecutor(max(1, workers)) as ex:
            for key, lw in zip(todo, ex.map(lambda k: self._convert(*k), todo)):
                self._keep(key, lw)

    def _convert(self, j: int, int4: bool) -> dict:
        src = self._layer_src(j)
        lw = {"g_attn": bf16_to_f64(src["g_attn"]), "g_ffn": bf16_to_f64(src["g_ffn"])}
        if int4:
            q4 = self.int4_layer(j)
            for m in MATS:
                packed, s = q4[m]
                in_dim = src[m].shape[1]
                lw[m] = dequant_int4(unpack_int4(packed, in_dim), s, self.cfg.quant_group)
        else:
            for m in MATS:
                lw[m] = bf16_to_f64(src[m])
        return lw


# ---------------------------------------------------------------------------
# one decoder layer, one position, with the KV history (page 2 §3.1 loop body)


def layer_decode(cfg: ModelConfig, lw: dict, h: np.ndarray, pos: int,
                 k_hist: np.ndarray, v_hist: np.ndarray):
    """Run one layer for one token at position ``pos``.  ``k_hist``/``v_hist``
    [max_ctx, Hkv, hd] hold this layer's history; the new K/V are written at
    ``pos`` first (shared-cache write, page 1 §4.3) and attention covers
    positions 0..pos.  Returns the new residual stream h."""
    hq, hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n = rmsnorm(h, lw["g_attn"], cfg.rms_eps)
    q = linear(n, lw["wq"]).reshape(hq, hd)
    k = linear(n, lw["wk"]).reshape(hkv, hd)
    v = linear(n, lw["wv"]).reshape(hkv, hd)
    q = rope(q, pos, cfg.rope_theta)
    k = rope(k, pos, cfg.rope_theta)
    k_hist[pos] = k
    v_hist[pos] = v
    o = attention_decode(q, k_hist[: pos + 1], v_hist[: pos + 1])
    h = h + linear(o.reshape(-1), lw["wo"])
    n2 = rmsnorm(h, lw["g_ffn"], cfg.rms_eps)
    a = swiglu(linear(n2, lw["wg"]), linear(n2, lw["wu"]))
    return h + linear(a, lw["wd"])


# ---------------------------------------------------------------------------
# full causal forward over all positions (page 1 §2.2 uncached loop; prefill)


def layer_full(cfg: ModelConfig, lws: Sequence[dict], x: np.ndarray, rows_q4: np.ndarray):
    """One decoder layer over positions 0..P-1 of one sequence, causal.
    ``lws[0]`` is the bf16 layer; rows where ``rows_q4`` is set use the int4
    copy ``lws[1]``.  Returns (new residual stream [P, d], K, V [P, Hkv, hd])."""
    P = x.shape[0]
    hq, hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    mask = np.triu(np.full((P, P), -np.inf), k=1)

    def proj(name, inp):
        out = linear(inp, lws[0][name])
        if rows_q4.any():
            out[rows_q4] = linear(inp[rows_q4], lws[1][name])
        return out

    n = rmsnorm(x, lws[0]["g_attn"], cfg.rms_eps)
    Q = proj("wq", n).reshape(P, hq, hd)
    K = proj("wk", n).reshape(P, hkv, hd)
    V = proj("wv", n).reshape(P, hkv, hd)
    for p in range(P):
        Q[p] = rope(Q[p], p, cfg.rope_theta)
        K[p] = rope(K[p], p, cfg.rope_theta)
    O = np.empty((P, hq, hd))
    for hh in range(hq):
        g = (hh * hkv) // hq
        S = Q[:, hh, :] @ K[:, g, :].T / math.sqrt(hd) + mask
        O[:, hh, :] = softmax(S, axis=-1) @ V[:, g, :]
    x = x + proj("wo", O.reshape(P, hq * hd))
    n2 = rmsnorm(x, lws[0]["g_ffn"], cfg.rms_eps)
    x = x + proj("wd", swiglu(proj("wg", n2), proj("wu", n2)))
    return x, K, V


def forward_full(cfg: ModelConfig, W: Weights, tokens: Sequence[int],
                 int4_after: Optional[Sequence[Optional[int]]] = None,
                 return_kv: bool = False):
    """Plain matrix-form forward of a whole token sequence with a causal mask.

    ``int4_after[p]`` = l means position p ran layers l+1..L-1 on the int4
    copies (None: all bf16).  Returns (hidden states [L, P, d] after each
    layer, logits of the last position[, K [L, P, Hkv, hd], V]).
    """
    P = len(tokens)
    L, hq, hkv, hd = cfg.n_layers, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    if int4_after is None:
        int4_after = [None] * P
    x = W.E[np.asarray(tokens, dtype=np.int64)].copy()
    hs = np.empty((L, P, cfg.d_model))
    Ks = np.empty((L, P, hkv, hd)) if return_kv else None
    Vs = np.empty((L, P, hkv, hd)) if return_kv else None
    for j in range(L):
        rows_q4 = np.array([a is not None and j > a for a in int4_after], dtype=bool)
        lws = [W.layer(j, False)]
        if rows_q4.any():
            lws.append(W.layer(j, True))
        x, K, V = layer_full(cfg, lws, x, rows_q4)
        if return_kv:
            Ks[j], Vs[j] = K, V
        hs[j] = x
    logits = head_logits(x[-1], W.g_final, W.E, cfg.rms_eps)
    if return_kv:
        return hs, logits, Ks, Vs
    return hs, logits


# ---------------------------------------------------------------------------
# the decode engine with a paged-slot bookkeeping model


@dataclass
class SeqState:
    pos: int = 0                       # tokens already in the cache
    blocks: List[int] = field(default_factory=list)
    tokens: List[int] = field(default_factory=list)
    int4_after: List[Optional[int]] = field(default_factory=list)


@dataclass
class StepResult:
    next_tokens: np.ndarray            # [B] int32
    exit_layers: np.ndarray            # [B] int32
    conf: np.ndarray                   # [B, n_ckpt] float64, nan where not evaluated
    hidden: np.ndarray                 # [L, B, d] residual stream after each layer
    final_logits: np.ndarray           # [B, V]
    margins: np.ndarray                # [B] top-2 final-logit margin


class Oracle:
    """Early-exit greedy decoding of B independent sequences.

    Each sequence keeps a contiguous K/V history per layer and a model of the
    paged cache's block table.  A decode step follows page 2 §3.1: embed,
    then per layer run it (bf16 until the sequence exits, the int4 copy
    after), write K/V at the current position, and at checkpoint layers
    score the exit criterion against the layer's threshold (strict >, page 3
    §2.2).  The token is the final head's argmax.

    Exit criteria (``criterion``):
    * ``"maxprob"`` -- max softmax(RMSNorm_final(h) T_l E^T) (page 3 §2.1-2.2),
      per sequence;
    * ``"sts"`` -- the state transition similarity of the checkpoint layer,
      cos(layer input, layer output) (River-LLM §5.1), per sequence: each
      generated token decides its own exit layer (§6.1);
    * ``"sts_batch"`` -- the same score with the batch rule of River-LLM §5.2
      (ExitDecision.should_exit): the sequences still on the full-precision
      path exit together when the minimum of their scores clears tau; the
      score recorded for each of them is that minimum.
    """

    CRITERIA = ("maxprob", "sts", "sts_batch")

    TOKEN_SOURCES = ("final", "exit_head")

    def __init__(self, cfg: ModelConfig, W: Weights, max_batch: int, max_seq_len: int,
                 criterion: str = "maxprob", token_source: str = "final"):
        self.cfg = cfg
        self.W = W
        self.max_batch = max_batch
        self.max_seq_len = max_seq_len
        self.blocks_per_seq = (max_seq_len + cfg.kv_block - 1) // cfg.kv_block
        self.n_blocks = max_batch * self.blocks_per_seq
        self.gamma = np.full(len(cfg.checkpoints), np.inf)
        assert criterion in self.CRITERIA
        assert token_source in self.TOKEN_SOURCES
        assert token_source == "final" or criterion == "maxprob", "an exit-head token needs the exit head"
        self.criterion = criterion
        # "final": the token is the final head's argmax after the int4 layers;
        # "exit_head": an exited sequence's token is the argmax of the exit
        # head that let it leave (the CALM article §3.1 loop returns the exit
        # head's prediction; page 3 §2.2), and its remaining layers only
        # write their K/V
        self.token_source = token_source
        self.reset()

    # -- lifecycle ---------------------------------------------------------
    def reset(self):
        self.free = list(range(self.n_blocks))   # ascending: lowest id first
        self.seqs: List[SeqState] = []
        L, hkv, hd = self.cfg.n_layers, self.cfg.n_kv_heads, self.cfg.head_dim
        self.K: List[np.ndarray] = []
        self.V: List[np.ndarray] = []
        self._kv_shape = (L, self.max_seq_len, hkv, hd)

    def set_thresholds(self, gamma):
        g = np.asarray(gamma, dtype=np.float64)
        assert g.shape == (len(self.cfg.checkpoints),)
        self.gamma = g.copy()

    def snapshot(self):
        return copy.deepcopy((self.free, self.seqs, self.K, self.V))

    def restore(self, snap):
        self.free, self.seqs, self.K, self.V = copy.deepcopy(snap)

    def _alloc_block(self, s: int):
        if not self.free:
            raise RuntimeError("KV cache out of blocks")
        self.seqs[s].blocks.append(self.free.pop(0))

    def slot(self, s: int, pos: int):
        """(block id, offset) of position pos of sequence s."""
        b = self.cfg.kv_block
        return self.seqs[s].blocks[pos // b], pos % b

    # -- prefill: plain bf16 stack over all prompt positions, no exit --------
    def prefill(self, prompts: Sequence[Sequence[int]], exit_tau=None) -> np.ndarray:
        """Prefill phase.  Without ``exit_tau`` the plain bf16 stack runs over
        every prompt position.  With it, sequence-level exit (River-LLM §6.1,
        the prefill half of its two-phase strategy): at each checkpoint layer
        l every token of a prompt is scored by the state transition
        similarity of layer l (§5.1), and the whole prompt leaves the
        full-precision path when the minimum over its tokens is above
        exit_tau[c] (the batch rule of §5.2 over the prompt's tokens); its
        layers after l run on the int4 copies for all its tokens and write
        their K/V.  ``self.prefill_exits[s]`` is the layer sequence s left at
        (n_layers - 1: none).  The first token is the final head's argmax."""
        assert 1 <= len(prompts) <= self.max_batch
        self.reset()
        cfg = self.cfg
        L, ck = cfg.n_layers, list(cfg.checkpoints)
        first = np.empty(len(prompts), dtype=np.int32)
        xs = []
        for s, toks in enumerate(prompts):
            P = len(toks)
            assert 1 <= P < self.max_seq_len
            self.seqs.append(SeqState(pos=P, tokens=list(int(t) for t in toks),
                                      int4_after=[None] * P))
            for _ in range((P + cfg.kv_block - 1) // cfg.kv_block):
                self._alloc_block(s)
            self.K.append(np.full(self._kv_shape, np.nan))
            self.V.append(np.full(self._kv_shape, np.nan))
            xs.append(self.W.E[np.asarray(toks, dtype=np.int64)].copy())
        exited: List[Optional[int]] = [None] * len(prompts)
        self.prefill_scores = np.full((len(prompts), len(ck)), np.nan)   # minimum over tokens
        # the sequences are independent: each layer's weights serve all of
        # them in turn (the same arithmetic as forward_full per sequence)
        for j in range(L):
            lws = {}
            for s in range(len(prompts)):
                P = xs[s].shape[0]
                q4 = exited[s] is not None
                if False not in lws:
                    lws[False] = self.W.layer(j, False)
                if q4 and True not in lws:
                    lws[True] = self.W.layer(j, True)
                x_in = xs[s]
                layers = [lws[False], lws[True]] if q4 else [lws[False]]
                xs[s], K, V = layer_full(cfg, layers, xs[s], np.full(P, q4, dtype=bool))
                self.K[s][j, :P], self.V[s][j, :P] = K, V
                if exit_tau is not None and j in ck and not q4:
                    c = ck.index(j)
                    low = min(state_transition_similarity(x_in[p], xs[s][p]) for p in range(P))
                    self.prefill_scores[s, c] = low
                    if low > exit_tau[c]:
                        exited[s] = j
        self.prefill_exits = np.array([L - 1 if e is None else e for e in exited], dtype=np.int32)
        for s in range(len(prompts)):
            self.seqs[s].int4_after = [exited[s]] * len(prompts[s])
            logits = head_logits(xs[s][-1], self.W.g_final, self.W.E, cfg.rms_eps)
            first[s] = argmax_lowest(logits)
        return first

    # -- one decode step ---------------------------------------------------
    def decode_step(self, in_tokens: Sequence[int],
                    forced_exit: Optional[Sequence[Optional[int]]] = None,
                    eval_heads: bool = True) -> StepResult:
        """Decode one token for every sequence.

        ``forced_exit[s]`` (a checkpoint layer, -1 for "never", or None to
        let the threshold decide) overrides the decision of sequence s; the
        heads are still scored so that confidences can be compared.
        ``eval_heads=False`` is the forced no-exit baseline (no head runs).
        """
        cfg = self.cfg
        B = len(self.seqs)
        assert len(in_tokens) == B
        L, d = cfg.n_layers, cfg.d_model
        ck = list(cfg.checkpoints)
        next_tokens = np.empty(B, dtype=np.int32)
        exit_layers = np.full(B, L - 1, dtype=np.int32)
        conf = np.full((B, len(ck)), np.nan)
        hidden = np.empty((L, B, d))
        logits_all = np.empty((B, cfg.vocab))
        margins = np.empty(B)
        for s in range(B):
            if self.seqs[s].pos >= self.max_seq_len:
                raise RuntimeError("sequence exceeds max_seq_len")
        h = []
        for s in range(B):
            if self.seqs[s].pos % cfg.kv_block == 0:
                self._alloc_block(s)
            h.append(self.W.E[int(in_tokens[s])].copy())
        exited_at: List[Optional[int]] = [None] * B
        head_z: List[Optional[np.ndarray]] = [None] * B   # logits of each checkpoint head scored
        # the sequences are independent: each layer's weights serve all of
        # them in turn; every sequence runs the per-token loop of page 2 §3.1
        for j in range(L):
            lws = {}
            scored = []   # sequences scored at this checkpoint
            for s in range(B):
                q4 = exited_at[s] is not None
                if q4 not in lws:
                    lws[q4] = self.W.layer(j, q4)
                pos = self.seqs[s].pos
                h_in = h[s]
                h[s] = layer_decode(cfg, lws[q4], h[s], pos, self.K[s][j], self.V[s][j])
                hidden[j, s] = h[s]
                if j in ck and exited_at[s] is None and eval_heads:
                    c = ck.index(j)
                    if self.criterion in ("sts", "sts_batch"):
                        conf[s, c] = state_transition_similarity(h_in, h[s])
                    else:
                        z = head_logits(h[s], self.W.g_final, self.W.E, cfg.rms_eps, self.W.T[c])
                        conf[s, c] = max_softmax(z)
                        head_z[s] = z
                    scored.append(s)
            if scored:
                c = ck.index(j)
                if self.criterion == "sts_batch":   # the batch's score is its minimum
                    low = min(conf[s, c] for s in scored)
                    for s in scored:
                        conf[s, c] = low
                for s in scored:
                    f = None if forced_exit is None else forced_exit[s]
                    go = conf[s, c] > self.gamma[c] if f is None else (f == j)
                    if go:
                        exited_at[s] = j
                        exit_layers[s] = j
        for s in range(B):
            st = self.seqs[s]
            if self.token_source == "exit_head" and exited_at[s] is not None:
                z = head_z[s]   # the exit head's logits at the exit layer
            else:
                z = head_logits(h[s], self.W.g_final, self.W.E, cfg.rms_eps)
            logits_all[s] = z
            margins[s] = top2_margin(z)
            next_tokens[s] = argmax_lowest(z)
            st.tokens.append(int(in_tokens[s]))
            st.int4_after.append(exited_at[s])
            st.pos = st.pos + 1
        return StepResult(next_tokens, exit_layers, conf, hidden, logits_all, margins)


# ---------------------------------------------------------------------------
# threshold calibration


def calibrate_gammas(orc: Oracle, prompts, steps: int, percentiles: Sequence[float]):
    """gamma_l = the p-th percentile (linear interpolation, numpy's default)
    of the confidences at checkpoint l over decode steps 1..steps with no
    exit (gamma = +inf), one sample per sequence and step.  Returns
    {p: gamma array} and the raw samples [steps, B, n_ckpt]."""
    orc.set_thresholds(np.full(len(orc.cfg.checkpoints), np.inf))
    tok = orc.prefill(prompts)
    samples = []
    for _ in range(steps):
        r = orc.decode_step(tok)
        samples.append(r.conf)
        tok = r.next_tokens
    S = np.stack(samples)
    flat = S.reshape(-1, S.shape[-1])
    return {p: np.percentile(flat, p, axis=0) for p in percentiles}, S


def build_oracle(workload, cache_bytes: int = 4 << 30, max_batch: Optional[int] = None,
                 max_seq_len: Optional[int] = None, criterion: str = "maxprob",
                 token_source: str = "final") -> Oracle:
    """Oracle over a workload's seeded synthetic weights (``synth`` module)."""
    import synth

    shape = workload.shape
    cfg = ModelConfig.from_shape(shape, workload.checkpoints)
    seed = workload.seed
    W = Weights(cfg, lambda j: synth.layer_weights(shape, seed, j), synth.embedding(shape, seed),
                synth.final_gain(shape),
                [synth.exit_transform(shape, seed, c) for c in range(len(workload.checkpoints))],
                cache_bytes=cache_bytes)
    return Oracle(cfg, W, max_batch or workload.batch, max_seq_len or workload.max_seq_len(), criterion,
                  token_source)
