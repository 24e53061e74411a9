"""Model shapes and decode workloads of the early-exit benchmark.

Shapes are those of the Llama-style decoders the workloads name (a tiny
4-layer model, Llama-3.2-1B, Llama-3.1-8B and CodeLlama-34B); the numbers are
architecture hyper-parameters, not method arithmetic.  Checkpoint layers are
zero-indexed; "every k" means layers k, 2k, ... up to L-2 (a decision after
the last layer could not skip anything).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Shape:
    name: str
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


def checkpoints_every(k: int, n_layers: int) -> Tuple[int, ...]:
    return tuple(range(k, n_layers - 1, k))


SHAPES = {
    "tiny": Shape("tiny", 4, 256, 4, 2, 64, 704, 2048),
    "llama3.2-1b": Shape("llama3.2-1b", 16, 2048, 32, 8, 64, 8192, 128256),
    "llama3.1-8b": Shape("llama3.1-8b", 32, 4096, 32, 8, 128, 14336, 128256),
    "codellama-34b": Shape("codellama-34b", 48, 8192, 64, 8, 128, 22016, 32016),
}


@dataclass(frozen=True)
class Workload:
    name: str
    shape: Shape
    checkpoints: Tuple[int, ...]
    batch: int
    prompt_len: int
    steps: int
    seed: int
    gamma_percentiles: Tuple[float, ...] = (40.0,)
    prompt_len_range: Optional[Tuple[int, int]] = None
    calib_steps: int = 8
    extra: dict = field(default_factory=dict)

    def max_prompt(self) -> int:
        return self.prompt_len_range[1] if self.prompt_len_range else self.prompt_len

    def max_seq_len(self) -> int:
        return self.max_prompt() + self.steps + 1


WORKLOADS = {
    "tiny-b1": Workload("tiny-b1", SHAPES["tiny"], (1, 2), 1, 32, 16, 1234),
    "llama3.2-1b-b1": Workload("llama3.2-1b-b1", SHAPES["llama3.2-1b"],
                               checkpoints_every(4, 16), 1, 512, 256, 1235),
    "llama3.1-8b-b1": Workload("llama3.1-8b-b1", SHAPES["llama3.1-8b"],
                               checkpoints_every(4, 32), 1, 2048, 256, 1236),
    "llama3.1-8b-b32": Workload("llama3.1-8b-b32", SHAPES["llama3.1-8b"],
                                checkpoints_every(4, 32), 32, 0, 128, 1237,
                                gamma_percentiles=(40.0, 70.0), prompt_len_range=(256, 2048)),
    "codellama-34b-b8": Workload("codellama-34b-b8", SHAPES["codellama-34b"],
                                 checkpoints_every(8, 48), 8, 4096, 256, 1238),
}
