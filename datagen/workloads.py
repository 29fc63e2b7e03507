"""Workload recipes: which tensors each synthetic configuration draws.

Every tensor is drawn from its own named stream of the configuration's master
seed, so a tensor does not depend on which others are generated or in what
order.  Distributions (all configurations):

* activations and upstream gradients (x, q, k, gate, up, every dy): N(0, 1)
* RMSNorm weight w: 1 + N(0, 0.1)
* lm_head weight W: N(0, 0.02)
* hidden states X feeding the lm_head: N(0, 1)
* labels: uniform in [0, V), with exactly round(p * T) distinct rows set to
  ignore_index = -100 (p = 0.05 on the tiny set, 0.10 elsewhere)

Shapes follow the Llama-3-8B / Qwen-7B decoder shapes: hidden 4096, 32 query
heads of 128, 8 KV heads (Llama-3-8B) or 32 (Qwen-7B), intermediate 11008,
vocab 128256 (Llama-3) or 151936 (Qwen).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

IGNORE_INDEX = -100


@dataclass(frozen=True)
class Tensor:
    name: str                 # stream name
    shape: tuple
    kind: str                 # "normal" | "labels"
    mean: float = 0.0
    std: float = 1.0
    float_dtype: bool = True  # stored in the workload's float dtype


@dataclass
class Workload:
    name: str
    seed: int
    dtype: str                               # "f32" or "bf16"
    params: dict
    tensors: dict = field(default_factory=dict)

    def spec(self, key: str) -> Tensor:
        return self.tensors[key]

    def make(self, key: str, out: np.ndarray | None = None) -> np.ndarray:
        """Draw tensor `key` (storage dtype; bf16 as uint16 bits)."""
        from . import labels, normal
        t = self.tensors[key]
        if t.kind == "labels":
            p = self.params
            return labels(self.seed, t.name, p["T"], p["V"], p["ignore_frac"], IGNORE_INDEX)
        return normal(self.seed, t.name, t.shape, self.dtype, t.mean, t.std, out=out)

    def make_all(self, keys=None) -> dict:
        return {k: self.make(k) for k in (keys or self.tensors)}


def _n(name, shape, mean=0.0, std=1.0):
    return Tensor(name, tuple(shape), "normal", mean, std)


def rmsnorm(seed, T, H, eps, dtype, prefix="rmsnorm") -> Workload:
    w = Workload(f"{prefix}[{T}x{H}]", seed, dtype, {"T": T, "H": H, "eps": eps})
    w.tensors = {"x": _n(f"{prefix}.x", (T, H)), "w": _n(f"{prefix}.w", (H,), 1.0, 0.1),
                 "dy": _n(f"{prefix}.dy", (T, H))}
    return w


def rope(seed, B, S, Hq, Hk, D, theta, dtype, prefix="rope") -> Workload:
    w = Workload(f"{prefix}[{B},{S},{Hq}/{Hk},{D}]", seed, dtype,
                 {"B": B, "S": S, "Hq": Hq, "Hk": Hk, "D": D, "theta": theta})
    w.tensors = {"q": _n(f"{prefix}.q", (B, S, Hq, D)), "k": _n(f"{prefix}.k", (B, S, Hk, D)),
                 "dq": _n(f"{prefix}.dq", (B, S, Hq, D)), "dk": _n(f"{prefix}.dk", (B, S, Hk, D))}
    return w


def swiglu(seed, shape, dtype, prefix="swiglu") -> Workload:
    n = int(np.prod(shape))
    w = Workload(f"{prefix}{list(shape)}", seed, dtype, {"shape": tuple(shape), "n": n})
    w.tensors = {"gate": _n(f"{prefix}.gate", shape), "up": _n(f"{prefix}.up", shape),
                 "dy": _n(f"{prefix}.dy", shape)}
    return w


def linear_ce(seed, T, H, V, ignore_frac, dtype, prefix="lce") -> Workload:
    w = Workload(f"{prefix}[T={T},H={H},V={V}]", seed, dtype,
                 {"T": T, "H": H, "V": V, "ignore_frac": ignore_frac, "ignore_index": IGNORE_INDEX})
    w.tensors = {"X": _n(f"{prefix}.X", (T, H)), "W": _n(f"{prefix}.W", (V, H), 0.0, 0.02),
                 "labels": Tensor(f"{prefix}.labels", (T,), "labels", float_dtype=False)}
    return w


# ---- the named configurations --------------------------------------------------------------

def tiny(dtype: str) -> dict:
    """Tiny decoder-op set: batch 2, seq 128, hidden 256, 4 heads x 64,
    intermediate 688, vocab 1024, eps 1e-6, RoPE theta 1e4, 5 % ignored labels,
    master seed 0."""
    B, S, H, NH, D, I, V = 2, 128, 256, 4, 64, 688, 1024
    T = B * S
    return {"rmsnorm": rmsnorm(0, T, H, 1e-6, dtype),
            "rope": rope(0, B, S, NH, NH, D, 1e4, dtype),
            "swiglu": swiglu(0, (T, I), dtype),
            "linear_ce": linear_ce(0, T, H, V, 0.05, dtype)}


def swiglu_llama(dtype: str = "bf16") -> Workload:
    """SwiGLU fwd+bwd on gate/up [4, 2048, 11008], master seed 1."""
    return swiglu(1, (4, 2048, 11008), dtype)


def rmsnorm_rope_llama3(dtype: str = "bf16") -> dict:
    """Llama-3-8B shapes, master seed 2: x [4*8192, 4096], eps 1e-5;
    Q [4, 8192, 32, 128], K [4, 8192, 8, 128], positions 0..8191, theta 5e5."""
    return {"rmsnorm": rmsnorm(2, 4 * 8192, 4096, 1e-5, dtype),
            "rope": rope(2, 4, 8192, 32, 8, 128, 5e5, dtype)}


def linear_ce_llama3(dtype: str = "bf16") -> Workload:
    """Fused linear-CE: 8192 tokens x hidden 4096, lm_head [128256, 4096],
    10 % ignored labels, mean reduction, master seed 3."""
    return linear_ce(3, 8192, 4096, 128256, 0.10, dtype)


QWEN_SEQS = (512, 2048, 8192, 32768)


def qwen_chain(S: int, dtype: str = "bf16") -> dict:
    """Qwen-7B-like layer chain at batch 1, seq S, master seed 4: RMSNorm
    [S, 4096] (eps 1e-6), RoPE Q/K [1, S, 32, 128] (theta 1e4), SwiGLU
    [S, 11008], linear-CE S x 4096 x 151936 with 10 % ignored labels."""
    return {"rmsnorm": rmsnorm(4, S, 4096, 1e-6, dtype),
            "rope": rope(4, 1, S, 32, 32, 128, 1e4, dtype),
            "swiglu": swiglu(4, (S, 11008), dtype),
            "linear_ce": linear_ce(4, S, 4096, 151936, 0.10, dtype)}
