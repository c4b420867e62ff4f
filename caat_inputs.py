"""Seeded synthetic inputs for the partial channel-reduce workloads.

This module is shared by the CUDA-path tests, the benchmark and the CPU oracle's
tests.  It holds none of the method's arithmetic: it draws seeded random tensors,
encodes them as bf16 words when a workload is bf16, and describes the workload
shapes (the 130M / TinyLlama-1.1B / Llama2-7B shaped row-parallel layers of
"Tensor-Parallelism with Partially Synchronized Activations", Experiments:
130M model with h = 768 and 12 layers, TinyLlama 1.1B, Llama2-7B, tensor-parallel
dimension 8, p = 0.5).

Seeds: X = 1000 + cfg, W = 2000 + cfg, upstream gradient = 3000 + cfg, channel
permutation = 4000 + cfg; the second layer of a config adds 100.
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np


def normal(seed: int, shape, std: float = 1.0) -> np.ndarray:
    """i.i.d. N(0, std^2) float32 from numpy's PCG64 default_rng(seed)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def bf16_words(a: np.ndarray) -> np.ndarray:
    """Encode float32 values as bf16 words (round to nearest even) -- input encoding."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def words_to_f32(w: np.ndarray) -> np.ndarray:
    """bf16 words back to float32 (exact)."""
    return (np.ascontiguousarray(w, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Layer:
    name: str      # "out_proj" (K = h) or "down_proj" (K = FFN width)
    K: int         # reduction width, split t ways


@dataclass
class Workload:
    name: str
    cfg: int                 # 1-based index into the list of workloads below
    t: int                   # emulated tensor-parallel ranks
    N: int                   # tokens (rows)
    h: int                   # hidden size = output channels
    layers: List[Layer] = field(default_factory=list)
    p: float = 0.5
    layout: int = 0          # 0 contiguous S, 1 seeded random S
    dtype: str = "bf16"
    backward: bool = True
    decode_N: Tuple[int, ...] = ()

    def seeds(self, layer_index: int = 0):
        off = self.cfg + 100 * layer_index
        return dict(X=1000 + off, W=2000 + off, G=3000 + off, perm=4000 + self.cfg)


WORKLOADS = {
    # standalone PCR, fp32, t=2 partial tensors [256, 768], p=0.5, S = first 384
    "pcr_f32_t2_256x768": Workload("pcr_f32_t2_256x768", 1, t=2, N=256, h=768,
                                   p=0.5, layout=0, dtype="f32", backward=False),
    # 130M: h=768, FFN 3072, t=8, N = 8 x 1024 tokens, fwd + bwd
    "130m": Workload("130m", 2, t=8, N=8192, h=768,
                     layers=[Layer("out_proj", 768), Layer("down_proj", 3072)]),
    # TinyLlama-1.1B: h=2048, SwiGLU FFN 5632, t=8, N = 4 x 2048 tokens, fwd + bwd
    "1.1b": Workload("1.1b", 3, t=8, N=8192, h=2048,
                     layers=[Layer("out_proj", 2048), Layer("down_proj", 5632)]),
    # Llama2-7B: h=4096, SwiGLU FFN 11008, t=8, prefill N = 4096, fwd only
    "7b_prefill": Workload("7b_prefill", 4, t=8, N=4096, h=4096,
                           layers=[Layer("out_proj", 4096), Layer("down_proj", 11008)],
                           backward=False, decode_N=(1, 8, 64)),
    # Llama2-7B decode step with 8 tokens in flight (weight streaming), fwd only
    "7b_decode8": Workload("7b_decode8", 4, t=8, N=8, h=4096,
                           layers=[Layer("out_proj", 4096), Layer("down_proj", 11008)],
                           backward=False),
    # Llama2-7B short prefill, 256 tokens (the few-token kernel in two token chunks)
    "7b_prefill256": Workload("7b_prefill256", 4, t=8, N=256, h=4096,
                              layers=[Layer("out_proj", 4096), Layer("down_proj", 11008)],
                              backward=False),
}


def layer_tensors(w: Workload, layer_index: int, N: int = None):
    """(X [N, K], W [K, h] logical, G [t, N, h]) float32 draws for one layer.

    X ~ N(0, 1), W ~ N(0, 0.02^2), G ~ N(0, 1).  With N smaller than the
    workload's, X and G are the leading rows of the full-size draw only when the
    caller asks for the full size; smaller N is its own draw (used for tests).
    """
    L = w.layers[layer_index]
    s = w.seeds(layer_index)
    N = w.N if N is None else N
    X = normal(s["X"], (N, L.K))
    W = normal(s["W"], (L.K, w.h), std=0.02)
    G = normal(s["G"], (w.t, N, w.h)) if w.backward else None
    return X, W, G
