"""Helpers for the GPU parity tests: move seeded host arrays to the device and
compare device results with the oracle."""
import numpy as np

import caat_inputs as ci


def torch():
    import torch as _t
    return _t


def dev(a: np.ndarray, dtype: str):
    """float32 host array -> CUDA tensor of dtype 'f32' or 'bf16' (bf16 = RNE words)."""
    T = torch()
    if dtype == "f32":
        return T.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    w = ci.bf16_words(a)
    return T.from_numpy(w.view(np.int16)).cuda().view(T.bfloat16)


def host_values(a: np.ndarray, dtype: str) -> np.ndarray:
    """The exact values the device holds for a float32 host array (f64)."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    return ci.words_to_f32(ci.bf16_words(a)).astype(np.float64)


def to_f64(t) -> np.ndarray:
    T = torch()
    if t.dtype == T.bfloat16:
        return t.detach().float().cpu().numpy().astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


def words(t) -> np.ndarray:
    """Raw bits of a device tensor (uint16 for bf16, uint32 for f32)."""
    T = torch()
    if t.dtype == T.bfloat16:
        return t.detach().contiguous().view(T.int16).cpu().numpy().view(np.uint16)
    return t.detach().contiguous().view(T.int32).cpu().numpy().view(np.uint32)


def rel_fro(got: np.ndarray, want: np.ndarray) -> float:
    num = np.linalg.norm((got - want).ravel())
    den = np.linalg.norm(want.ravel())
    return float(num / den) if den > 0 else float(num)


def sel_dev(S: np.ndarray):
    T = torch()
    return T.from_numpy(np.ascontiguousarray(S, dtype=np.int32)).cuda()


TOL = {"f32": 1e-5, "bf16": 1e-2}
