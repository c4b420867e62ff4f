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


# Element-wise bound next to the relative Frobenius one:
#   |got - want| <= REL * |want| + TAU * rms(want)
# REL covers the one rounding of the result to its dtype (bf16: half an ulp is
# 2^-9 relative, fp32: 2^-24) with a factor-2 margin for the fp32 accumulation.
# TAU is an absolute floor at a fixed share of the result's scale, for elements
# near zero where a relative bound means nothing: the fp32 accumulation errors
# of a K-term sum stay far below it, while any misplaced, missing or extra term
# (a wrong tile, shard, rank, sign or channel) moves an element by O(rms).
# The backward's floor is twice the forward's: with the contiguous S the summed
# gradient of the S channels is rounded once to bf16 before it enters the GEMMs
# (2^-9 relative per term, random sign), which the float64 oracle never does.
# In the backward, rms is taken per column of the result: a column of dW belongs
# to one channel, and the channels of S carry the sum of the t ranks' gradients
# (about sqrt(t) times the scale of the others), so their rounding error is
# larger in the same proportion.  With a small S the matrix-wide rms would
# understate the scale of exactly those columns.
ELEM = {"bf16": (2.0 ** -8, 2.0 ** -7), "f32": (2.0 ** -18, 2.0 ** -16)}
ELEM_BWD = {"bf16": (2.0 ** -8, 2.0 ** -6), "f32": (2.0 ** -18, 2.0 ** -15)}


def check(got: np.ndarray, want: np.ndarray, dtype: str, bwd: bool = False, what="", spread=None):
    """Relative Frobenius error within TOL[dtype], and every element within the
    element-wise bound above (NaN or inf in `got` fails).

    spread: for results that sum the ranks' partials after rounding each to the
    dtype (the forward with an index list of S, whose S channels are the rank-order
    fold of the rounded partials), sum_r |Y_r| per element; each rounded partial
    adds up to half an ulp of itself, so REL * spread joins the bound there."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    e = rel_fro(got, want)
    assert e <= TOL[dtype], ("relative Frobenius", what, e)
    if want.size == 0:
        return
    rel, tau = (ELEM_BWD if bwd else ELEM)[dtype]
    if bwd and want.ndim == 2 and want.shape[0] > 0:
        rms = np.sqrt(np.mean(want * want, axis=0, keepdims=True))     # per column
    else:
        rms = float(np.sqrt(np.mean(want * want)))
    err = np.abs(got - want)
    bound = rel * np.abs(want) + tau * rms
    if spread is not None:
        bound = bound + rel * np.asarray(spread, dtype=np.float64)
    ok = err <= bound                      # NaN compares false: it fails
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError("element-wise bound: %s, %d of %d elements outside; first at %s: got %r, "
                             "want %r, bound %r" % (what, len(bad), want.size, i, got[i], want[i], bound[i]))
