"""Shared test helpers: tolerance checks against the fp64 oracle."""

import numpy as np
import torch

from oracle import bf16 as ob

# Tolerances of the update step (fp32 kernels against the fp64 oracle):
#   master, m, v:     |x - x_ref| <= 2e-6 * max(|x_ref|, x_abs)
#   S, applied W:     |x - x_ref| <= 1e-4 * max(|x_ref|, x_abs)
#   bf16 weights:     at most 1 ulp (ordered bit distance) from RNE(x_ref)
# x_abs is the oracle's absolute-term magnitude (the same expression with
# every term replaced by its absolute value), which bounds rounding error
# where terms cancel.
TOL_STATE = 2e-6
TOL_LSP = 1e-4


def f64(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().double().cpu().numpy()


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_close(name, got, ref, mag, tol):
    got = f64(got)
    bound = tol * np.maximum(np.abs(ref), mag)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.flatnonzero(bad.ravel())[0]
        raise AssertionError(
            f"{name}: {bad.sum()} of {bad.size} outside tolerance; first at {i}: "
            f"got {got.ravel()[i]!r} ref {ref.ravel()[i]!r} bound {bound.ravel()[i]!r}")
    rel = float(np.max(err / np.maximum(np.abs(ref), 1e-300))) if err.size else 0.0
    return rel


def check_bf16(name, got_bits, ref_f64, max_ulp=1):
    d = ob.ulp_distance(got_bits, ob.bf16_bits(ref_f64))
    if d.size and d.max() > max_ulp:
        i = int(np.argmax(d))
        raise AssertionError(f"{name}: {int((d > max_ulp).sum())} elements beyond {max_ulp} ulp; "
                             f"worst {int(d.max())} at {i}")


HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def check_bf16_applied(name, got_bits, w_in, D, D_abs):
    """bf16 W after W -= D: within 1 ulp of RNE(W - D), or, where W and D
    cancel so that the bf16 spacing of the result is finer than the fp32
    accumulation error of D, within the applied-W bound
    TOL_LSP * (|W| + |D|_abs) of the exact result."""
    ref = w_in - D
    d = ob.ulp_distance(got_bits, ob.bf16_bits(ref))
    err = np.abs(ob.bits_to_f64(got_bits) - ref)
    ok = (d <= 1) | (err <= TOL_LSP * (np.abs(w_in) + D_abs))
    if not ok.all():
        i = int(np.flatnonzero(~ok.ravel())[0])
        raise AssertionError(f"{name}: {int((~ok).sum())} elements out; first at {i}: {int(d.ravel()[i])} ulp, "
                             f"err {err.ravel()[i]!r}")
