"""Shared helpers of the GPU parity tests (host-side marshalling only)."""
import numpy as np
import torch

import oracle as O

# Tolerances (per matrix, relative Frobenius):
NS_TOL = 2e-2          # bf16 Newton-Schulz output vs the fp64 iteration on the same input
NS_SMALL_TOL = 4e-3    # fp32 path for min(rows, cols) <= 64: bounded by the final bf16 rounding (2^-9)
UPDATE_TOL = 1e-6      # fp32 weight after the update, given the same NS output
MOMENTUM_TOL = 1e-6    # fp32 momentum buffer
STATE_TOL = 4e-6       # NorMuon fp32 row state: fp32 sums over up to a few thousand squares


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev())


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.exp2(e - 7)


def u_bound(u_exact, g_bits, buf_new):
    """Allowed |u_gpu - u|: one bf16 ulp of u plus the fp32 evaluation error of the two lerps,
    a few fp32 ulps of the operands (u can be tiny where the momentum term cancels g)."""
    g = np.abs(O.bf16_bits_to_f64(g_bits))
    return bf16_ulp(u_exact) + 2.0 ** -21 * (g + np.abs(np.asarray(buf_new, np.float64)))


def ws_matrix(ws: torch.Tensor, offset: int, shape, pitch: int) -> np.ndarray:
    """bf16 bits [batch, rows, cols] stored at `offset` with row pitch `pitch` inside a workspace."""
    B, R, C = shape
    host = ws[offset:offset + B * R * pitch * 2].cpu().numpy()
    return host.view(np.uint16).reshape(B, R, pitch)[:, :, :C].copy()


def ns_tol(rows, cols, steps=5):
    """relF bound of the GPU Newton-Schulz output against the fp64 iteration.

    The bound is stated for the method's 5 steps.  Each bf16-rounded step adds
    error (a bf16 emulation of the kernel's rounding gives about 1.0e-2 at 5
    steps, 1.9e-2 at 8, 3.4e-2 at 16 on Gaussian 256x384), so beyond 5 steps
    the bound grows by the same 4e-3 per step that gives 2e-2 at 5.
    """
    if min(rows, cols) <= 64:
        return NS_SMALL_TOL
    return NS_TOL if steps <= 5 else NS_TOL * steps / 5


def check_ns(u_bits, v_bits, steps=5, mats=None):
    """Per-matrix relF of the GPU output v against the fp64 iteration started from the GPU's u."""
    B, R, C = u_bits.shape
    errs = []
    for k in (range(B) if mats is None else mats):
        ref = O.newton_schulz(O.bf16_bits_to_f64(u_bits[k]), steps)
        errs.append(O.rel_frobenius(O.bf16_bits_to_f64(v_bits[k]), ref))
    return np.array(errs)


def check_update(w0, m0, v_bits, w1, m1, lr, wd, rows, cols, mats=None, vhat=None):
    """relF of the GPU's fp32 weight vs the oracle's, given the same v; returns the max."""
    worst = 0.0
    for i, k in enumerate(range(w0.shape[0]) if mats is None else mats):
        v = vhat[i] if vhat is not None else O.bf16_bits_to_f64(v_bits[k])
        _, _, ref = O.weight_update(w0[k], m0[k], v, lr, wd, rows, cols)
        got = O.recombine_f32(w1[k], m1[k])
        worst = max(worst, O.rel_frobenius(got, ref))
    return worst
