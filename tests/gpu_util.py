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

# Element-wise bounds, derived from the kernels' fp32 arithmetic against the oracle's one
# rounding of the fp64 result (unit roundoff U = 2^-24; the smallest fp32 subnormal as a floor).
F32_U = 2.0 ** -24
F32_TINY = 2.0 ** -149


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


def update_bound(w, ref, step):
    """Allowed |w_gpu - w_oracle| per element of the update.

    The kernel forms fl(fl(w * fl(1 - lr*wd)) + fl(fl(-lr*f) * v)) with lr and wd given as fp32
    (f = sqrt(max(1, rows/cols))); the oracle forms w (1 - lr wd) - lr f v in fp64 and rounds
    once.  With U = 2^-24 the kernel's result is within U |r| + 2 U |w| + 3 U |lr f v| of the
    exact value (the final sum; the decay factor and its product; lr's fp32 value, the factor's
    rounding and its product) and the oracle's within U |r|, so the two differ by at most
    2 U |r| + 2 U |w| + 3 U |lr f v| plus second-order terms, which a factor of 1.01 covers."""
    w = np.abs(np.asarray(w, np.float64))
    ref = np.abs(np.asarray(ref, np.float64))
    return 1.01 * F32_U * (2.0 * ref + 2.0 * w + 3.0 * np.abs(step)) + F32_TINY


def rowscale_rel(rows, cols):
    """Relative error bound of the kernels' fp32 NorMuon per-row factor: each row's sum of
    squares runs cols/32 terms per lane then a 5-level shuffle tree, the matrix-wide sums
    rows/256 terms per thread, a 5-level tree and 8 warp partials, and the factor a few
    roundings more (square roots, quotients, the state update); sums of non-negative terms lose
    at most one U per addition, and the factor halves the sums' errors through its roots.
    Twice the count of sequential roundings, plus 30, bounds it."""
    return 2.0 * F32_U * (cols / 32.0 + rows / 256.0 + 30.0)


def check_update(w0, m0, v_bits, w1, m1, lr, wd, rows, cols, mats=None, vhat=None, vhat_rel=None):
    """The GPU's fp32 weights against the oracle's, given the same v: every element within
    update_bound (asserted here), and the largest per-matrix relF, which is returned.

    With NorMuon (vhat given) the kernel scales v by its fp32 per-row factor, whose relative
    error (vhat_rel, by default rowscale_rel) enters the step term of the bound."""
    if vhat is not None and vhat_rel is None:
        vhat_rel = rowscale_rel(rows, cols)
    worst = 0.0
    for i, k in enumerate(range(w0.shape[0]) if mats is None else mats):
        v = vhat[i] if vhat is not None else O.bf16_bits_to_f64(v_bits[k])
        _, _, ref = O.weight_update(w0[k], m0[k], v, lr, wd, rows, cols)
        got = O.recombine_f32(w1[k], m1[k])
        w_in = O.recombine_f32(w0[k], m0[k]).astype(np.float64)
        step = O.effective_lr(lr, rows, cols) * np.asarray(v, np.float64)
        bound = update_bound(w_in, ref, step)
        if vhat is not None:
            bound = bound + vhat_rel * np.abs(step)
        err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
        bad = np.argwhere(~(err <= bound))
        assert bad.size == 0, (f"matrix {k}: {len(bad)} elements outside the update bound, first at "
                               f"{tuple(bad[0])}: got {got[tuple(bad[0])]!r}, oracle {ref[tuple(bad[0])]!r}")
        worst = max(worst, O.rel_frobenius(got, ref))
    return worst


def momentum_bound(b_ref, g_bits, b0):
    """Allowed |buf_gpu - buf_oracle| per element of the momentum buffer.

    The kernel forms fl(fl(1 - mu) * fl(g - b) + b) (one fused multiply-add) with mu given as
    fp32; the oracle forms b + (1 - mu)(g - b) in fp64 and rounds once.  The kernel is within
    U |buf| + U |g - b| (1 + (1 - mu)) of the exact value and the oracle within U |buf|, so they
    differ by at most 2 U |buf| + 2 U |g - b|, with 1.01 for second-order terms."""
    d = np.abs(O.bf16_bits_to_f64(g_bits) - np.asarray(b0, np.float64))
    return 1.01 * F32_U * (2.0 * np.abs(np.asarray(b_ref, np.float64)) + 2.0 * d) + F32_TINY


def check_momentum(b_gpu, g_bits, b0, mu):
    """The GPU's fp32 momentum buffer of one matrix against the oracle's: every element within
    momentum_bound (asserted here); returns the relF of the matrix."""
    b_ref, _, u_exact = O.momentum(g_bits, b0, mu)
    err = np.abs(np.asarray(b_gpu, np.float64) - b_ref.astype(np.float64))
    bad = np.argwhere(~(err <= momentum_bound(b_ref, g_bits, b0)))
    assert bad.size == 0, (f"{len(bad)} momentum elements outside the bound, first at {tuple(bad[0])}: "
                           f"got {b_gpu[tuple(bad[0])]!r}, oracle {b_ref[tuple(bad[0])]!r}")
    return O.rel_frobenius(b_gpu, b_ref), b_ref, u_exact
