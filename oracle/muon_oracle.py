"""fp64 oracle of the Muon step over stacked parameter banks (test infrastructure only).

Sources, by page and section:
  [P1] "modded-nanogpt record: unified zero-copy optimizer and transposed LM head"
       (record 2026-01-18 UnifiedOptimizers), section 1.1 parameter banks.
  [P2] "Muon Custom Sizing" write-up (record 2025-09-23), section 2.3 (batched NS
       over the attention reshape) and section 4 (three-pass distributed step:
       momentum lerps, effective lr / weight decay).
  [P3] "GPT-2 Medium track record 7" write-up (2025-04-16), section 4.1
       (bf16 weight + uint16 mantissa update) and section 4.2 (quintic NS).
  [P4] "UNetDoubleLr" write-up (record 2024-11-10), optimizer section (NS
       coefficients, 5 steps, max(1, rows/cols)^0.5 scale, Nesterov momentum).

Readings taken where the pages are silent or garbled (each also listed in the
design notes):
  * The NS step printed in [P2] s2.3 is flattened and dimensionally wrong; the
    quintic form X <- a*X + b*A*X + c*A^2*X with A = X*X^T is used ([P3] s4.2
    calls it a fifth-order polynomial iteration).
  * Normalisation: once, before the iterations, by the Frobenius norm plus
    eps = 1e-7 (the pages say "by the spectral norm"; Frobenius bounds it).
  * Tall slices (rows > cols) iterate on the transpose; square ones do not.
  * Momentum buffer is fp32; buf is updated first, then u = lerp(g, buf, mu).
  * The mixed-precision split truncates: bf16 = high half, mantissa = low half.
  * NorMuon (named in [P1], formula absent): per-row EMA of mean(v^2) with
    beta2, rows scaled by 1/sqrt(max(s, 1e-10)), then the matrix is rescaled so
    its Frobenius norm equals that of v.
"""
from __future__ import annotations

import math

import numpy as np

# [P2] s2.3 and [P4]: quintic coefficients (a, b, c) and the step count.
NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315
NS_STEPS = 5
NS_EPS = 1e-7
NORMUON_FLOOR = 1e-10

_F64 = np.float64


# ----------------------------------------------------------------------------
# Storage encodings
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of bf16 bit patterns: a bf16 is the high half of an fp32 ([P3] s4.1)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(_F64)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values once to bf16 (round to nearest, ties to even).

    bf16 keeps 8 significant bits for normal numbers (exponent >= -126) and a
    fixed quantum of 2^-133 below that; values beyond the largest finite bf16
    after rounding become infinities.
    """
    x = np.asarray(x, dtype=_F64)
    out = np.empty(x.shape, dtype=_F64)
    ax = np.abs(x)
    tiny = ax < 2.0 ** -126
    # normal range: x = m * 2^e with 0.5 <= |m| < 1; keep 8 bits of m
    m, e = np.frexp(np.where(tiny, 1.0, x))
    out_norm = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    out_tiny = np.ldexp(np.rint(np.ldexp(x, 133)), -133)
    out = np.where(tiny, out_tiny, out_norm)
    max_bf16 = (2.0 - 2.0 ** -7) * 2.0 ** 127
    out = np.where(np.abs(out) > max_bf16, np.copysign(np.inf, out), out)
    out = np.where(np.isnan(x), np.nan, out)
    return (out.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def recombine_f32(w_bits: np.ndarray, mantissa: np.ndarray) -> np.ndarray:
    """fp32 weight from (bf16 bits << 16) | mantissa ([P3] s4.1)."""
    u = (np.asarray(w_bits, np.uint16).astype(np.uint32) << np.uint32(16)) | \
        np.asarray(mantissa, np.uint16).astype(np.uint32)
    return u.view(np.float32)


def split_f32(w32: np.ndarray):
    """Split fp32 values into (bf16 bits = high half, mantissa = low half) ([P3] s4.1)."""
    u = np.ascontiguousarray(w32, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16), (u & np.uint32(0xFFFF)).astype(np.uint16)


# ----------------------------------------------------------------------------
# S1 momentum ([P2] s4 pass two; Nesterov form named in [P4])
# ----------------------------------------------------------------------------

def momentum(g_bits: np.ndarray, buf: np.ndarray, mu: float):
    """One SGD-momentum step in the lerp form of [P2] s4.

    buf <- lerp(buf, g, 1 - mu); u <- lerp(g, buf_new, mu).
    Returns (buf_new rounded to fp32, u rounded to bf16 bits, u in fp64).
    """
    g = bf16_bits_to_f64(g_bits)
    b = np.asarray(buf, dtype=np.float32).astype(_F64)
    mu = float(mu)
    b_new = b + (1.0 - mu) * (g - b)
    u = g + mu * (b_new - g)
    return b_new.astype(np.float32), round_to_bf16_bits(u), u


# ----------------------------------------------------------------------------
# S2-S4 Frobenius normalisation and quintic Newton-Schulz ([P2] s2.3, [P3] s4.2, [P4])
# ----------------------------------------------------------------------------

def frobenius_scale(u: np.ndarray) -> float:
    """s = 1 / (||u||_F + eps): the normalisation applied once before the iterations."""
    return 1.0 / (math.sqrt(float(np.sum(np.square(np.asarray(u, _F64))))) + NS_EPS)


def step_coeffs(steps: int, coeffs) -> list:
    """(a, b, c) of each of `steps` steps: one triple for every step, or one triple per step
    (a schedule of per-iteration coefficients)."""
    c = np.asarray(coeffs, dtype=_F64)
    if c.shape == (3,):
        return [tuple(c)] * steps
    if c.shape != (steps, 3):
        raise ValueError(f"coefficients must be one (a, b, c) or one per step, got shape {c.shape}")
    return [tuple(r) for r in c]


def newton_schulz(u: np.ndarray, steps: int = NS_STEPS, coeffs=(NS_A, NS_B, NS_C)) -> np.ndarray:
    """Quintic Newton-Schulz orthogonalisation of one matrix, in fp64.

    X0 = u / (||u||_F + eps); a tall matrix iterates on its transpose so that
    A is min(r, c) square; step i forms A = X X^T, B = b_i A + c_i A A and
    X <- a_i X + B X; the result is returned in the input's orientation.
    `coeffs` is one (a, b, c) for every step, or one per step.
    """
    x = np.asarray(u, dtype=_F64) * frobenius_scale(u)
    tall = x.shape[0] > x.shape[1]
    if tall:
        x = x.T
    for a, b, c in step_coeffs(steps, coeffs):
        A = x @ x.T
        B = b * A + c * (A @ A)
        x = a * x + B @ x
    return x.T.copy() if tall else x


def quintic(x, steps: int = NS_STEPS, coeffs=(NS_A, NS_B, NS_C)):
    """The scalar maps p_i(x) = a_i x + b_i x^3 + c_i x^5 composed over `steps` steps."""
    x = np.asarray(x, dtype=_F64)
    for a, b, c in step_coeffs(steps, coeffs):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


# ----------------------------------------------------------------------------
# S5 mixed-precision update ([P3] s4.1; effective lr and decay from [P2] s4 and [P4])
# ----------------------------------------------------------------------------

def shape_factor(rows: int, cols: int) -> float:
    """max(1, rows/cols)^0.5 of the stored matrix ([P2] s4, [P4])."""
    return math.sqrt(max(1.0, rows / cols))


def effective_lr(lr: float, rows: int, cols: int) -> float:
    return float(lr) * shape_factor(rows, cols)


def effective_wd(lr: float, wd: float) -> float:
    """Decoupled decay amount lr * wd ([P2] s4, with the multipliers folded into wd)."""
    return float(lr) * float(wd)


def weight_update(w_bits: np.ndarray, mantissa: np.ndarray, v: np.ndarray, lr: float, wd: float,
                  rows: int, cols: int):
    """Rebuild fp32 from bf16 + mantissa, decay, subtract the scaled update, split back.

    The result is formed in fp64 and rounded once to fp32.  Returns
    (new bf16 bits, new mantissa, new fp32 weight).
    """
    w = recombine_f32(w_bits, mantissa).astype(_F64)
    r = w * (1.0 - effective_wd(lr, wd)) - effective_lr(lr, rows, cols) * np.asarray(v, _F64)
    r32 = r.astype(np.float32)
    hi, lo = split_f32(r32)
    return hi, lo, r32


# ----------------------------------------------------------------------------
# S6 NorMuon per-row second moment (named in [P1]; formula is the stated reading)
# ----------------------------------------------------------------------------

def normuon(v: np.ndarray, row_state: np.ndarray, beta2: float):
    """Per-row second-moment normalisation of one orthogonalised update (rows x cols).

    q_i = mean_j v_ij^2; s_i <- beta2 s_i + (1 - beta2) q_i;
    vhat_ij = v_ij / sqrt(max(s_i, 1e-10)); vhat <- vhat * ||v||_F / ||vhat||_F.
    Returns (vhat in fp64, new row state in fp64).
    """
    v = np.asarray(v, dtype=_F64)
    q = np.mean(v * v, axis=1)
    s = float(beta2) * np.asarray(row_state, dtype=_F64) + (1.0 - float(beta2)) * q
    vhat = v / np.sqrt(np.maximum(s, NORMUON_FLOOR))[:, None]
    n_v = math.sqrt(float(np.sum(v * v)))
    n_h = math.sqrt(float(np.sum(vhat * vhat)))
    vhat = vhat * (n_v / n_h) if n_h > 0.0 else np.zeros_like(vhat)
    return vhat, s


# ----------------------------------------------------------------------------
# Whole step over a bank ([P1] s1.1 banks; [P2] s4 step; [P3] s4.1 update)
# ----------------------------------------------------------------------------

def bank_step(w_bits, mantissa, buf, g_bits, lr, wd, mu, ns_steps=NS_STEPS,
              normuon_beta2=None, row_state=None, matrices=None):
    """One Muon step over a bank [batch, rows, cols]: every matrix independently.

    Returns a dict of per-stage results for the matrices listed in `matrices`
    (all when None): buf (fp32), u (bf16 bits), v (fp64 NS output), and the new
    weight bits / mantissa / fp32 weight; with NorMuon also the row state and
    the normalised update.
    """
    batch, rows, cols = np.shape(w_bits)
    idx = range(batch) if matrices is None else matrices
    out = {k: [] for k in ("index", "buf", "u", "v", "vhat", "row_state", "w_bits", "mantissa", "w32")}
    for k in idx:
        b_new, u_bits, _ = momentum(g_bits[k], buf[k], mu)
        v = newton_schulz(bf16_bits_to_f64(u_bits), ns_steps)
        upd = v
        if normuon_beta2 is not None:
            upd, s = normuon(v, row_state[k], normuon_beta2)
            out["row_state"].append(s)
            out["vhat"].append(upd)
        hi, lo, w32 = weight_update(w_bits[k], mantissa[k], upd, lr, wd, rows, cols)
        out["index"].append(k)
        out["buf"].append(b_new)
        out["u"].append(u_bits)
        out["v"].append(v)
        out["w_bits"].append(hi)
        out["mantissa"].append(lo)
        out["w32"].append(w32)
    return out


def rel_frobenius(x, ref) -> float:
    """||x - ref||_F / ||ref||_F (0 when both are zero)."""
    x = np.asarray(x, _F64)
    ref = np.asarray(ref, _F64)
    d = math.sqrt(float(np.sum((x - ref) ** 2)))
    n = math.sqrt(float(np.sum(ref ** 2)))
    if n == 0.0:
        return 0.0 if d == 0.0 else math.inf
    return d / n
