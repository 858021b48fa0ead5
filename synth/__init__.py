"""Seeded synthetic inputs for the Muon bank step.

This module only draws random numbers and encodes them in the storage types
the step consumes (bf16 bit patterns, uint16 low-mantissa halves, fp32
buffers).  It holds none of the step's arithmetic, so both the CPU oracle and
the CUDA path can take their inputs from here without sharing method code.

Workloads follow the speedrun pages' parameter banks:
  * GPT-2-small attention bank, stored (10, 4*768, 768) and viewed with no
    copy as (40, 768, 768): slot k is layer k//4, projection k%4 in q,k,v,o
    ("Unified zero-copy optimizer" record, section 1.1 "parameter banks").
  * GPT-2-small MLP bank (12, 2, 3072, 768) viewed as (24, 3072, 768): slot k
    is layer k//2, matrix k%2 in fc,proj; one slot is padding that is still
    optimised ("dead slot", same section).
  * Gate parameters smear_gate (1, 12, 768) and attn_gate (10, 6, 12).
  * GPT-2-medium banks (96, 1024, 1024) and (48, 4096, 1024) (Track-2
    record 7, model dim 1024).
  * The successor banks of the same write-up's section 1.1: qk_bank
    (slots, 2*head_dim, model_dim), vo_bank (slots, hdim, model_dim) and
    mlp_bank (12, 2, 2816, 768) viewed as (24, 2816, 768), whose slot 7 of
    the (12, 2) view stays dead.  Slot counts are not printed; the reading
    here is 10 layers x 6 heads of 128 = 60 qk slots padded to 64, and
    10 layers x (v, o) = 20 vo slots of 768 x 768 padded to 24, the padding
    slots dead.

Seeds: initial state of bank b in workload w uses PCG64(1000*w + b); the
gradient of optimizer step k >= 1 uses PCG64(1000*w + 10*k + b).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class BankSpec:
    name: str
    batch: int
    rows: int
    cols: int
    grad_kind: str = "gauss"      # "gauss" (std grad_std) or "lowrank"
    grad_std: float = 1e-3
    dead_slots: tuple = ()        # slots whose grad, weight and mantissa are all zero

    @property
    def shape(self):
        return (self.batch, self.rows, self.cols)

    @property
    def numel(self):
        return self.batch * self.rows * self.cols


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    banks: tuple
    steps: int
    lr: float = 0.02
    wd: float = 0.01
    mu: float = 0.95
    ns_steps: int = 5
    normuon: bool = False
    beta2: float = 0.95
    notes: str = field(default="", compare=False)


ATTN_SMALL = BankSpec("attn", 40, 768, 768)
MLP_SMALL = BankSpec("mlp", 24, 3072, 768, dead_slots=(23,))

WORKLOADS = {
    1: Workload(1, "tiny 4x128x128", (BankSpec("tiny", 4, 128, 128, "gauss", 1.0),), steps=1),
    2: Workload(2, "gpt2-small attn bank 40x768x768", (ATTN_SMALL,), steps=10),
    3: Workload(3, "gpt2-small mlp bank 24x3072x768", (MLP_SMALL,), steps=10),
    4: Workload(4, "gpt2-small full muon step (attn+mlp+gates)", (
        BankSpec("attn", 40, 768, 768, "lowrank"),
        BankSpec("mlp", 24, 3072, 768, "lowrank", dead_slots=(23,)),
        BankSpec("smear_gate", 1, 12, 768, "lowrank"),
        BankSpec("attn_gate", 10, 6, 12, "lowrank"),
    ), steps=10),
    5: Workload(5, "gpt2-medium attn+mlp banks, NorMuon", (
        BankSpec("attn", 96, 1024, 1024, "lowrank"),
        BankSpec("mlp", 48, 4096, 1024, "lowrank"),
    ), steps=20, normuon=True),
    6: Workload(6, "successor banks qk 64x256x768 + vo 24x768x768 + mlp 24x2816x768", (
        BankSpec("qk", 64, 256, 768, "lowrank", dead_slots=(60, 61, 62, 63)),
        BankSpec("vo", 24, 768, 768, "lowrank", dead_slots=(20, 21, 22, 23)),
        BankSpec("mlp", 24, 2816, 768, "lowrank", dead_slots=(14, 15)),
    ), steps=3),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode float values as bf16 bit patterns (torch's round-to-nearest-even cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _lowrank_matrix(rng, rows, cols, rank_cap=16, noise=1e-4):
    r = min(rank_cap, rows, cols)
    u, _ = np.linalg.qr(rng.standard_normal((rows, r)))
    v, _ = np.linalg.qr(rng.standard_normal((cols, r)))
    sig = np.logspace(0.0, -3.0, r)
    g = (u * sig) @ v.T
    g += noise * rng.standard_normal((rows, cols))
    return g.astype(np.float32)


def draw_grad(rng, spec: BankSpec) -> np.ndarray:
    """bf16 bit patterns [batch, rows, cols] of one step's gradient."""
    out = np.empty(spec.shape, dtype=np.uint16)
    for k in range(spec.batch):
        if k in spec.dead_slots:
            out[k] = 0
            continue
        if spec.grad_kind == "lowrank":
            g = _lowrank_matrix(rng, spec.rows, spec.cols)
        else:
            g = rng.standard_normal((spec.rows, spec.cols), dtype=np.float32) * np.float32(spec.grad_std)
        out[k] = to_bf16_bits(g)
    return out


def draw_state(rng, spec: BankSpec):
    """Initial (weight bf16 bits, mantissa u16, momentum f32, normuon row state f32)."""
    std = spec.cols ** -0.5
    w = np.empty(spec.shape, dtype=np.uint16)
    mant = np.empty(spec.shape, dtype=np.uint16)
    for k in range(spec.batch):
        if k in spec.dead_slots:
            w[k] = 0
            mant[k] = 0
            continue
        w[k] = to_bf16_bits(rng.standard_normal((spec.rows, spec.cols), dtype=np.float32) * np.float32(std))
        mant[k] = rng.integers(0, 1 << 16, size=(spec.rows, spec.cols), dtype=np.uint16)
    mom = np.zeros(spec.shape, dtype=np.float32)
    row_v = np.zeros((spec.batch, spec.rows), dtype=np.float32)
    return w, mant, mom, row_v


def init_state(wid: int, bank_id: int):
    spec = WORKLOADS[wid].banks[bank_id]
    return draw_state(_rng(1000 * wid + bank_id), spec)


def grad(wid: int, step: int, bank_id: int) -> np.ndarray:
    assert step >= 1
    spec = WORKLOADS[wid].banks[bank_id]
    return draw_grad(_rng(1000 * wid + 10 * step + bank_id), spec)


def case(seed: int, batch: int, rows: int, cols: int, kind: str = "gauss", grad_std: float = 1.0,
         dead_slots=()):
    """A free-form bank for parity tests: (weight bits, mantissa, momentum, row state, grad bits).

    The momentum buffer is drawn non-zero (as after earlier steps) so the
    momentum arithmetic is exercised from the first call.
    """
    spec = BankSpec("case", batch, rows, cols, kind, grad_std, tuple(dead_slots))
    rng = _rng(seed)
    w, mant, _, row_v = draw_state(rng, spec)
    mom = (rng.standard_normal(spec.shape, dtype=np.float32) * np.float32(grad_std * 0.5))
    for k in spec.dead_slots:
        mom[k] = 0
    g = draw_grad(rng, spec)
    return w, mant, mom, row_v, g


def v_bits(seed: int, batch: int, rows: int, cols: int, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of an orthogonalised-update stand-in (for update-only tests)."""
    rng = _rng(seed)
    return to_bf16_bits(rng.standard_normal((batch, rows, cols), dtype=np.float32) * np.float32(scale))


def grid_grad_bits(seed: int, batch: int, rows: int, cols: int, kmax: int = 64,
                   quantum: float = 2.0 ** -10) -> np.ndarray:
    """bf16 bit patterns of k * quantum with integer k drawn uniformly from [-kmax, kmax].

    With kmax = 64, sums of up to three such values have |k| <= 192 < 2^8, so bf16
    holds them exactly: any summation order over up to three ranks gives the same
    bits (multi-rank gradient averaging tests).
    """
    rng = _rng(seed)
    k = rng.integers(-kmax, kmax + 1, size=(batch, rows, cols))
    return to_bf16_bits((k * quantum).astype(np.float32))
