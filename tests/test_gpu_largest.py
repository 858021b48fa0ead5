"""Parity at the largest matrix the library accepts: 2^30 elements in one matrix.

At this size the fp64 oracle cannot run the iteration, so the inputs are chosen
to have a closed form.  Under the quintic iteration of "Muon Custom Sizing",
section 2.3, a diagonal X keeps A = X X^T, B = bA + cA^2 and aX + BX diagonal,
so each diagonal entry x follows the scalar map a x + b x^3 + c x^5 from its
normalised value, and every other entry stays exactly zero.  The element-wise
stages are checked against the oracle on a seeded sample of positions spread
over the whole matrix, plus every diagonal position.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import MOMENTUM_TOL, NS_TOL, UPDATE_TOL, check_momentum, check_update, to_dev, u16, u_bound, ws_matrix

pytestmark = pytest.mark.gpu

LR, WD, MU = 0.02, 0.01, 0.95
LARGEST = [(1, 1 << 15, 1 << 15), (1, 1 << 14, 1 << 16), (1, 1 << 16, 1 << 14)]


@pytest.fixture(scope="module")
def nss():
    from newton_schulz_stacked_gb300.build import build_library
    build_library()
    import newton_schulz_stacked_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load_library()
    return m


def _repeat_block(rng, n, length, lo, hi):
    """n values drawn from a seeded block of a prime length, repeated: they differ from their
    neighbours at every offset but multiples of that length, and 2^30 of them take a second."""
    return np.resize(rng.integers(lo, hi, size=length, dtype=np.uint16), n)


def _diagonal_values(rng, m, scale=1.0):
    """bf16 bits of m positive values spread over a factor of 20."""
    return synth.to_bf16_bits(scale * np.exp(rng.uniform(np.log(0.05), 0.0, m)))


def _check_diagonal_ns(u_diag_bits, v, m):
    """v (bf16 bits [rows, cols]) against the closed form of a diagonal input, then zero
    everywhere else (as a value: a zero may carry either sign)."""
    x = O.bf16_bits_to_f64(u_diag_bits)
    ref = O.quintic(x * O.frobenius_scale(x))
    idx = np.arange(m)
    got = O.bf16_bits_to_f64(v[idx, idx])
    err = O.rel_frobenius(got, ref)
    assert err <= NS_TOL, err
    v[idx, idx] = 0
    assert not np.any(v & np.uint16(0x7FFF))


@pytest.mark.parametrize("shape", LARGEST)
def test_newton_schulz_at_the_largest_matrix_size(nss, shape):
    _, R, C = shape
    m = min(R, C)
    rng = np.random.default_rng(R + 3 * C)
    d = _diagonal_values(rng, m)
    u = np.zeros(shape, dtype=np.uint16)
    idx = np.arange(m)
    u[0, idx, idx] = d
    ut = to_dev(u)
    del u
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, vt, ns_steps=5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    del ut
    v = u16(vt)[0]
    del vt
    _check_diagonal_ns(d, v, m)
    torch.cuda.empty_cache()


def test_full_step_at_the_largest_matrix_size(nss):
    """One muon_bank_step on a tall 65536 x 16384 matrix (shape factor 2, iterated as its
    transpose): momentum, Newton-Schulz and the update through the C ABI."""
    shape = (1, 1 << 16, 1 << 14)
    _, R, C = shape
    E = R * C
    rng = np.random.default_rng(2024)
    idx = np.arange(C)
    # weights: bf16 of either sign between 2^-11 and 2^-2; any low mantissa half
    w = _repeat_block(rng, E, 1_000_003, 0x3A00, 0x3E80)
    w |= _repeat_block(rng, E, 999_983, 0, 2) << np.uint16(15)
    mant = _repeat_block(rng, E, 1_000_033, 0, 1 << 16)
    # diagonal gradient and momentum: u, and with it the iteration, stay diagonal
    g = np.zeros((R, C), dtype=np.uint16)
    g[idx, idx] = _diagonal_values(rng, C, 1e-3)
    b0 = np.zeros((R, C), dtype=np.float32)
    b0[idx, idx] = (1e-3 * rng.standard_normal(C)).astype(np.float32)
    sample = np.unique(np.concatenate([rng.choice(E, size=1 << 20, replace=False), idx * C + idx]))
    w_s, mant_s, g_s, b0_s = w[sample], mant[sample], g.reshape(-1)[sample], b0.reshape(-1)[sample]

    bank, mt = to_dev(w.reshape(shape)), to_dev(mant.reshape(shape))
    grad, mom = to_dev(g.reshape(shape)), to_dev(b0.reshape(shape))
    del w, mant, g, b0
    ws = nss.muon_bank_step(bank, grad, mom, mt, LR, WD, MU, ns_steps=5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0

    st = torch.from_numpy(sample).to(bank.device)
    b1_s = mom.view(-1)[st].cpu().numpy()
    w1_s = u16(bank.view(-1)[st])
    m1_s = u16(mt.view(-1)[st])
    del bank, grad, mom, mt, st
    u_off, v_off, pitch = nss.mb_workspace_views(shape, False, 5)
    u = ws_matrix(ws, u_off, shape, pitch)[0]
    v = ws_matrix(ws, v_off, shape, pitch)[0]
    del ws
    torch.cuda.empty_cache()

    # S1 on the sample
    relf, b_ref, u_exact = check_momentum(b1_s, g_s, b0_s, MU)
    assert relf <= MOMENTUM_TOL
    u_s = u.reshape(-1)[sample]
    assert np.all(np.abs(O.bf16_bits_to_f64(u_s) - u_exact) <= u_bound(u_exact, g_s, b_ref))
    # S2-S4: the GPU's own u is diagonal, so v has the closed form
    u_diag = u[idx, idx].copy()
    u[idx, idx] = 0
    assert not np.any(u & np.uint16(0x7FFF))
    v_s = O.bf16_bits_to_f64(v.reshape(-1)[sample])
    _check_diagonal_ns(u_diag, v, C)
    # S5 on the sample, given the GPU's v
    assert check_update(w_s[None], mant_s[None], None, w1_s[None], m1_s[None], LR, WD, R, C,
                        vhat=[v_s], vhat_rel=0.0) <= UPDATE_TOL
