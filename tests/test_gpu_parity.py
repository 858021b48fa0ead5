"""GPU parity of the C ABI against the fp64 oracle, stage by stage.

Every call goes through libmuonbank.so; the oracle gets the GPU's own
intermediate (u for Newton-Schulz, v for the update), as the tolerances are
stated "given identical input".
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import (MOMENTUM_TOL, check_momentum, NS_TOL, STATE_TOL, UPDATE_TOL, check_ns, check_update, f32, ns_tol, to_dev,
                      u16, u_bound, ws_matrix)

pytestmark = pytest.mark.gpu

LR, WD, MU = 0.02, 0.01, 0.95


@pytest.fixture(scope="module")
def nss():
    from newton_schulz_stacked_gb300.build import build_library
    build_library()
    import newton_schulz_stacked_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load_library()
    return m


def _case(seed, shape, kind="gauss", std=1e-3, dead=()):
    return synth.case(seed, *shape, kind=kind, grad_std=std, dead_slots=dead)


# ---------------------------------------------------------------- S1

@pytest.mark.parametrize("shape", [(4, 128, 128), (3, 200, 328), (2, 6, 12), (2, 13, 77), (1, 768, 3072), (5, 1, 1)])
def test_momentum(nss, shape):
    w, mant, mom, _, g = _case(11, shape, std=1.0)
    gt, mt = to_dev(g), to_dev(mom)
    ut = torch.empty_like(gt)
    nss.mb_momentum(gt, mt, ut, MU)
    torch.cuda.synchronize()
    b_gpu, u_gpu = f32(mt), O.bf16_bits_to_f64(u16(ut))
    for k in range(shape[0]):
        relf, b_ref, u_exact = check_momentum(b_gpu[k], g[k], mom[k], MU)
        assert relf <= MOMENTUM_TOL
        assert np.all(np.abs(u_gpu[k] - u_exact) <= u_bound(u_exact, g[k], b_ref))


# the ends of the momentum range: mu = 0 keeps only the gradient, mu = 1 only the buffer
@pytest.mark.parametrize("mu", [0.0, 0.5, 1.0])
def test_momentum_edge_coefficients(nss, mu):
    shape = (3, 200, 328)
    w, mant, mom, _, g = _case(16, shape, std=1.0)
    mom = np.random.default_rng(17).standard_normal(shape).astype(np.float32)
    gt, mt = to_dev(g), to_dev(mom)
    ut = torch.empty_like(gt)
    nss.mb_momentum(gt, mt, ut, mu)
    torch.cuda.synchronize()
    b_gpu, u_gpu = f32(mt), O.bf16_bits_to_f64(u16(ut))
    for k in range(shape[0]):
        relf, b_ref, u_exact = check_momentum(b_gpu[k], g[k], mom[k], mu)
        assert relf <= MOMENTUM_TOL
        assert np.all(np.abs(u_gpu[k] - u_exact) <= u_bound(u_exact, g[k], b_ref))
    if mu == 1.0:
        np.testing.assert_array_equal(b_gpu, mom)      # nothing of the gradient enters the buffer


# ---------------------------------------------------------------- S5

@pytest.mark.parametrize("shape", [(4, 128, 128), (3, 200, 328), (2, 6, 12), (2, 3072, 768), (1, 7, 9), (5, 1, 1)])
def test_update(nss, shape):
    w, mant, _, _, _ = _case(12, shape)
    v = synth.v_bits(13, *shape, scale=shape[1] ** -0.5)
    wt, mt = to_dev(w), to_dev(mant)
    nss.mb_update(wt, mt, to_dev(v), LR, WD)
    torch.cuda.synchronize()
    assert check_update(w, mant, v, u16(wt), u16(mt), LR, WD, shape[1], shape[2]) <= UPDATE_TOL


def test_update_bit_exact_cases(nss):
    shape = (2, 64, 200)
    w, mant, _, _, _ = _case(14, shape)
    v = synth.v_bits(15, *shape)
    # lr = 0: nothing moves
    wt, mt = to_dev(w), to_dev(mant)
    nss.mb_update(wt, mt, to_dev(v), 0.0, 0.3)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(u16(wt), w)
    np.testing.assert_array_equal(u16(mt), mant)
    # decay factor exactly 1/2 with v = 0: exact halving, the split must match bit for bit
    wt, mt = to_dev(w), to_dev(mant)
    nss.mb_update(wt, mt, to_dev(np.zeros_like(v)), 1.0, 0.5)
    torch.cuda.synchronize()
    hi, lo, _ = O.weight_update(w, mant, np.zeros(shape), 1.0, 0.5, shape[1], shape[2])
    np.testing.assert_array_equal(u16(wt), hi)
    np.testing.assert_array_equal(u16(mt), lo)


# ---------------------------------------------------------------- S2-S4

NS_SHAPES = [
    ((4, 128, 128), "gauss"), ((2, 256, 384), "gauss"), ((2, 384, 256), "gauss"),
    ((2, 200, 328), "gauss"), ((2, 328, 200), "gauss"), ((2, 65, 130), "gauss"), ((2, 130, 65), "gauss"),
    # three 128-blocks per side of A: the second 256-row pair tile has a partial even CTA and an
    # odd CTA wholly past the matrix; 520 columns end in an 8-column tile
    ((2, 300, 520), "gauss"), ((2, 520, 300), "lowrank"),
    ((2, 768, 768), "lowrank"), ((1, 768, 3072), "gauss"), ((2, 3072, 768), "lowrank"),
    ((3, 12, 768), "lowrank"), ((3, 6, 12), "lowrank"), ((2, 64, 64), "gauss"), ((2, 1, 40), "gauss"),
    ((5, 1, 1), "gauss"), ((2, 40, 1), "gauss"),
    # small min(rows, cols) whose fp32 iteration does not fit in shared memory: workspace path
    ((2, 40, 2000), "gauss"), ((2, 1500, 50), "lowrank"),
    # the largest here: 16 row blocks of A, hundreds of tiles per phase of one matrix
    ((1, 2048, 6144), "gauss"), ((1, 6144, 2048), "lowrank"),
]


@pytest.mark.parametrize("shape,kind", NS_SHAPES)
def test_newton_schulz(nss, shape, kind):
    rng = np.random.default_rng(sum(shape))
    if kind == "gauss":
        u = synth.to_bf16_bits(rng.standard_normal(shape))
    else:
        u = np.stack([synth.to_bf16_bits(synth._lowrank_matrix(rng, *shape[1:])) for _ in range(shape[0])])
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, vt, ns_steps=5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    errs = check_ns(u, u16(vt))
    assert errs.max() <= ns_tol(*shape[1:]), errs


# one matrix for every count T of 128-blocks per side of A from 2 to 17: T = 3 .. 16 take their
# GRAM and POLY tasks from the table covers of the block pairs, 2 and 17 the plain 2 x 2 tiling;
# the last block is ragged, and wide and tall slices alternate
@pytest.mark.parametrize("T", range(2, 18))
def test_newton_schulz_every_block_count(nss, T):
    m = 128 * T - 50
    shape = (1, m, m + 72) if T % 2 else (1, m + 72, m)
    u = synth.to_bf16_bits(np.random.default_rng(500 + T).standard_normal(shape))
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, vt, ns_steps=5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    errs = check_ns(u, u16(vt))
    assert errs.max() <= ns_tol(*shape[1:]), errs


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 8, 16])   # 16: the most one call accepts
@pytest.mark.parametrize("shape", [(2, 256, 384), (2, 384, 256), (2, 12, 40)])
def test_newton_schulz_steps(nss, steps, shape):
    rng = np.random.default_rng(steps * 7 + shape[1])
    u = synth.to_bf16_bits(rng.standard_normal(shape))
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, vt, ns_steps=steps)
    torch.cuda.synchronize()
    errs = check_ns(u, u16(vt), steps)
    assert errs.max() <= ns_tol(*shape[1:], steps=steps), errs


# a schedule of per-step coefficients: the pages' quintic, then the classical (15/8, -10/8, 3/8)
SCHEDULE = [(3.4445, -4.7750, 2.0315)] * 3 + [(1.875, -1.25, 0.375)] * 2


@pytest.mark.parametrize("shape", [(2, 256, 384), (2, 384, 256), (2, 12, 40), (1, 768, 3072)])
def test_newton_schulz_coefficient_schedule(nss, shape):
    rng = np.random.default_rng(sum(shape) + 1)
    u = synth.to_bf16_bits(rng.standard_normal(shape))
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz_coeffs(ut, vt, SCHEDULE)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    v = u16(vt)
    errs = np.array([O.rel_frobenius(O.bf16_bits_to_f64(v[k]),
                                     O.newton_schulz(O.bf16_bits_to_f64(u[k]), 5, SCHEDULE)) for k in range(shape[0])])
    assert errs.max() <= ns_tol(*shape[1:]), errs
    # the pages' quintic written out for every step is the plain call, bit for bit
    wt = torch.empty_like(ut)
    nss.mb_newton_schulz_coeffs(ut, wt, [(3.4445, -4.7750, 2.0315)] * 5)
    xt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, xt, ns_steps=5)
    torch.cuda.synchronize()
    assert np.array_equal(u16(wt), u16(xt))


# steps whose b or c is zero: b A alone (c = 0), c A^2 alone (b = 0) and a I alone (both zero)
DEGENERATE = [(3.4445, -4.7750, 2.0315), (1.5, -0.5, 0.0), (1.875, 0.0, -0.875), (1.0, 0.0, 0.0),
              (3.4445, -4.7750, 2.0315)]


@pytest.mark.parametrize("shape", [(2, 256, 384), (2, 384, 256), (3, 200, 328), (2, 12, 40)])
def test_newton_schulz_zero_coefficients(nss, shape):
    rng = np.random.default_rng(sum(shape) + 2)
    u = synth.to_bf16_bits(rng.standard_normal(shape))
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz_coeffs(ut, vt, DEGENERATE)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    v = u16(vt)
    errs = np.array([O.rel_frobenius(O.bf16_bits_to_f64(v[k]),
                                     O.newton_schulz(O.bf16_bits_to_f64(u[k]), 5, DEGENERATE)) for k in range(shape[0])])
    assert errs.max() <= ns_tol(*shape[1:]), errs


def test_newton_schulz_zero_and_scaled_input(nss):
    shape = (4, 256, 256)
    u = synth.to_bf16_bits(np.random.default_rng(3).standard_normal(shape))
    u[1] = 0
    # exact power-of-two rescales of slot 0, small enough that eps = 1e-7 stays below one fp32 ulp
    # of the norm (||u0|| ~ 256): then s*u is the same fp32 product and the outputs agree bit for bit
    u[2] = synth.to_bf16_bits(O.bf16_bits_to_f64(u[0]) * 2.0 ** -4)
    u[3] = synth.to_bf16_bits(O.bf16_bits_to_f64(u[0]) * 2.0 ** 6)
    ut = to_dev(u)
    vt = torch.empty_like(ut)
    nss.mb_newton_schulz(ut, vt, ns_steps=5)
    torch.cuda.synchronize()
    v = u16(vt)
    assert not np.any(v[1])
    # scale invariance: the power-of-two rescales change nothing after normalisation
    np.testing.assert_array_equal(v[2], v[0])
    np.testing.assert_array_equal(v[3], v[0])


# ---------------------------------------------------------------- whole step

def _run_step(nss, shape, seed, steps=1, ns_steps=5, kind="gauss", std=1e-3, dead=(), normuon=False):
    w, mant, mom, row, g = _case(seed, shape, kind, std, dead)
    t = dict(w=to_dev(w), m=to_dev(mant), b=to_dev(mom), g=to_dev(g), r=to_dev(row))
    for _ in range(steps):
        if normuon:
            ws = nss.normuon_bank_step(t["w"], t["g"], t["b"], t["m"], t["r"], LR, WD, MU, 0.95, ns_steps)
        else:
            ws = nss.muon_bank_step(t["w"], t["g"], t["b"], t["m"], LR, WD, MU, ns_steps)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    return (w, mant, mom, row, g), t, ws


@pytest.mark.parametrize("shape", [(4, 128, 128), (3, 328, 200), (2, 200, 328), (10, 6, 12), (1, 12, 768), (5, 1, 1)])
def test_full_step(nss, shape):
    (w, mant, mom, _, g), t, ws = _run_step(nss, shape, 21, std=1.0)
    B, R, C = shape
    u_off, v_off, pitch = nss.mb_workspace_views(shape)
    u_gpu = ws_matrix(ws, u_off, shape, pitch)
    v_gpu = ws_matrix(ws, v_off, shape, pitch)
    b_gpu = f32(t["b"])
    for k in range(B):
        relf, b_ref, u_exact = check_momentum(b_gpu[k], g[k], mom[k], MU)
        assert relf <= MOMENTUM_TOL
        assert np.all(np.abs(O.bf16_bits_to_f64(u_gpu[k]) - u_exact) <= u_bound(u_exact, g[k], b_ref))
    assert check_ns(u_gpu, v_gpu).max() <= ns_tol(R, C)
    assert check_update(w, mant, v_gpu, u16(t["w"]), u16(t["m"]), LR, WD, R, C) <= UPDATE_TOL


def test_dead_slot(nss):
    shape = (4, 384, 256)
    (w, mant, mom, _, g), t, ws = _run_step(nss, shape, 22, dead=(3,))
    u_off, v_off, pitch = nss.mb_workspace_views(shape)
    assert not np.any(ws_matrix(ws, v_off, shape, pitch)[3])
    assert not np.any(u16(t["w"])[3]) and not np.any(u16(t["m"])[3]) and not np.any(f32(t["b"])[3])


@pytest.mark.parametrize("shape", [(3, 256, 128), (2, 128, 384), (4, 6, 12), (2, 200, 328)])
def test_normuon_step(nss, shape):
    (w, mant, mom, row, g), t, ws = _run_step(nss, shape, 23, normuon=True)
    B, R, C = shape
    u_off, v_off, pitch = nss.mb_workspace_views(shape, normuon=True)
    v_gpu = ws_matrix(ws, v_off, shape, pitch)
    state = f32(t["r"])
    vhat = []
    for k in range(B):
        vh, s = O.normuon(O.bf16_bits_to_f64(v_gpu[k]), row[k], 0.95)
        assert O.rel_frobenius(state[k], s) <= STATE_TOL
        vhat.append(vh)
    assert check_update(w, mant, v_gpu, u16(t["w"]), u16(t["m"]), LR, WD, R, C, vhat=vhat) <= UPDATE_TOL


@pytest.mark.parametrize("beta2", [0.9, 0.0, 1.0])
def test_normuon_update_stage(nss, beta2):
    shape = (3, 300, 136)
    w, mant, _, row, _ = _case(24, shape)
    row = np.random.default_rng(25).uniform(0, 1e-3, row.shape).astype(np.float32)
    v = synth.v_bits(26, *shape, scale=0.05)
    v[1, 7] = 0   # a zero row
    wt, mt, rt = to_dev(w), to_dev(mant), to_dev(row)
    nss.mb_normuon_update(wt, mt, to_dev(v), rt, LR, WD, beta2)
    torch.cuda.synchronize()
    vhat = []
    for k in range(3):
        vh, s = O.normuon(O.bf16_bits_to_f64(v[k]), row[k], beta2)
        assert O.rel_frobenius(f32(rt)[k], s) <= STATE_TOL
        vhat.append(vh)
    assert check_update(w, mant, v, u16(wt), u16(mt), LR, WD, shape[1], shape[2], vhat=vhat) <= UPDATE_TOL


# the default step and the step with the update fused into the last Newton-Schulz epilogue
# (large banks whose columns are a multiple of 8, at least 3 steps; the separate update kernel
# for the rest) give the same bits as the stage calls
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("shape,ns_steps", [((3, 256, 384), 5), ((2, 384, 256), 5), ((2, 200, 328), 5),
                                            ((1, 768, 3072), 5), ((2, 3072, 768), 5), ((2, 256, 384), 3),
                                            ((2, 256, 384), 2), ((2, 200, 330), 5), ((3, 300, 520), 4)])
def test_step_equals_its_stage_calls(nss, shape, ns_steps, fuse):
    """A whole step gives the same bits as the same step run as separate stage calls (momentum,
    Newton-Schulz, the update kernel), the bank copy included."""
    w, mant, mom, _, g = _case(70 + ns_steps, shape, std=1e-3)
    a = nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), None, torch.zeros_like(to_dev(w)))
    nss.muon_multi_step([a], LR, WD, MU, ns_steps=ns_steps, flags=nss.MB_STEP_FUSE_UPDATE if fuse else 0)
    gt, mt, wt, at = to_dev(g), to_dev(mom), to_dev(w), to_dev(mant)
    ut, vt = torch.empty_like(gt), torch.empty_like(gt)
    nss.mb_momentum(gt, mt, ut, MU)
    nss.mb_newton_schulz(ut, vt, ns_steps=ns_steps)
    nss.mb_update(wt, at, vt, LR, WD)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    np.testing.assert_array_equal(f32(a.momentum), f32(mt))
    np.testing.assert_array_equal(u16(a.bank), u16(wt))
    np.testing.assert_array_equal(u16(a.mantissa), u16(at))
    np.testing.assert_array_equal(u16(a.bank_copy), u16(wt))


@pytest.mark.parametrize("fuse", [False, True])
def test_normuon_multi_step_mixed_banks(nss, fuse):
    """NorMuon over tensor-core banks and an fp32 gate bank in one call, with the tensor-core
    banks' row sums from their own pass or from the last Newton-Schulz epilogue (the gate bank's
    always from the pass, ragged 328-column rows included): every bank's row state and update
    against the oracle given the GPU's v."""
    shapes = [(3, 256, 384), (4, 6, 12), (2, 200, 328)]
    states = [_case(90 + i, s) for i, s in enumerate(shapes)]
    banks = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), to_dev(row))
             for (w, mant, mom, row, g) in states]
    ws = torch.empty(nss.mb_multi_workspace_bytes(banks, True), dtype=torch.uint8, device="cuda:0")
    nss.muon_multi_step(banks, LR, WD, MU, normuon=True, beta2=0.95, ns_steps=5, workspace=ws,
                        flags=nss.MB_STEP_FUSE_ROWSTATS if fuse else 0)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    off = 0
    for (w, mant, mom, row, g), b, shape in zip(states, banks, shapes):
        B, R, C = shape
        u_off, v_off, pitch = nss.mb_workspace_views(shape, normuon=True)
        v_gpu = ws_matrix(ws, off + v_off, shape, pitch)
        u_gpu = ws_matrix(ws, off + u_off, shape, pitch)
        off += nss.mb_workspace_bytes(shape, True)
        assert check_ns(u_gpu, v_gpu).max() <= ns_tol(R, C)
        state = f32(b.row_state)
        vhat = []
        for k in range(B):
            vh, st = O.normuon(O.bf16_bits_to_f64(v_gpu[k]), row[k], 0.95)
            assert O.rel_frobenius(state[k], st) <= STATE_TOL, (shape, k)
            vhat.append(vh)
        assert check_update(w, mant, v_gpu, u16(b.bank), u16(b.mantissa), LR, WD, R, C, vhat=vhat) <= UPDATE_TOL


def test_multi_step_equals_single_steps(nss):
    shapes = [(8, 256, 256), (6, 512, 256), (1, 12, 768), (10, 6, 12)]
    states = [_case(30 + i, s, dead=((5,) if i == 1 else ())) for i, s in enumerate(shapes)]
    multi, single = [], []
    for (w, mant, mom, row, g) in states:
        multi.append(nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)))
        single.append(nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)))
    for _ in range(2):
        nss.muon_multi_step(multi, LR, WD, MU, ns_steps=5)
        for b in single:
            nss.muon_bank_step(b.bank, b.grad, b.momentum, b.mantissa, LR, WD, MU, 5)
    torch.cuda.synchronize()
    for a, b in zip(multi, single):
        np.testing.assert_array_equal(u16(a.bank), u16(b.bank))
        np.testing.assert_array_equal(u16(a.mantissa), u16(b.mantissa))
        np.testing.assert_array_equal(f32(a.momentum), f32(b.momentum))


def test_more_large_banks_than_one_fused_launch_takes(nss):
    """Six large banks in one call run as two fused Newton-Schulz launches (four banks each at
    most), each with its own task counter; the result is bit-identical to six single-bank steps."""
    shapes = [(3, 256, 384), (2, 384, 256), (4, 200, 328), (1, 768, 768), (2, 128, 640), (3, 300, 520)]
    states = [_case(80 + i, s) for i, s in enumerate(shapes)]
    multi = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)) for (w, mant, mom, row, g) in states]
    single = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)) for (w, mant, mom, row, g) in states]
    for _ in range(2):
        nss.muon_multi_step(multi, LR, WD, MU, ns_steps=5)
        for b in single:
            nss.muon_bank_step(b.bank, b.grad, b.momentum, b.mantissa, LR, WD, MU, 5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    for a, b in zip(multi, single):
        np.testing.assert_array_equal(u16(a.bank), u16(b.bank))
        np.testing.assert_array_equal(u16(a.mantissa), u16(b.mantissa))
        np.testing.assert_array_equal(f32(a.momentum), f32(b.momentum))


@pytest.mark.parametrize("normuon", [False, True])
def test_bank_copy_receives_the_updated_bank(nss, normuon):
    """A bank's optional copy gets exactly the updated bank, on both update paths (columns a
    multiple of 8 and not), and the step is otherwise the same as without it."""
    shapes = [(4, 256, 384), (3, 200, 328), (10, 6, 12), (2, 7, 9)]
    states = [_case(60 + i, s) for i, s in enumerate(shapes)]
    with_copy, plain = [], []
    for (w, mant, mom, row, g) in states:
        rt = to_dev(row) if normuon else None
        with_copy.append(nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), rt, torch.zeros_like(to_dev(w))))
        plain.append(nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), rt.clone() if normuon else None))
    nss.muon_multi_step(with_copy, LR, WD, MU, normuon=normuon, ns_steps=5)
    nss.muon_multi_step(plain, LR, WD, MU, normuon=normuon, ns_steps=5)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    for a, b in zip(with_copy, plain):
        np.testing.assert_array_equal(u16(a.bank_copy), u16(a.bank))
        np.testing.assert_array_equal(u16(a.bank), u16(b.bank))
        np.testing.assert_array_equal(u16(a.mantissa), u16(b.mantissa))


def test_step_on_a_caller_stream(nss):
    """The step is ordered on the stream it is given, including the fp32 gate banks that run on the
    library's side stream (forked from and joined back to the caller's stream)."""
    shapes = [(4, 256, 384), (1, 12, 768), (10, 6, 12)]
    states = [_case(60 + i, s) for i, s in enumerate(shapes)]
    ref = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)) for (w, mant, mom, row, g) in states]
    nss.muon_multi_step(ref, LR, WD, MU, ns_steps=5)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        # the inputs are made on the caller's stream, and the step follows them there
        banks = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant))
                 for (w, mant, mom, row, g) in states]
        nss.muon_multi_step(banks, LR, WD, MU, ns_steps=5, stream=side)
        out = [(b.bank.clone(), b.mantissa.clone(), b.momentum.clone()) for b in banks]
    side.synchronize()
    assert nss.mb_sync_status(side) == 0
    for (bank, mant, mom), r in zip(out, ref):
        np.testing.assert_array_equal(u16(bank), u16(r.bank))
        np.testing.assert_array_equal(u16(mant), u16(r.mantissa))
        np.testing.assert_array_equal(f32(mom), f32(r.momentum))


def test_concurrent_host_threads(nss):
    """Two host threads step their own banks on their own streams at the same time (the C calls
    release the GIL); each result matches the same steps run one after the other."""
    import threading
    shapes = [[(4, 256, 384), (10, 6, 12)], [(3, 384, 256), (1, 12, 768)]]
    states = [[_case(80 + 10 * t + i, s) for i, s in enumerate(sh)] for t, sh in enumerate(shapes)]

    def banks_of(st):
        return [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant)) for (w, mant, mom, row, g) in st]

    ref = [banks_of(st) for st in states]
    for banks in ref:
        for _ in range(3):
            nss.muon_multi_step(banks, LR, WD, MU, ns_steps=5)
    torch.cuda.synchronize()
    out, errors = [None, None], []

    def run(t):
        try:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                banks = banks_of(states[t])
                for _ in range(3):
                    nss.muon_multi_step(banks, LR, WD, MU, ns_steps=5, stream=stream)
                out[t] = [(u16(b.bank), u16(b.mantissa)) for b in banks]
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert nss.mb_sync_status() == 0
    for t in range(2):
        for (bank, mant), r in zip(out[t], ref[t]):
            np.testing.assert_array_equal(bank, u16(r.bank))
            np.testing.assert_array_equal(mant, u16(r.mantissa))


def test_deterministic(nss):
    shape = (3, 512, 256)
    outs = []
    for _ in range(2):
        _, t, _ = _run_step(nss, shape, 40, steps=2)
        outs.append((u16(t["w"]), u16(t["m"]), f32(t["b"])))
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("shape", [(6, 256, 384), (5, 520, 300), (7, 6, 12)])
def test_slot_permutation_is_bit_exact(nss, shape):
    """Every slot of a bank is its own problem: the step on the slots permuted is the step's
    outputs permuted, bit for bit (no slot reads another's data, scale or completion counters)."""
    w, mant, mom, _, g = _case(44, shape, std=1.0)
    perm = np.random.default_rng(45).permutation(shape[0])
    while np.array_equal(perm, np.arange(shape[0])):
        perm = np.roll(perm, 1)

    def run(idx):
        t = [to_dev(np.ascontiguousarray(x[idx])) for x in (w, mom, mant)]
        for _ in range(2):
            nss.muon_bank_step(t[0], to_dev(np.ascontiguousarray(g[idx])), t[1], t[2], LR, WD, MU, 5)
        torch.cuda.synchronize()
        assert nss.mb_sync_status() == 0
        return [x.cpu().numpy() for x in t]

    plain = run(np.arange(shape[0]))
    permuted = run(perm)
    for a, b in zip(plain, permuted):
        np.testing.assert_array_equal(a[perm], b)


def test_resume_is_bit_exact(nss):
    shape = (2, 256, 384)
    w, mant, mom, _, g = _case(41, shape)
    run = lambda t, n: [nss.muon_bank_step(t[0], to_dev(g), t[1], t[2], LR, WD, MU, 5) for _ in range(n)]
    a = [to_dev(w), to_dev(mom), to_dev(mant)]
    run(a, 4)
    b = [to_dev(w), to_dev(mom), to_dev(mant)]
    run(b, 2)
    torch.cuda.synchronize()
    saved = [x.cpu() for x in b]                     # checkpoint, then restore into fresh buffers
    b = [x.to("cuda:0") for x in saved]
    run(b, 2)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.cpu(), y.cpu())


def test_guard_bands_untouched(nss):
    shape = (3, 200, 328)
    w, mant, mom, _, g = _case(42, shape)
    n = int(np.prod(shape))
    pad = 4096

    def guarded(a, fill):
        flat = np.full(n + 2 * pad, fill, dtype=a.dtype)
        flat[pad:pad + n] = a.reshape(-1)
        return to_dev(flat)

    bw, bm, bb, bg = guarded(w, 0x7E7E), guarded(mant, 0x5A5A), guarded(mom, np.float32(7.25)), guarded(g, 0x3C3C)
    view = lambda t: t[pad:pad + n].view(*shape)
    nss.muon_bank_step(view(bw), view(bg), view(bb), view(bm), LR, WD, MU, 5)
    torch.cuda.synchronize()
    for t, fill in ((bw, 0x7E7E), (bm, 0x5A5A), (bg, 0x3C3C)):
        h = u16(t)
        assert np.all(h[:pad] == fill) and np.all(h[pad + n:] == fill)
    h = f32(bb)
    assert np.all(h[:pad] == 7.25) and np.all(h[pad + n:] == 7.25)
    np.testing.assert_array_equal(u16(bg)[pad:pad + n], g.reshape(-1))   # grad is read-only


def test_device_timeout_is_reported_and_recoverable(nss):
    assert nss.mb_sync_status() == 0
    nss.mb_selftest_timeout(20000)                  # 20 ms bounded wait on a barrier nothing completes
    from newton_schulz_stacked_gb300 import _binding
    assert nss.mb_sync_status() == _binding.MB_ERR_TIMEOUT
    assert nss.mb_sync_status() == 0                # cleared after reading
    _run_step(nss, (2, 128, 128), 43)               # the context is still usable
