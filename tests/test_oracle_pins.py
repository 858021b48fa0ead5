"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test checks the oracle against a closed form, an invariant, a library
routine or brute force, chosen so that a plausible mistake (a dropped term, a
wrong sign, a transposed operand, a swapped lerp order, a rounding in place of
a truncation) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _orth(rng, n, k):
    q, _ = np.linalg.qr(rng.standard_normal((n, k)))
    return q


# ---------------------------------------------------------------- constants from the pages

def test_coefficients_are_the_pages():
    g = _gold("ns_coefficients.json")
    assert (O.NS_A, O.NS_B, O.NS_C) == (g["a"], g["b"], g["c"])
    assert O.NS_STEPS == g["steps"]


def test_workload_hyperparameters_are_the_pages_defaults():
    g = _gold("muon_defaults.json")
    for w in synth.WORKLOADS.values():
        assert (w.lr, w.wd, w.mu) == (g["lr"], g["weight_decay"], g["momentum"])


def test_bank_shapes_and_shape_factor():
    g = _gold("bank_shapes.json")
    assert synth.ATTN_SMALL.shape == tuple(g["attn"]["view"])
    assert synth.MLP_SMALL.shape == tuple(g["mlp"]["view"])
    assert O.shape_factor(*g["attn"]["view"][1:]) == g["attn"]["shape_factor"]
    assert O.shape_factor(*g["mlp"]["view"][1:]) == g["mlp"]["shape_factor"]
    # a wide matrix gets no boost (the factor uses rows/cols of the stored slice)
    assert O.shape_factor(768, 3072) == 1.0


def test_effective_lr_and_decay_of_the_pages_defaults():
    """With the pages' defaults, the MLP slices (shape factor 2) step at twice the learning rate
    and every slice decays by lr * wd = 2e-4 per step; an exactly representable case checks
    that the decay amount is a product, not a sum or a quotient."""
    g, shapes = _gold("muon_defaults.json"), _gold("bank_shapes.json")
    lr, wd = g["lr"], g["weight_decay"]
    assert O.effective_lr(lr, *shapes["mlp"]["view"][1:]) == pytest.approx(0.04, rel=1e-15)
    assert O.effective_lr(lr, *shapes["attn"]["view"][1:]) == lr
    assert O.effective_wd(lr, wd) == pytest.approx(2e-4, rel=1e-15)
    assert O.effective_wd(0.5, 0.25) == 0.125
    assert O.effective_lr(0.5, 4096, 1024) == 1.0      # sqrt(4) = 2, exact


def test_frobenius_scale_of_a_known_norm():
    """diag(3, 4) has Frobenius norm 5 (and spectral norm 4); the scale is 1 / (5 + eps), and a
    Gaussian matrix scaled by it has unit Frobenius norm to within eps relative."""
    assert O.frobenius_scale(np.diag([3.0, 4.0])) == pytest.approx(1.0 / (5.0 + 1e-7), rel=1e-15)
    assert O.frobenius_scale(np.zeros((3, 5))) == pytest.approx(1e7, rel=1e-15)
    u = np.random.default_rng(8).standard_normal((40, 70))
    n = np.linalg.norm(u * O.frobenius_scale(u))
    assert 1.0 - 1e-7 / np.linalg.norm(u) - 1e-15 <= n < 1.0


def test_step_coeffs_forms():
    """One triple repeats for every step; a schedule gives each step its own triple, in order;
    a schedule of the wrong length is refused."""
    one = (3.4445, -4.7750, 2.0315)
    assert O.step_coeffs(3, one) == [one] * 3
    sched = [(1.0, 2.0, 3.0), (4.0, 5.0, 6.0)]
    assert O.step_coeffs(2, sched) == sched
    with pytest.raises(ValueError):
        O.step_coeffs(3, sched)


def test_bank_view_slot_rule():
    # the stored attention bank (L, 4*d, d) viewed with no copy as (4L, d, d):
    # slot k must be layer k//4, projection k%4
    L, d = 3, 4
    stored = np.arange(L * 4 * d * d).reshape(L, 4 * d, d)
    view = stored.reshape(4 * L, d, d)
    assert np.shares_memory(stored, view)
    for k in range(4 * L):
        np.testing.assert_array_equal(view[k], stored[k // 4, (k % 4) * d:(k % 4 + 1) * d, :])
    mlp = np.arange(L * 2 * 6 * d).reshape(L, 2, 6, d)
    mv = mlp.reshape(2 * L, 6, d)
    for k in range(2 * L):
        np.testing.assert_array_equal(mv[k], mlp[k // 2, k % 2])


# ---------------------------------------------------------------- encodings vs library routines

def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000) * np.exp(rng.uniform(-85, 85, 20000)),
        rng.standard_normal(2000) * 2.0 ** -130,                    # bf16 subnormals
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895313892515355e38, 3.4e38, -3.4e38, 1e-45, np.inf, -np.inf]),
    ]).astype(np.float32)
    # exact ties in both directions
    base = rng.integers(0x3F00, 0x4F00, 1000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.round_to_bf16_bits(vals.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_is_single_rounding_from_f64():
    # 1 + 2^-8 + 2^-40 lies just above a bf16 tie: once-rounded it goes up to
    # 1 + 2^-7; a detour through fp32 would land on the tie and round to 1.0
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    got = O.bf16_bits_to_f64(O.round_to_bf16_bits(np.array([x])))[0]
    assert got == 1.0 + 2.0 ** -7


def test_recombine_matches_torch_bf16_value():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 1 << 16, 100000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]                        # finite patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = O.recombine_f32(bits, np.zeros_like(bits))
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.slow
def test_split_recombine_exhaustive():
    """Every fp32 bit pattern survives split -> recombine unchanged."""
    chunk = 1 << 26
    base = np.arange(chunk, dtype=np.uint32)
    for start in range(0, 1 << 32, chunk):
        u = base + np.uint32(start)
        hi, lo = O.split_f32(u.view(np.float32))
        back = O.recombine_f32(hi, lo).view(np.uint32)
        assert np.array_equal(back, u), hex(start)


def test_split_truncates_not_rounds():
    # low half 0xFFFF: rounding would carry into the bf16 half, truncation must not
    w = np.array([0x3F80FFFF, 0xBF80FFFF, 0x7F7FFFFF], dtype=np.uint32).view(np.float32)
    hi, lo = O.split_f32(w)
    np.testing.assert_array_equal(hi, [0x3F80, 0xBF80, 0x7F7F])
    np.testing.assert_array_equal(lo, [0xFFFF, 0xFFFF, 0xFFFF])


# ---------------------------------------------------------------- Newton-Schulz

@pytest.mark.parametrize("rows,cols", [(16, 16), (8, 24), (24, 8), (1, 5), (5, 1)])
def test_ns_spectral_closed_form(rows, cols):
    """For G = U diag(s) V^T, NS(G) = U diag(p^5(s / (||s||_2 + eps))) V^T."""
    rng = np.random.default_rng(rows * 100 + cols)
    k = min(rows, cols)
    U, V = _orth(rng, rows, k), _orth(rng, cols, k)
    s = np.concatenate([[2.0], np.exp(rng.uniform(-6, 0, k - 1))]) if k > 1 else np.array([0.7])
    G = (U * s) @ V.T
    expect = (U * O.quintic(s / (np.linalg.norm(s) + O.NS_EPS))) @ V.T
    got = O.newton_schulz(G)
    assert O.rel_frobenius(got, expect) < 1e-12


def test_ns_per_step_coefficients_closed_form():
    """A schedule of per-step (a, b, c): NS(G) = U diag(p_5 o ... o p_1(s / (||s||_2 + eps))) V^T,
    the matrix iteration against the scalar maps on the singular values."""
    rng = np.random.default_rng(77)
    sched = [(O.NS_A, O.NS_B, O.NS_C)] * 3 + [(1.875, -1.25, 0.375)] * 2
    for rows, cols in [(12, 20), (20, 12)]:
        k = min(rows, cols)
        U, V = _orth(rng, rows, k), _orth(rng, cols, k)
        s = np.exp(rng.uniform(-4, 0, k))
        G = (U * s) @ V.T
        expect = (U * O.quintic(s / (np.linalg.norm(s) + O.NS_EPS), steps=5, coeffs=sched)) @ V.T
        assert O.rel_frobenius(O.newton_schulz(G, steps=5, coeffs=sched), expect) < 1e-12
    # one triple for every step is the same schedule written out
    G = rng.standard_normal((9, 14))
    assert np.array_equal(O.newton_schulz(G, 4, [(O.NS_A, O.NS_B, O.NS_C)] * 4), O.newton_schulz(G, 4))
    with pytest.raises(ValueError):
        O.newton_schulz(G, 5, sched[:4])


def test_ns_classical_quintic_reaches_the_polar_factor():
    """The classical quintic (15/8, -10/8, 3/8) has p(1) = 1 and p'(1) = 0: iterated long enough
    from a well-conditioned matrix it reaches the polar factor U V^T of the SVD."""
    rng = np.random.default_rng(5)
    for shape in [(12, 8), (8, 12)]:
        G = rng.standard_normal(shape)
        Uf, _, Vt = np.linalg.svd(G, full_matrices=False)
        got = O.newton_schulz(G, steps=40, coeffs=(1.875, -1.25, 0.375))
        assert O.rel_frobenius(got, Uf @ Vt) < 1e-10


def test_ns_svd_brute_force_small():
    """U^T NS(G) V is diagonal and holds the scalar map of the normalised singular values."""
    rng = np.random.default_rng(5)
    for (r, c) in [(6, 6), (4, 9), (9, 4), (32, 48), (64, 64)]:
        G = rng.standard_normal((r, c))
        U, s, Vt = np.linalg.svd(G, full_matrices=False)
        M = U.T @ O.newton_schulz(G) @ Vt.T
        off = M - np.diag(np.diag(M))
        assert np.max(np.abs(off)) < 1e-12
        np.testing.assert_allclose(np.diag(M), O.quintic(s / (np.linalg.norm(s) + O.NS_EPS)),
                                   rtol=1e-11, atol=1e-13)
        # approximates the polar factor U V^T as a bounded quantity (the quintic does not converge to 1)
        assert O.rel_frobenius(O.newton_schulz(G), U @ Vt) < 0.5


def _band(threshold=5.2e-3):
    x0 = np.exp(np.linspace(math.log(threshold), 0.0, 200001))
    y = O.quintic(x0)
    return float(y.min()), float(y.max())


def test_quintic_band():
    """Normalised singular values >= 5.2e-3 end in about [0.68, 1.13] after 5 steps."""
    lo, hi = _band()
    assert 0.675 < lo < 0.685 and 1.125 < hi < 1.14
    rng = np.random.default_rng(7)
    G = rng.standard_normal((64, 256))
    s0 = np.linalg.svd(G, compute_uv=False) / np.linalg.norm(G)
    assert s0.min() >= 5.2e-3
    s = np.linalg.svd(O.newton_schulz(G), compute_uv=False)
    assert s.min() >= lo - 1e-9 and s.max() <= hi + 1e-9


def test_ns_invariants():
    rng = np.random.default_rng(9)
    G = rng.standard_normal((12, 20))
    # zero steps: the normalised input
    np.testing.assert_allclose(O.newton_schulz(G, steps=0), G / (np.linalg.norm(G) + O.NS_EPS), rtol=1e-15)
    # zero matrix stays zero (dead slot)
    assert not np.any(O.newton_schulz(np.zeros((7, 9))))
    # scale invariance, up to the eps in the normaliser (eps/||G|| ~ 6e-9 here)
    assert O.rel_frobenius(O.newton_schulz(37.5 * G), O.newton_schulz(G)) < 1e-7
    # transpose equivariance: exercises the tall branch
    assert O.rel_frobenius(O.newton_schulz(G.T), O.newton_schulz(G).T) < 1e-13
    # diagonal input -> scalar map entrywise
    d = np.array([3.0, -1.0, 0.5, 0.25, 0.0])
    D = np.diag(d)
    np.testing.assert_allclose(np.diag(O.newton_schulz(D)), O.quintic(d / (np.linalg.norm(d) + O.NS_EPS)),
                               rtol=1e-13, atol=0)
    # orthogonal Q (n x n) -> p^5(1/sqrt(n)) Q
    n = 10
    Q = _orth(rng, n, n)
    np.testing.assert_allclose(O.newton_schulz(Q), O.quintic(1.0 / (math.sqrt(n) + O.NS_EPS)) * Q,
                               rtol=1e-12, atol=1e-14)


def test_ns_eps_is_added_to_the_norm():
    # a matrix of Frobenius norm 1e-7: X0 = G / (1e-7 + 1e-7) = G / 2e-7
    G = np.diag([6e-8, 8e-8])
    np.testing.assert_allclose(O.newton_schulz(G, steps=0), G / 2e-7, rtol=1e-12)


# ---------------------------------------------------------------- momentum

def test_momentum_closed_form_constant_grad():
    """From zero state with a constant g: buf_k = (1 - mu^k) g, u_k = (1 - mu) g + mu buf_k."""
    mu = 0.95
    g_bits = synth.to_bf16_bits(np.array([[0.75, -1.5, 3.0, 2.0 ** -10]]))
    g = O.bf16_bits_to_f64(g_bits)
    buf = np.zeros(g.shape, np.float32)
    for k in range(1, 6):
        buf, u_bits, u = O.momentum(g_bits, buf, mu)
        np.testing.assert_allclose(buf, (1 - mu ** k) * g, rtol=3e-7)
        np.testing.assert_allclose(u, (1 - mu) * g + mu * (1 - mu ** k) * g, rtol=3e-7)
        np.testing.assert_array_equal(u_bits, O.round_to_bf16_bits(u))


def test_momentum_two_steps_nesterov_order():
    # buf1 = (1-mu) g1, buf2 = mu (1-mu) g1 + (1-mu) g2, u2 = (1-mu) g2 + mu buf2
    mu = 0.9
    g1 = synth.to_bf16_bits(np.array([1.0, 0.0]))
    g2 = synth.to_bf16_bits(np.array([0.0, 1.0]))
    b, _, _ = O.momentum(g1, np.zeros(2, np.float32), mu)
    b, _, u = O.momentum(g2, b, mu)
    np.testing.assert_allclose(b, [mu * (1 - mu), 1 - mu], rtol=1e-7)
    np.testing.assert_allclose(u, [mu * mu * (1 - mu), (1 - mu) + mu * (1 - mu)], rtol=1e-7)


# ---------------------------------------------------------------- update

def _state(seed, shape):
    rng = np.random.default_rng(seed)
    w = synth.to_bf16_bits(rng.standard_normal(shape) * 0.05)
    m = rng.integers(0, 1 << 16, shape, dtype=np.uint16)
    return w, m


def test_update_zero_lr_keeps_bits():
    w, m = _state(11, (8, 16))
    v = np.random.default_rng(12).standard_normal((8, 16))
    hi, lo, _ = O.weight_update(w, m, v, 0.0, 0.01, 8, 16)
    np.testing.assert_array_equal(hi, w)
    np.testing.assert_array_equal(lo, m)


def test_update_decay_only_and_linearity():
    rows, cols = 24, 8                      # tall: shape factor sqrt(3)
    w, m = _state(13, (rows, cols))
    v = np.random.default_rng(14).standard_normal((rows, cols))
    lr, wd = 0.02, 0.01
    w32 = O.recombine_f32(w, m).astype(np.float64)
    # v = 0: pure decoupled decay
    _, _, r0 = O.weight_update(w, m, np.zeros_like(v), lr, wd, rows, cols)
    np.testing.assert_array_equal(r0, (w32 * (1 - lr * wd)).astype(np.float32))
    # w = 0: pure scaled step with the shape factor of the stored slice
    z = np.zeros_like(w)
    _, _, r1 = O.weight_update(z, z, v, lr, wd, rows, cols)
    np.testing.assert_array_equal(r1, (-lr * math.sqrt(3.0) * v).astype(np.float32))
    # decay does not touch the update term; the step does not touch the decay
    _, _, r2 = O.weight_update(w, m, v, lr, wd, rows, cols)
    # (each of r0, r1, r2 is rounded once to fp32, so allow one ulp of each)
    slack = np.abs(np.spacing(r0)) + np.abs(np.spacing(r1)) + np.abs(np.spacing(r2))
    err = np.abs(r2.astype(np.float64) - (r0.astype(np.float64) + r1.astype(np.float64)))
    assert np.all(err <= slack)


def test_update_split_is_exact_given_fp32():
    w, m = _state(15, (4, 32))
    v = np.random.default_rng(16).standard_normal((4, 32))
    hi, lo, r32 = O.weight_update(w, m, v, 0.02, 0.01, 4, 32)
    np.testing.assert_array_equal(O.recombine_f32(hi, lo).view(np.uint32), r32.view(np.uint32))


# ---------------------------------------------------------------- NorMuon reading

def test_normuon_invariants():
    rng = np.random.default_rng(17)
    v = rng.standard_normal((12, 40))
    v[3] = 0.0
    vhat, s = O.normuon(v, np.zeros(12), 0.95)
    # Frobenius norm preserved
    assert abs(np.linalg.norm(vhat) - np.linalg.norm(v)) < 1e-12 * np.linalg.norm(v)
    # zero row stays zero
    assert not np.any(vhat[3])
    # first step from zero state: every non-zero row ends with the same norm
    rn = np.linalg.norm(np.delete(vhat, 3, axis=0), axis=1)
    np.testing.assert_allclose(rn, rn[0], rtol=1e-12)
    # state: s = (1 - beta2) * mean(v^2) per row
    np.testing.assert_allclose(s, 0.05 * np.mean(v * v, axis=1), rtol=1e-14)
    # rows with equal RMS pass through unchanged, whatever the state
    e = rng.standard_normal((5, 30))
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    out, _ = O.normuon(e, np.full(5, 0.3), 0.95)
    np.testing.assert_allclose(out, e, rtol=1e-12, atol=1e-15)


def test_normuon_state_constant_rows():
    # constant per-row second moment q: s_k = (1 - beta2^k) q
    v = np.tile(np.array([[2.0], [0.5]]), (1, 8))
    s = np.zeros(2)
    for k in range(1, 5):
        _, s = O.normuon(v, s, 0.9)
        np.testing.assert_allclose(s, (1 - 0.9 ** k) * np.array([4.0, 0.25]), rtol=1e-13)


# ---------------------------------------------------------------- whole step

def test_dead_slot_only_decays():
    w, m = _state(19, (2, 8, 8))
    w[1] = 0
    m[1] = 0
    g = synth.to_bf16_bits(np.random.default_rng(20).standard_normal((2, 8, 8)))
    g[1] = 0
    buf = np.zeros((2, 8, 8), np.float32)
    out = O.bank_step(w, m, buf, g, 0.02, 0.01, 0.95)
    assert not np.any(out["v"][1]) and not np.any(out["w_bits"][1]) and not np.any(out["mantissa"][1])
    # a live slot with a zero gradient still decays
    w2, m2 = _state(21, (1, 8, 8))
    out2 = O.bank_step(w2, m2, np.zeros((1, 8, 8), np.float32), np.zeros((1, 8, 8), np.uint16),
                       0.02, 0.01, 0.95)
    expect = (O.recombine_f32(w2[0], m2[0]).astype(np.float64) * (1 - 0.02 * 0.01)).astype(np.float32)
    np.testing.assert_array_equal(out2["w32"][0], expect)


def test_bank_matrices_are_independent():
    rng = np.random.default_rng(23)
    w, m = _state(24, (3, 6, 10))
    g = synth.to_bf16_bits(rng.standard_normal((3, 6, 10)))
    buf = (rng.standard_normal((3, 6, 10)) * 0.1).astype(np.float32)
    full = O.bank_step(w, m, buf, g, 0.02, 0.01, 0.95)
    perm = [2, 0, 1]
    pm = O.bank_step(w[perm], m[perm], buf[perm], g[perm], 0.02, 0.01, 0.95)
    for j, k in enumerate(perm):
        np.testing.assert_array_equal(pm["w_bits"][j], full["w_bits"][k])
        np.testing.assert_array_equal(pm["mantissa"][j], full["mantissa"][k])


def test_bank_step_diagonal_closed_form():
    """One whole step on 8 x 2 (tall) slices with a diagonal gradient and a diagonal momentum
    buffer, each holding one of the two diagonal entries: the step's result follows from the
    scalars alone.

    mu = 1/2 gives buf = (1/2, 1/2) and u = (3/4, 1/4) on the diagonal, exactly; the quintic
    of the pages maps each normalised singular value u_i / (||u||_F + 1e-7) through its five
    steps; the update subtracts lr * sqrt(8 / 2) * v from the decayed weight.  Feeding g or the
    buffer to Newton-Schulz instead of u, dropping the shape factor, the decay or the sign of
    the step each changes the result far beyond fp32 rounding."""
    coef = _gold("ns_coefficients.json")
    a, b, c, steps = coef["a"], coef["b"], coef["c"], coef["steps"]
    lr, wd, mu = 0.02, 0.01, 0.5
    shape = (2, 8, 2)
    g = np.zeros(shape, np.uint16)
    buf = np.zeros(shape, np.float32)
    g[:, 0, 0] = synth.to_bf16_bits(np.array(1.0))
    buf[:, 1, 1] = 1.0
    w = np.zeros(shape, np.uint16)
    m = np.zeros(shape, np.uint16)
    w[1] = synth.to_bf16_bits(np.ones((8, 2)))           # slice 1 starts at w = 1 everywhere, slice 0 at 0
    out = O.bank_step(w, m, buf, g, lr, wd, mu)

    u_diag = (0.75, 0.25)
    norm = math.sqrt(0.75 ** 2 + 0.25 ** 2) + 1e-7
    v_diag = []
    for ui in u_diag:
        x = ui / norm
        for _ in range(steps):
            x = a * x + b * x ** 3 + c * x ** 5
        v_diag.append(x)
    eff_lr = lr * 2.0                                   # sqrt(max(1, 8 / 2))
    for k in range(2):
        buf_expect = np.zeros((8, 2), np.float32)
        buf_expect[0, 0] = buf_expect[1, 1] = 0.5
        np.testing.assert_array_equal(out["buf"][k], buf_expect)
        u_vals = O.bf16_bits_to_f64(out["u"][k])
        np.testing.assert_array_equal(u_vals[[0, 1], [0, 1]], u_diag)
        assert np.count_nonzero(u_vals) == 2
        v_expect = np.zeros((8, 2))
        v_expect[0, 0], v_expect[1, 1] = v_diag
        np.testing.assert_allclose(out["v"][k], v_expect, rtol=1e-12, atol=1e-15)
        w0 = 1.0 if k == 1 else 0.0
        w_expect = (w0 * (1.0 - lr * wd) - eff_lr * v_expect).astype(np.float32)
        np.testing.assert_allclose(out["w32"][k], w_expect, rtol=2.0 ** -23, atol=0)
        hi, lo = O.split_f32(w_expect)
        np.testing.assert_array_equal(out["w_bits"][k], hi)
        np.testing.assert_array_equal(out["mantissa"][k], lo)


# ---------------------------------------------------------------- the parity comparator

def test_rel_frobenius_known_values():
    """||x - ref||_F / ||ref||_F on cases whose value is exact in binary floating point, chosen
    so that a dropped square root, a division by ||ref||^2 or by ||x||, a norm over one axis
    only, or a comparator that returns 0 gives another value."""
    eye = np.eye(4)
    assert O.rel_frobenius(eye, 2.0 * eye) == 0.5             # ||I|| / ||2I|| = 2 / 4
    assert O.rel_frobenius(2.0 * eye, eye) == 1.0             # ||I|| / ||I||
    assert O.rel_frobenius([3.0, 0.0], [0.0, 4.0]) == 1.25    # ||(3, -4)|| / 4 = 5 / 4
    ref = np.ones((4, 4))
    assert O.rel_frobenius(-ref, ref) == 2.0                  # a sign flip is reported as large
    x = ref.copy()
    x[3, 3] += 3.0
    assert O.rel_frobenius(x, ref) == 0.75                    # one element of 16: 3 / 4
    x = ref.copy()
    x[0, :] += 1.0
    assert O.rel_frobenius(x, ref) == 0.5                     # a whole row: 2 / 4
    assert O.rel_frobenius(ref, ref) == 0.0
    assert O.rel_frobenius(np.zeros((2, 3)), np.zeros((2, 3))) == 0.0
    assert O.rel_frobenius(np.eye(2), np.zeros((2, 2))) == math.inf
    # it compares values, not bit patterns: -0 equals +0
    assert O.rel_frobenius(np.array([-0.0, 1.0]), np.array([0.0, 1.0])) == 0.0
