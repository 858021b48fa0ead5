"""Step hyperparameters read from device memory, and CUDA-graph replay of the step.

muon_multi_step_dev reads each bank's {lr, wd, mu, beta2} from a device buffer
when the step runs ("Unified zero-copy optimizer" write-up, section 4: one fp32
device buffer of every bank's step scalars, uploaded once per step and read by
the CUDA graph on replay).  Its results must be bit-identical to the by-value
calls with the same values, including when a captured graph of the step is
replayed after the buffer has been rewritten.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import f32, to_dev, u16

pytestmark = pytest.mark.gpu

SHAPES = [(4, 256, 384), (3, 384, 256), (10, 6, 12)]
# per bank: lr, wd, mu, beta2
SCALARS = [(0.02, 0.01, 0.95, 0.95), (0.035, 0.0, 0.9, 0.9), (0.005, 0.1, 0.85, 0.99)]


@pytest.fixture(scope="module")
def nss():
    from newton_schulz_stacked_gb300.build import build_library
    build_library()
    import newton_schulz_stacked_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.load_library()
    return m


def _banks(nss, seed, normuon):
    out = []
    for i, shape in enumerate(SHAPES):
        w, mant, mom, row, g = synth.case(seed + i, *shape, kind="lowrank")
        out.append(nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), to_dev(row) if normuon else None))
    return out


def _clone(nss, banks):
    return [nss.BankState(b.bank.clone(), b.grad.clone(), b.momentum.clone(), b.mantissa.clone(),
                          b.row_state.clone() if b.row_state is not None else None) for b in banks]


def _by_value(nss, banks, scalars, normuon):
    for b, (lr, wd, mu, beta2) in zip(banks, scalars):
        if normuon:
            nss.normuon_bank_step(b.bank, b.grad, b.momentum, b.mantissa, b.row_state, lr, wd, mu, beta2, ns_steps=5)
        else:
            nss.muon_bank_step(b.bank, b.grad, b.momentum, b.mantissa, lr, wd, mu, ns_steps=5)


def _assert_same(a, b):
    for x, y in zip(a, b):
        assert np.array_equal(u16(x.bank), u16(y.bank))
        assert np.array_equal(u16(x.mantissa), u16(y.mantissa))
        assert np.array_equal(f32(x.momentum).view(np.uint32), f32(y.momentum).view(np.uint32))
        if x.row_state is not None:
            assert np.array_equal(f32(x.row_state).view(np.uint32), f32(y.row_state).view(np.uint32))


def _dev_scalars(scalars):
    return torch.tensor(np.asarray(scalars, dtype=np.float32).reshape(-1), device="cuda:0")


@pytest.mark.parametrize("normuon", [False, True])
def test_device_scalars_match_by_value_calls(nss, normuon):
    banks = _banks(nss, 4100, normuon)
    ref = _clone(nss, banks)
    nss.muon_multi_step_dev(banks, _dev_scalars(SCALARS), normuon=normuon, ns_steps=5)
    _by_value(nss, ref, SCALARS, normuon)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    _assert_same(banks, ref)


def test_graph_replay_reads_the_current_scalars(nss):
    banks = _banks(nss, 4200, False)
    ref = _clone(nss, banks)
    scal = _dev_scalars(SCALARS)
    ws = torch.empty(nss.mb_multi_workspace_bytes(banks, False), dtype=torch.uint8, device="cuda:0")
    # a first call outside the capture sets up the library's per-device state
    nss.muon_multi_step_dev(banks, scal, workspace=ws)
    _by_value(nss, ref, SCALARS, False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nss.muon_multi_step_dev(banks, scal, workspace=ws)
    torch.cuda.synchronize()
    # two replays, each after new gradients and new scalars are written into the captured buffers
    host = torch.empty(scal.numel(), dtype=torch.float32, pin_memory=True)
    for step in (2, 3):
        new = [(lr * step, wd, mu - 0.01 * step, b2) for lr, wd, mu, b2 in SCALARS]
        host.copy_(torch.tensor(np.asarray(new, dtype=np.float32).reshape(-1)))
        scal.copy_(host, non_blocking=True)
        for i, (b, r) in enumerate(zip(banks, ref)):
            gnew = to_dev(synth.case(4300 + 10 * step + i, *SHAPES[i], kind="lowrank")[4])
            b.grad.copy_(gnew)
            r.grad.copy_(gnew)
        g.replay()
        _by_value(nss, ref, new, False)
        torch.cuda.synchronize()
        assert nss.mb_sync_status() == 0
        _assert_same(banks, ref)


def test_bad_device_scalar_is_reported(nss):
    from newton_schulz_stacked_gb300 import _binding as b
    banks = _banks(nss, 4400, False)
    bad = [list(s) for s in SCALARS]
    bad[1][0] = float("nan")
    nss.muon_multi_step_dev(banks, _dev_scalars(bad))
    assert nss.mb_sync_status() == b.MB_ERR_ARG
    # the status is cleared, and a good call afterwards runs clean
    nss.muon_multi_step_dev(banks, _dev_scalars(SCALARS))
    assert nss.mb_sync_status() == 0
