"""The sharded step's library path on one GPU: a one-rank NCCL group.

With one rank the mean gradient is the gradient and the rank owns every slot,
so the sharded step (reduce-scatter, the library's step on the shard views,
all-gather) must give the same bits as muon_multi_step on the whole banks.
Multi-rank data movement is covered on CPU ranks (test_sharded_cpu.py); no
test here uses more than one GPU.
"""
import numpy as np
import pytest
import torch
import torch.distributed as dist

import synth
from gpu_util import f32, to_dev, u16

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


@pytest.fixture
def one_rank_group():
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1)
    yield dist.group.WORLD
    dist.destroy_process_group()


@pytest.mark.parametrize("normuon", [False, True])
def test_one_rank_sharded_step_is_the_plain_step(nss, one_rank_group, normuon):
    from newton_schulz_stacked_gb300.sharded import ShardedBank, ShardPlan, sharded_step
    shapes = [(3, 256, 384), (2, 384, 256), (4, 6, 12)]
    states = [synth.case(110 + i, *s) for i, s in enumerate(shapes)]
    plain = [nss.BankState(to_dev(w), to_dev(g), to_dev(mom), to_dev(mant), to_dev(row) if normuon else None)
             for (w, mant, mom, row, g) in states]
    sharded = [ShardedBank(ShardPlan(s[0], 1), 0, to_dev(w), to_dev(mom), to_dev(mant),
                           to_dev(row) if normuon else None)
               for s, (w, mant, mom, row, g) in zip(shapes, states)]
    grads = [to_dev(g) for (w, mant, mom, row, g) in states]
    for _ in range(2):
        nss.muon_multi_step(plain, LR, WD, MU, normuon=normuon, ns_steps=5)
        sharded_step(sharded, grads, LR, WD, MU, normuon=normuon, ns_steps=5, group=one_rank_group)
    torch.cuda.synchronize()
    assert nss.mb_sync_status() == 0
    for a, b in zip(plain, sharded):
        np.testing.assert_array_equal(u16(b.weights), u16(a.bank))
        np.testing.assert_array_equal(u16(b.mantissa), u16(a.mantissa))
        np.testing.assert_array_equal(f32(b.momentum), f32(a.momentum))
        if normuon:
            np.testing.assert_array_equal(f32(b.row_state), f32(a.row_state))
