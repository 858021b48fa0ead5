"""The sharded data-parallel step's plan and data movement on gloo CPU ranks (no GPU).

Each rank runs the local part of the step through a stand-in that applies the
fp64 oracle's whole step to its slots (the library's CUDA path needs a GPU);
everything else is the product code: the slot plan, the averaging
reduce-scatter of bf16 gradients and the all-gather of bf16 weights.  After two
steps every rank's weights must equal, bit for bit, the oracle's single-rank
step over the whole bank fed with the mean of the ranks' gradients, and each
rank's momentum and mantissa must be the oracle's for its slots.

Two ranks draw Gaussian gradients (a two-term bf16 sum is the same in either
order).  Three ranks draw gradients on a grid of 2^-10 whose sums are exact in
bf16, so the reduction's order cannot change the mean; there the banks split
unevenly and the last rank owns one live slot and one padding slot of the
first bank and only padding of the second.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from newton_schulz_stacked_gb300.sharded import ShardPlan  # noqa: E402

LR, WD, MU, BETA2 = 0.02, 0.01, 0.95, 0.95
# (batch, rows, cols): an odd square bank (one padding slot on two ranks), a tall bank
BANKS = [(5, 16, 16), (4, 24, 8)]


def test_plan_splits_the_leading_dimension():
    # the pages' split of the GPT-2-small banks over 8 ranks: 5 attention and 3 MLP slots each
    assert ShardPlan(40, 8).per == 5 and ShardPlan(24, 8).per == 3
    p = ShardPlan(5, 2)
    assert (p.per, p.padded) == (3, 6)
    assert p.owned(0) == (0, 3) and p.owned(1) == (3, 6)
    assert p.live(0) == (0, 3) and p.live(1) == (3, 5)
    assert ShardPlan(1, 4).live(3) == (3, 3)            # a rank may own only padding
    with pytest.raises(ValueError):
        p.owned(2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _initial(shape, seed):
    import synth
    w, mant, mom, row, _ = synth.case(seed, *shape, grad_std=1.0)
    return w, mant, mom, row


def _grad(shape, step, rank, world):
    import synth
    if world == 2:
        return synth.case(1000 + 10 * step + rank, *shape, grad_std=1e-2)[4]
    return synth.grid_grad_bits(2000 + 10 * step + rank, *shape)


def _oracle_local_step(banks, grads, lr, wd, mu, normuon, beta2, ns_steps, workspace):
    """Stand-in for the library's local step on CPU ranks: the oracle's whole step on each slot."""
    import oracle as O
    for b, g in zip(banks, grads):
        w = b.shard.numpy().view(np.uint16)
        m = b.mantissa.numpy().view(np.uint16)
        mom = b.momentum.numpy()
        gb = g.contiguous().view(torch.int16).numpy().view(np.uint16)
        out = O.bank_step(w, m, mom, gb, lr, wd, mu, ns_steps,
                          normuon_beta2=beta2 if normuon else None,
                          row_state=b.row_state.numpy() if normuon else None)
        for k in range(w.shape[0]):
            w[k] = out["w_bits"][k]
            m[k] = out["mantissa"][k]
            mom[k] = out["buf"][k]
            if normuon:
                b.row_state.numpy()[k] = out["row_state"][k].astype(np.float32)
    return None


def _worker(rank, world, port, normuon, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from newton_schulz_stacked_gb300.sharded import ShardedBank, ShardPlan, sharded_step
        banks = []
        for i, shape in enumerate(BANKS):
            plan = ShardPlan(shape[0], world)
            w, mant, mom, row = _initial(shape, 50 + i)
            pad = plan.padded - shape[0]
            wfull = np.concatenate([w, np.zeros((pad,) + shape[1:], np.uint16)])
            mfull = np.concatenate([mant, np.zeros((pad,) + shape[1:], np.uint16)])
            bfull = np.concatenate([mom, np.zeros((pad,) + shape[1:], np.float32)])
            rfull = np.concatenate([row, np.zeros((pad, shape[1]), np.float32)])
            lo, hi = plan.owned(rank)
            banks.append(ShardedBank(plan, rank, torch.from_numpy(wfull.view(np.int16).copy()),
                                     torch.from_numpy(bfull[lo:hi].copy()),
                                     torch.from_numpy(mfull[lo:hi].view(np.int16).copy()),
                                     torch.from_numpy(rfull[lo:hi].copy()) if normuon else None))
        for step in (1, 2):
            grads = []
            for i, shape in enumerate(BANKS):
                pad = banks[i].plan.padded - shape[0]
                g = np.concatenate([_grad(shape, step, rank, world), np.zeros((pad,) + shape[1:], np.uint16)])
                grads.append(torch.from_numpy(g.view(np.int16).copy()))
            sharded_step(banks, grads, LR, WD, MU, normuon=normuon, beta2=BETA2,
                         local_step=_oracle_local_step)
        q.put((rank, [(b.weights.numpy().view(np.uint16).copy(), b.momentum.numpy().copy(),
                       b.mantissa.numpy().view(np.uint16).copy(),
                       b.row_state.numpy().copy() if normuon else None) for b in banks]))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def _expected(world, normuon):
    """The oracle's single-rank steps over each whole bank, fed with the ranks' mean gradient:
    the bf16 sum of the ranks' bf16 gradients (one rounding for two ranks, exact on the grid
    for three), divided by the world size in bf16."""
    import oracle as O
    out = []
    for i, shape in enumerate(BANKS):
        w, mant, mom, row = _initial(shape, 50 + i)
        w, mant, mom, row = w.copy(), mant.copy(), mom.copy(), row.copy()
        for step in (1, 2):
            gs = [torch.from_numpy(_grad(shape, step, r, world).view(np.int16)).view(torch.bfloat16) for r in range(world)]
            total = gs[0].clone()
            for g in gs[1:]:
                total = total + g
            mean = (total / world).view(torch.int16).numpy().view(np.uint16)
            res = O.bank_step(w, mant, mom, mean, LR, WD, MU, normuon_beta2=BETA2 if normuon else None,
                              row_state=row if normuon else None)
            w = np.stack(res["w_bits"])
            mant = np.stack(res["mantissa"])
            mom = np.stack(res["buf"])
            if normuon:
                row = np.stack(res["row_state"]).astype(np.float32)
        out.append((w, mant, mom, row))
    return out


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("normuon", [False, True])
def test_ranks_match_the_single_rank_step(world, normuon):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, normuon, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = _expected(world, normuon)
    for i, shape in enumerate(BANKS):
        plan = ShardPlan(shape[0], world)
        w_ref, m_ref, b_ref, r_ref = expect[i]
        for rank in range(world):
            w, mom, mant, row = got[rank][i]
            np.testing.assert_array_equal(w[:shape[0]], w_ref)          # every rank holds the whole bank
            assert not np.any(w[shape[0]:])                             # padding slots stay zero
            lo, hi = plan.live(rank)
            n = hi - lo
            np.testing.assert_array_equal(mom[:n], b_ref[lo:hi])        # state only for the owned slots
            np.testing.assert_array_equal(mant[:n], m_ref[lo:hi])
            assert not np.any(mom[n:]) and not np.any(mant[n:])
            if normuon:
                np.testing.assert_array_equal(row[:n], r_ref[lo:hi])
