"""The allocation-free Newton-Schulz entry point, checked against the workspace one.

Some callers of this library cannot call cudaMalloc: code that runs inside a
memory-pool or allocator callback, a host program whose device allocator
belongs to another framework, or a service that must not grow its device
footprint after start-up.  They cannot hand mb_newton_schulz a workspace, so
mb_newton_schulz_noalloc runs the same stage out of a fixed scratch array that
the library itself holds on each device.  This file checks, through the C ABI,
that two calls in a row give the same result as mb_newton_schulz (within the
Newton-Schulz tolerance of the other GPU tests), and that a shape too large for
the fixed scratch is refused without touching the output.

It sits in a file of its own, named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import oracle as O
from gpu_util import NS_TOL, to_dev, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_stacked_gb300.build import build_library
    build_library()
    from newton_schulz_stacked_gb300 import _binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return _binding.load()


def _noalloc(lib, u, v, shape, steps=5):
    from newton_schulz_stacked_gb300 import _binding as b
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mb_newton_schulz_noalloc(ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                        b.shape_of(*shape), steps, ctypes.c_void_p(stream))


def test_noalloc_matches_workspace_entry_point(lib):
    import newton_schulz_stacked_gb300 as nss
    # two calls in a row, different shapes: the second one finds the first one's leftovers in the scratch
    for seed, shape in ((1, (4, 256, 384)), (2, (3, 384, 200))):
        rng = np.random.default_rng(seed)
        u = synth.to_bf16_bits(rng.standard_normal(shape))
        ut = to_dev(u)
        v_ref, v_na = torch.empty_like(ut), torch.empty_like(ut)
        nss.mb_newton_schulz(ut, v_ref, ns_steps=5)
        assert _noalloc(lib, ut, v_na, shape) == 0
        torch.cuda.synchronize()
        assert nss.mb_sync_status() == 0
        a, r = u16(v_na), u16(v_ref)
        for k in range(shape[0]):
            err = O.rel_frobenius(O.bf16_bits_to_f64(a[k]), O.bf16_bits_to_f64(r[k]))
            assert err <= NS_TOL, (shape, k, err)


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    from newton_schulz_stacked_gb300 import _binding as b
    shape = (40, 768, 768)                      # needs far more than the fixed scratch
    need = ctypes.c_size_t()
    assert lib.mb_workspace_bytes(b.shape_of(*shape), 0, ctypes.byref(need)) == 0
    assert need.value > b.MB_NOALLOC_SCRATCH_BYTES
    ut = torch.zeros(shape, dtype=torch.int16, device="cuda:0")
    vt = torch.full(shape, 0x1234, dtype=torch.int16, device="cuda:0")
    assert _noalloc(lib, ut, vt, shape) == b.MB_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((vt == 0x1234).all())
