"""The allocation-free Newton-Schulz entry point, checked against the workspace one.

Some callers of this library cannot call cudaMalloc: code that runs inside a
memory-pool or allocator callback, a host program whose device allocator
belongs to another framework, or a service that must not grow its device
footprint after start-up.  They cannot hand mb_newton_schulz a workspace, so
mb_newton_schulz_noalloc runs the same stage out of a fixed scratch array that
the library itself holds on each device.

This file checks, through the C ABI, a sequence of calls in a row on one
stream: each call's output must equal mb_newton_schulz's on the same input bit
for bit (the two run the same kernels; only the scratch differs) and lie within
the Newton-Schulz tolerance of the fp64 oracle.  The sequence mixes the
tensor-core path, both fp32 small-matrix paths (in shared memory, and through
the scratch) and ns_steps = 0, so that every call starts on what the previous
one left in the shared array, and ends by repeating its first call.  A shape
too large for the fixed scratch must be refused without touching the output.

It sits in a file of its own, named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import check_ns, ns_tol, to_dev, u16

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


# (seed, shape, ns_steps): tensor-core path, fp32 path in shared memory, fp32 path through the
# scratch (wide and tall), v = X0 with no iteration, a tall tensor-core bank, and the first again
SEQUENCE = [
    (1, (4, 256, 384), 5),
    (2, (5, 40, 300), 5),
    (3, (3, 40, 2000), 5),
    (4, (3, 500, 48), 5),
    (5, (2, 200, 328), 0),
    (6, (3, 384, 200), 5),
    (1, (4, 256, 384), 5),
]


def test_noalloc_matches_workspace_entry_point(lib):
    import newton_schulz_stacked_gb300 as nss
    first = None
    for seed, shape, steps in SEQUENCE:
        rng = np.random.default_rng(seed)
        u = synth.to_bf16_bits(rng.standard_normal(shape))
        ut = to_dev(u)
        v_ref = torch.empty_like(ut)
        v_na = torch.full_like(ut, 0x7F7F)           # a pattern the result cannot keep by accident
        nss.mb_newton_schulz(ut, v_ref, ns_steps=steps)
        assert _noalloc(lib, ut, v_na, shape, steps) == 0
        torch.cuda.synchronize()
        assert nss.mb_sync_status() == 0
        a, r = u16(v_na), u16(v_ref)
        np.testing.assert_array_equal(a, r, err_msg=f"{shape} ns_steps={steps}")
        if steps == 0:
            s = np.array([O.frobenius_scale(O.bf16_bits_to_f64(u[k])) for k in range(shape[0])])
            ref = O.bf16_bits_to_f64(u) * s[:, None, None]
            errs = np.array([O.rel_frobenius(O.bf16_bits_to_f64(a[k]), ref[k]) for k in range(shape[0])])
            assert errs.max() <= 2.0 ** -8, errs               # one bf16 rounding of s * u
        else:
            errs = check_ns(u, a, steps)
            assert errs.max() <= ns_tol(*shape[1:], steps=steps), (shape, errs)
        if first is None:
            first = (shape, a)
        elif shape == first[0]:
            np.testing.assert_array_equal(a, first[1])         # the same call again gives the same bits


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
