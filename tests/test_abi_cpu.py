"""The C ABI without a GPU: the library loads, exports every declared entry
point, sizes workspaces, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muonbank.h")


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_stacked_gb300.build import build_library
    build_library()
    from newton_schulz_stacked_gb300 import _binding
    return _binding.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:mb|muon|normuon)_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_step_calls():
    names = _declared()
    for n in ("muon_bank_step", "normuon_bank_step", "muon_multi_step", "mb_workspace_bytes", "mb_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert lib.mb_version() >> 16 == 1
    from newton_schulz_stacked_gb300 import _binding as b
    for code in (b.MB_OK, b.MB_ERR_NULL, b.MB_ERR_SHAPE, b.MB_ERR_ALIGN, b.MB_ERR_NS_STEPS, b.MB_ERR_WORKSPACE,
                 b.MB_ERR_CUDA, b.MB_ERR_TIMEOUT, b.MB_ERR_ARG, b.MB_ERR_UNSUPPORTED, b.MB_ERR_TOO_MANY,
                 b.MB_ERR_SCRATCH_LIMIT, b.MB_ERR_DEVICE):
        assert lib.mb_status_string(code)
    assert lib.mb_status_string(12345) == b"unknown status"


def _ws(lib, shape, normuon=0):
    from newton_schulz_stacked_gb300 import _binding as b
    out = ctypes.c_size_t()
    st = lib.mb_workspace_bytes(b.shape_of(*shape), normuon, ctypes.byref(out))
    return st, out.value


def test_workspace_bytes(lib):
    st, n = _ws(lib, (40, 768, 768))
    assert st == 0
    # two X buffers + A and B (bf16) + partial sums + scale, each 1 KiB aligned
    x = 40 * 768 * 768 * 2
    assert n >= 4 * x
    assert n % 1024 == 0
    st, n_nm = _ws(lib, (40, 768, 768), 1)
    assert st == 0 and n_nm > n
    # small matrices carry fp32 scratch instead of A and B
    st, n_small = _ws(lib, (10, 6, 12))
    assert st == 0 and n_small >= 2 * 10 * 6 * 16 * 2 + 2 * 10 * 72 * 4


@pytest.mark.parametrize("shape", [(0, 4, 4), (1, 0, 4), (1, 4, -1), (1, 1 << 16, 1 << 16),
                                   (1, (1 << 15) + 1, 1 << 15),          # one element past 2^30 per matrix
                                   ((1 << 30) + 1, 1, 1),                # 2^30 rows (and matrices) per bank
                                   (1 << 11, 1 << 15, 1 << 15)])         # 2^41 elements in one bank
def test_workspace_rejects_bad_shapes(lib, shape):
    from newton_schulz_stacked_gb300 import _binding as b
    st, _ = _ws(lib, shape)
    assert st == b.MB_ERR_SHAPE


@pytest.mark.parametrize("shape", [(1, 1 << 15, 1 << 15), (1 << 30, 1, 1), (1 << 10, 1 << 15, 1 << 15)])
def test_workspace_accepts_the_largest_shapes(lib, shape):
    st, n = _ws(lib, shape)
    assert st == 0 and n >= 3 * shape[0] * shape[1] * shape[2] * 2


def test_banks_of_one_call_share_the_launch_limits(lib):
    """Each of these banks is legal alone; two of them overflow the 32-bit grid and the counts of
    matrices and rows that the launches of one call share, so the call refuses them."""
    from newton_schulz_stacked_gb300 import _binding as b
    good = 1 << 12
    arr = (b.MbBankDesc * 2)()
    for i in range(2):
        arr[i] = b.MbBankDesc(good, good, good, good, None, b.shape_of(1 << 30, 1, 1))
    out = ctypes.c_size_t()
    assert lib.mb_multi_workspace_bytes(arr, 1, 0, ctypes.byref(out)) == 0
    assert lib.mb_multi_workspace_bytes(arr, 2, 0, ctypes.byref(out)) == b.MB_ERR_SHAPE
    assert lib.muon_multi_step(arr, 2, 0.02, 0.01, 0.95, 0, 0.95, 5, good, 1 << 62, None) == b.MB_ERR_SHAPE
    assert lib.muon_multi_step_dev(arr, 2, good, 0, 5, good, 1 << 62, None) == b.MB_ERR_SHAPE
    # half as many matrices each: together exactly at the limit
    for i in range(2):
        arr[i].shape = b.shape_of(1 << 29, 1, 1)
    assert lib.mb_multi_workspace_bytes(arr, 2, 0, ctypes.byref(out)) == 0


def test_a_failing_cuda_call_is_reported(lib):
    """Where no CUDA device is usable, every call that needs one fails in the CUDA runtime: the
    library returns MB_ERR_CUDA and keeps the runtime's message, instead of crashing.  The calls
    used take no device pointers, so nothing can be touched on a machine that has a device."""
    import torch
    from newton_schulz_stacked_gb300 import _binding as b
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is usable here")
    assert lib.mb_sync_status(None) == b.MB_ERR_CUDA
    assert lib.mb_last_cuda_error()
    assert lib.mb_selftest_timeout(1000, None) == b.MB_ERR_CUDA
    assert lib.mb_timing_begin(4) == b.MB_ERR_CUDA
    assert lib.mb_timing_end(0, None, None, None) == b.MB_ERR_ARG    # the failed begin left no session
    assert lib.mb_launch_count() == 0


def test_workspace_views(lib):
    from newton_schulz_stacked_gb300 import _binding as b
    u, v, p = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    seen = {}
    for steps in (0, 1, 2, 4, 5):
        assert lib.mb_workspace_views(b.shape_of(3, 10, 13), 0, steps, ctypes.byref(u), ctypes.byref(v),
                                      ctypes.byref(p)) == 0
        assert p.value == 16 and u.value != v.value      # u survives the iterations
        seen[steps] = v.value
    assert seen[0] == seen[1] == seen[5] and seen[2] == seen[4] and seen[1] != seen[2]
    assert lib.mb_workspace_views(b.shape_of(3, 10, 13), 0, 17, ctypes.byref(u), ctypes.byref(v),
                                  ctypes.byref(p)) == b.MB_ERR_NS_STEPS


def test_step_argument_errors_need_no_device(lib):
    from newton_schulz_stacked_gb300 import _binding as b
    sh = b.shape_of(2, 8, 8)
    good = 1 << 12      # aligned, never dereferenced: every call below fails its checks first
    odd = good + 2
    call = lambda *a: lib.muon_bank_step(*a)
    assert call(None, good, good, good, sh, 0.02, 0.01, 0.95, 5, good, 1 << 20, None) == b.MB_ERR_NULL
    assert call(odd, good, good, good, sh, 0.02, 0.01, 0.95, 5, good, 1 << 20, None) == b.MB_ERR_ALIGN
    assert call(good, good, good, good, b.shape_of(2, 0, 8), 0.02, 0.01, 0.95, 5, good, 1 << 20, None) == b.MB_ERR_SHAPE
    assert call(good, good, good, good, sh, 0.02, 0.01, 0.95, 17, good, 1 << 20, None) == b.MB_ERR_NS_STEPS
    assert call(good, good, good, good, sh, 0.02, 0.01, 0.95, -1, good, 1 << 20, None) == b.MB_ERR_NS_STEPS
    assert call(good, good, good, good, sh, float("nan"), 0.01, 0.95, 5, good, 1 << 20, None) == b.MB_ERR_ARG
    assert call(good, good, good, good, sh, 0.02, 0.01, 1.5, 5, good, 1 << 20, None) == b.MB_ERR_ARG
    assert call(good, good, good, good, sh, 0.02, 0.01, 0.95, 5, good, 16, None) == b.MB_ERR_WORKSPACE
    assert call(good, good, good, good, sh, 0.02, 0.01, 0.95, 5, None, 1 << 20, None) == b.MB_ERR_WORKSPACE
    assert call(good, good, good, good, sh, 0.02, 0.01, 0.95, 5, good + 16, 1 << 20, None) == b.MB_ERR_ALIGN
    # NorMuon needs its row state
    assert lib.normuon_bank_step(good, good, good, good, None, sh, 0.02, 0.01, 0.95, 0.95, 5, good, 1 << 20,
                                 None) == b.MB_ERR_NULL
    assert lib.normuon_bank_step(good, good, good, good, good, sh, 0.02, 0.01, 0.95, 1.5, 5, good, 1 << 20,
                                 None) == b.MB_ERR_ARG


def test_multi_step_argument_errors(lib):
    from newton_schulz_stacked_gb300 import _binding as b
    good = 1 << 12
    arr = (b.MbBankDesc * 9)()
    for i in range(9):
        arr[i] = b.MbBankDesc(good, good, good, good, None, b.shape_of(1, 8, 8))
    out = ctypes.c_size_t()
    assert lib.mb_multi_workspace_bytes(arr, 9, 0, ctypes.byref(out)) == b.MB_ERR_TOO_MANY
    assert lib.mb_multi_workspace_bytes(arr, 2, 0, ctypes.byref(out)) == 0
    two = out.value
    assert lib.mb_multi_workspace_bytes(arr, 1, 0, ctypes.byref(out)) == 0 and 2 * out.value == two
    assert lib.muon_multi_step(arr, 9, 0.02, 0.01, 0.95, 0, 0.95, 5, good, 1 << 30, None) == b.MB_ERR_TOO_MANY
    assert lib.muon_multi_step(arr, 0, 0.02, 0.01, 0.95, 0, 0.95, 5, good, 1 << 30, None) == b.MB_ERR_ARG
    assert lib.muon_multi_step(None, 1, 0.02, 0.01, 0.95, 0, 0.95, 5, good, 1 << 30, None) == b.MB_ERR_NULL
    # normuon over banks without row state
    assert lib.muon_multi_step(arr, 2, 0.02, 0.01, 0.95, 1, 0.95, 5, good, 1 << 30, None) == b.MB_ERR_NULL
    # the optional copy of the updated bank must be 16-byte aligned
    arr[1].bank_copy = good + 2
    assert lib.muon_multi_step(arr, 2, 0.02, 0.01, 0.95, 0, 0.95, 5, good, 1 << 30, None) == b.MB_ERR_ALIGN
    arr[1].bank_copy = None
    # device-memory hyperparameters: the buffer pointer is checked before anything else
    assert lib.muon_multi_step_dev(arr, 2, None, 0, 5, good, 1 << 30, None) == b.MB_ERR_NULL
    assert lib.muon_multi_step_dev(arr, 2, good + 4, 0, 5, good, 1 << 30, None) == b.MB_ERR_ALIGN
    assert lib.muon_multi_step_dev(arr, 9, good, 0, 5, good, 1 << 30, None) == b.MB_ERR_TOO_MANY
    assert lib.muon_multi_step_dev(arr, 2, good, 0, 17, good, 1 << 30, None) == b.MB_ERR_NS_STEPS
    assert lib.muon_multi_step_dev(arr, 2, good, 1, 5, good, 1 << 30, None) == b.MB_ERR_NULL
    # options: unknown bits are refused; the known ones pass the argument checks (and then
    # meet the bad workspace size like the plain call)
    assert lib.muon_multi_step_ex(arr, 2, 0.02, 0.01, 0.95, 0, 0.95, 5, 4, good, 1 << 62, None) == b.MB_ERR_ARG
    for flags in (b.MB_STEP_FUSE_UPDATE, b.MB_STEP_FUSE_ROWSTATS, 3):
        assert lib.muon_multi_step_ex(arr, 2, 0.02, 0.01, 0.95, 0, 0.95, 5, flags, good, 16, None) == \
            b.MB_ERR_WORKSPACE


def test_stage_argument_errors(lib):
    from newton_schulz_stacked_gb300 import _binding as b
    good = 1 << 12
    sh = b.shape_of(1, 8, 8)
    assert lib.mb_momentum(None, good, good, sh, 0.9, None) == b.MB_ERR_NULL
    assert lib.mb_newton_schulz(good, good, sh, 99, good, 1 << 20, None) == b.MB_ERR_NS_STEPS
    abc = (ctypes.c_float * 6)(3.4445, -4.775, 2.0315, 1.875, -1.25, 0.375)
    assert lib.mb_newton_schulz_coeffs(good, good, sh, 2, None, good, 1 << 20, None) == b.MB_ERR_NULL
    assert lib.mb_newton_schulz_coeffs(good, good, sh, 17, abc, good, 1 << 20, None) == b.MB_ERR_NS_STEPS
    abc[4] = float("nan")
    assert lib.mb_newton_schulz_coeffs(good, good, sh, 2, abc, good, 1 << 20, None) == b.MB_ERR_ARG
    abc[4] = -1.25
    assert lib.mb_newton_schulz_coeffs(good, good, b.shape_of(0, 8, 8), 2, abc, good, 1 << 20, None) == b.MB_ERR_SHAPE
    assert lib.mb_update(good, good, None, sh, 0.02, 0.01, None) == b.MB_ERR_NULL
    assert lib.mb_normuon_update(good, good, good, good, sh, 0.02, 0.01, 0.95, good, 8, None) == b.MB_ERR_WORKSPACE


def test_python_binding_requires_cuda_tensors():
    import torch
    import newton_schulz_stacked_gb300 as nss
    x = torch.zeros(1, 4, 4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        nss.mb_update(x, x, x, 0.02, 0.01)
