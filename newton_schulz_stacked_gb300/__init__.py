"""GB300-native Muon step over stacked parameter banks.

Thin Python face of libmuonbank.so: each function has the name of the C
entry point it calls, takes CUDA tensors (bf16 banks may be passed as
torch.bfloat16, int16 or uint16 tensors: only the bits matter) and enqueues
the work on the current CUDA stream.  All arithmetic runs in the library's
kernels.  Buffers are the caller's; a workspace tensor is created with
torch only when the caller does not pass one.
"""
from __future__ import annotations

import contextlib
import ctypes
from typing import Optional, Sequence

import torch

from . import _binding as _b
from ._binding import MuonBankError, MB_MAX_BANKS, MB_STEP_FUSE_ROWSTATS, MB_STEP_FUSE_UPDATE  # noqa: F401

__all__ = [
    "muon_bank_step", "normuon_bank_step", "muon_multi_step", "mb_workspace_bytes",
    "mb_multi_workspace_bytes", "muon_multi_step_dev", "mb_momentum", "mb_newton_schulz",
    "mb_newton_schulz_coeffs", "mb_update", "mb_normuon_update", "mb_newton_schulz_noalloc", "mb_workspace_views",
    "mb_sync_status", "mb_selftest_timeout", "mb_status_string", "MuonBankError",
    "BankState", "load_library", "mb_launch_count", "StageTimer",
]

_TWO_BYTE = (torch.bfloat16, torch.int16, torch.uint16, torch.float16)


def load_library():
    return _b.load()


def _ptr(t: Optional[torch.Tensor], dtypes, what: str) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{what} has dtype {t.dtype}, expected one of {dtypes}")
    return t.data_ptr()


def _same(what: str, ref: torch.Tensor, t: Optional[torch.Tensor], numel: Optional[int] = None):
    """The kernels index every tensor of a call with one shape: a tensor of another size or
    on another device would be read or written out of bounds, so it is refused here."""
    if t is None:
        return
    want = ref.numel() if numel is None else numel
    if t.numel() != want:
        raise ValueError(f"{what} has {t.numel()} elements, expected {want}")
    if t.device != ref.device:
        raise ValueError(f"{what} is on {t.device}, the call's tensors are on {ref.device}")


def _on(t: torch.Tensor):
    """Runs the call with the tensors' device current (the library launches on the current device)."""
    return torch.cuda.device(t.device) if t.is_cuda else contextlib.nullcontext()


def _shape(t: torch.Tensor) -> _b.MbShape:
    if t.dim() == 2:
        return _b.shape_of(1, t.shape[0], t.shape[1])
    if t.dim() != 3:
        raise ValueError("a bank is [batch, rows, cols] (or one [rows, cols] matrix)")
    return _b.shape_of(*t.shape)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _workspace(nbytes: int, workspace: Optional[torch.Tensor], device) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device)
    if not workspace.is_cuda or workspace.device != torch.device(device):
        raise ValueError(f"workspace must be a CUDA tensor on {device}")
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, needs {nbytes}")
    return workspace


def mb_status_string(status: int) -> str:
    return _b.load().mb_status_string(status).decode()


def mb_workspace_bytes(shape, normuon: bool = False) -> int:
    out = ctypes.c_size_t(0)
    _b.check("mb_workspace_bytes", _b.load().mb_workspace_bytes(_b.shape_of(*shape), int(normuon), ctypes.byref(out)))
    return out.value


def muon_bank_step(bank, grad, momentum, mantissa, lr: float, wd: float, mu: float, ns_steps: int = 5,
                   workspace=None, stream=None):
    """One Muon step over the bank, in place (bank, momentum, mantissa)."""
    sh = _shape(bank)
    for name, t in (("grad", grad), ("momentum", momentum), ("mantissa", mantissa)):
        _same(name, bank, t)
    ws = _workspace(mb_workspace_bytes((sh.batch, sh.rows, sh.cols)), workspace, bank.device)
    with _on(bank):
        st = _b.load().muon_bank_step(
            _ptr(bank, _TWO_BYTE, "bank"), _ptr(grad, _TWO_BYTE, "grad"), _ptr(momentum, (torch.float32,), "momentum"),
            _ptr(mantissa, _TWO_BYTE, "mantissa"), sh, lr, wd, mu, ns_steps, ws.data_ptr(),
            ws.numel() * ws.element_size(), _stream(stream))
    _b.check("muon_bank_step", st)
    return ws


def normuon_bank_step(bank, grad, momentum, mantissa, row_state, lr: float, wd: float, mu: float,
                      beta2: float = 0.95, ns_steps: int = 5, workspace=None, stream=None):
    """One Muon step with NorMuon per-row normalisation, in place (row_state too)."""
    sh = _shape(bank)
    for name, t in (("grad", grad), ("momentum", momentum), ("mantissa", mantissa)):
        _same(name, bank, t)
    _same("row_state", bank, row_state, sh.batch * sh.rows)
    ws = _workspace(mb_workspace_bytes((sh.batch, sh.rows, sh.cols), True), workspace, bank.device)
    with _on(bank):
        st = _b.load().normuon_bank_step(
            _ptr(bank, _TWO_BYTE, "bank"), _ptr(grad, _TWO_BYTE, "grad"), _ptr(momentum, (torch.float32,), "momentum"),
            _ptr(mantissa, _TWO_BYTE, "mantissa"), _ptr(row_state, (torch.float32,), "row_state"), sh, lr, wd, mu,
            beta2, ns_steps, ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    _b.check("normuon_bank_step", st)
    return ws


class BankState:
    """The caller-owned tensors of one bank: bank, grad, momentum, mantissa (and row_state).

    bank_copy, when set, is a second bf16 tensor of the bank's shape that each step's update
    also writes the new bank into (for example a buffer to download while the next step runs).
    """

    def __init__(self, bank, grad, momentum, mantissa, row_state=None, bank_copy=None):
        self.bank, self.grad, self.momentum, self.mantissa, self.row_state = bank, grad, momentum, mantissa, row_state
        self.bank_copy = bank_copy

    def desc(self) -> _b.MbBankDesc:
        for name, t in (("grad", self.grad), ("momentum", self.momentum), ("mantissa", self.mantissa),
                        ("bank_copy", self.bank_copy)):
            _same(name, self.bank, t)
        if self.row_state is not None:
            sh = _shape(self.bank)
            _same("row_state", self.bank, self.row_state, sh.batch * sh.rows)
        return _b.MbBankDesc(_ptr(self.bank, _TWO_BYTE, "bank"), _ptr(self.grad, _TWO_BYTE, "grad"),
                             _ptr(self.momentum, (torch.float32,), "momentum"),
                             _ptr(self.mantissa, _TWO_BYTE, "mantissa"),
                             _ptr(self.row_state, (torch.float32,), "row_state"), _shape(self.bank),
                             _ptr(self.bank_copy, _TWO_BYTE, "bank_copy"))


def _descs(banks: Sequence[BankState]):
    if len(banks) == 0:
        raise ValueError("no banks")
    for b in banks[1:]:
        if b.bank.device != banks[0].bank.device:
            raise ValueError("all banks of one call must be on one device")
    arr = (_b.MbBankDesc * len(banks))()
    for i, b in enumerate(banks):
        arr[i] = b.desc()
    return arr


def mb_multi_workspace_bytes(banks: Sequence[BankState], normuon: bool = False) -> int:
    out = ctypes.c_size_t(0)
    _b.check("mb_multi_workspace_bytes",
             _b.load().mb_multi_workspace_bytes(_descs(banks), len(banks), int(normuon), ctypes.byref(out)))
    return out.value


def muon_multi_step(banks: Sequence[BankState], lr: float, wd: float, mu: float, normuon: bool = False,
                    beta2: float = 0.95, ns_steps: int = 5, workspace=None, stream=None, flags: int = 0):
    """One step over several banks as one launch sequence (flags: MB_STEP_* options, which go
    through muon_multi_step_ex)."""
    arr = _descs(banks)
    ws = _workspace(mb_multi_workspace_bytes(banks, normuon), workspace, banks[0].bank.device)
    lib = _b.load()
    with _on(banks[0].bank):
        if flags:
            st = lib.muon_multi_step_ex(arr, len(banks), lr, wd, mu, int(normuon), beta2, ns_steps, flags,
                                        ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
        else:
            st = lib.muon_multi_step(arr, len(banks), lr, wd, mu, int(normuon), beta2, ns_steps, ws.data_ptr(),
                                     ws.numel() * ws.element_size(), _stream(stream))
    _b.check("muon_multi_step_ex" if flags else "muon_multi_step", st)
    return ws


def muon_multi_step_dev(banks: Sequence[BankState], scalars, normuon: bool = False, ns_steps: int = 5,
                        workspace=None, stream=None):
    """muon_multi_step with the hyperparameters read on the device from `scalars`.

    `scalars` is a CUDA float32 tensor of len(banks) x 4 values (lr, wd, mu, beta2 per bank).
    The step reads it when it runs, so a CUDA graph that captured this call replays
    with whatever the tensor holds at replay time.
    """
    if not (isinstance(scalars, torch.Tensor) and scalars.is_cuda and scalars.dtype == torch.float32
            and scalars.is_contiguous() and scalars.numel() == 4 * len(banks)):
        raise ValueError("scalars must be a contiguous CUDA float32 tensor of 4 values per bank")
    arr = _descs(banks)
    if scalars.device != banks[0].bank.device:
        raise ValueError("scalars must be on the banks' device")
    ws = _workspace(mb_multi_workspace_bytes(banks, normuon), workspace, banks[0].bank.device)
    with _on(banks[0].bank):
        st = _b.load().muon_multi_step_dev(arr, len(banks), scalars.data_ptr(), int(normuon), ns_steps,
                                           ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    _b.check("muon_multi_step_dev", st)
    return ws


def mb_momentum(grad, momentum, u, mu: float, stream=None):
    sh = _shape(grad)
    _same("momentum", grad, momentum)
    _same("u", grad, u)
    with _on(grad):
        _b.check("mb_momentum", _b.load().mb_momentum(
            _ptr(grad, _TWO_BYTE, "grad"), _ptr(momentum, (torch.float32,), "momentum"), _ptr(u, _TWO_BYTE, "u"), sh,
            mu, _stream(stream)))


def mb_newton_schulz_coeffs(u, v, coeffs, workspace=None, stream=None):
    """mb_newton_schulz with a per-step coefficient schedule: `coeffs` is a sequence of
    (a, b, c), one per step (its length is the number of steps)."""
    flat = [float(x) for abc in coeffs for x in abc]
    if len(flat) != 3 * len(coeffs):
        raise ValueError("coeffs must be a sequence of (a, b, c) triples")
    arr = (ctypes.c_float * max(len(flat), 1))(*flat)
    sh = _shape(u)
    _same("v", u, v)
    ws = _workspace(mb_workspace_bytes((sh.batch, sh.rows, sh.cols)), workspace, u.device)
    with _on(u):
        _b.check("mb_newton_schulz_coeffs", _b.load().mb_newton_schulz_coeffs(
            _ptr(u, _TWO_BYTE, "u"), _ptr(v, _TWO_BYTE, "v"), sh, len(coeffs), arr, ws.data_ptr(),
            ws.numel() * ws.element_size(), _stream(stream)))
    return ws


def mb_newton_schulz(u, v, ns_steps: int = 5, workspace=None, stream=None):
    sh = _shape(u)
    _same("v", u, v)
    ws = _workspace(mb_workspace_bytes((sh.batch, sh.rows, sh.cols)), workspace, u.device)
    with _on(u):
        _b.check("mb_newton_schulz", _b.load().mb_newton_schulz(
            _ptr(u, _TWO_BYTE, "u"), _ptr(v, _TWO_BYTE, "v"), sh, ns_steps, ws.data_ptr(),
            ws.numel() * ws.element_size(), _stream(stream)))
    return ws


def mb_newton_schulz_noalloc(u, v, ns_steps: int = 5, stream=None):
    """mb_newton_schulz without a workspace, for callers that cannot allocate device memory.

    The library serves the scratch from its fixed per-device array (at most
    MB_NOALLOC_SCRATCH_BYTES); calls share it, so do not overlap them on the GPU.
    """
    sh = _shape(u)
    _same("v", u, v)
    with _on(u):
        _b.check("mb_newton_schulz_noalloc", _b.load().mb_newton_schulz_noalloc(
            _ptr(u, _TWO_BYTE, "u"), _ptr(v, _TWO_BYTE, "v"), sh, ns_steps, _stream(stream)))


def mb_update(bank, mantissa, v, lr: float, wd: float, stream=None):
    sh = _shape(bank)
    _same("mantissa", bank, mantissa)
    _same("v", bank, v)
    with _on(bank):
        _b.check("mb_update", _b.load().mb_update(
            _ptr(bank, _TWO_BYTE, "bank"), _ptr(mantissa, _TWO_BYTE, "mantissa"), _ptr(v, _TWO_BYTE, "v"), sh, lr,
            wd, _stream(stream)))


def mb_normuon_update(bank, mantissa, v, row_state, lr: float, wd: float, beta2: float = 0.95, workspace=None,
                      stream=None):
    sh = _shape(bank)
    _same("mantissa", bank, mantissa)
    _same("v", bank, v)
    _same("row_state", bank, row_state, sh.batch * sh.rows)
    ws = _workspace(mb_workspace_bytes((sh.batch, sh.rows, sh.cols), True), workspace, bank.device)
    with _on(bank):
        _b.check("mb_normuon_update", _b.load().mb_normuon_update(
            _ptr(bank, _TWO_BYTE, "bank"), _ptr(mantissa, _TWO_BYTE, "mantissa"), _ptr(v, _TWO_BYTE, "v"),
            _ptr(row_state, (torch.float32,), "row_state"), sh, lr, wd, beta2, ws.data_ptr(),
            ws.numel() * ws.element_size(), _stream(stream)))
    return ws


def mb_workspace_views(shape, normuon: bool = False, ns_steps: int = 5):
    """(u byte offset, v byte offset, row pitch in elements) inside a step's workspace."""
    u, v, p = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _b.check("mb_workspace_views", _b.load().mb_workspace_views(
        _b.shape_of(*shape), int(normuon), ns_steps, ctypes.byref(u), ctypes.byref(v), ctypes.byref(p)))
    return u.value, v.value, p.value


def mb_sync_status(stream=None) -> int:
    return _b.load().mb_sync_status(_stream(stream))


def mb_selftest_timeout(limit_us: int, stream=None):
    _b.check("mb_selftest_timeout", _b.load().mb_selftest_timeout(limit_us, _stream(stream)))


def mb_launch_count() -> int:
    """Kernels this thread has launched through the library so far."""
    return int(_b.load().mb_launch_count())


class StageTimer:
    """Records CUDA events at the library's stage boundaries while active.

    with StageTimer(max_marks) as t: ...steps...
    t.marks -> list of (stage name, ms since the previous mark)
    """

    def __init__(self, max_marks: int = 4096):
        self.max_marks = max_marks
        self.marks = []

    def __enter__(self):
        _b.check("mb_timing_begin", _b.load().mb_timing_begin(self.max_marks))
        return self

    def __exit__(self, *exc):
        n = self.max_marks
        labels = (ctypes.c_int * n)()
        ms = (ctypes.c_float * n)()
        got = ctypes.c_int(0)
        _b.check("mb_timing_end", _b.load().mb_timing_end(n, labels, ms, ctypes.byref(got)))
        self.marks = [(_b.MARK_NAMES.get(labels[i], str(labels[i])), float(ms[i])) for i in range(min(got.value, n))]
        return False

    def totals(self):
        """Per stage: (total ms, number of marks)."""
        out = {}
        for name, ms in self.marks:
            if name == "begin":
                continue
            t, c = out.get(name, (0.0, 0))
            out[name] = (t + ms, c + 1)
        return out
