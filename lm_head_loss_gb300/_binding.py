"""ctypes binding of include/flce.h: the same entry points, argument marshalling only.

Every function here converts its arguments (torch tensors or raw integer
addresses, a stream) into the plain pointers and sizes of the C-ABI and
returns the C status code. Nothing here computes any part of the loss.
Importing this module loads libflce.so and fails loudly when it is missing.
"""

from __future__ import annotations

import ctypes
import enum
import os
import re

from .build_lib import INCLUDE, LIB_PATH

HEADER = os.path.join(INCLUDE, "flce.h")


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARGUMENT = 1
    ERR_WORKSPACE_TOO_SMALL = 2
    ERR_BAD_TARGET = 3
    ERR_UNSUPPORTED = 4
    ERR_CUDA = 5
    ERR_TIMEOUT = 6


FLAG_TEST_SHORT_WAITS = 0x1
FLAG_FILTER_FULL_DW = 0x2
FLAG_FILTER_FULL_DH = 0x4
FLAG_COMPACT_IGNORED = 0x8
FLAG_SORT_VOCAB = 0x10
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}


class FlceError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name}" if where else self.status.name)


class FlceProblem(ctypes.Structure):
    _fields_ = [
        ("n_rows", ctypes.c_int64),
        ("hidden", ctypes.c_int64),
        ("vocab", ctypes.c_int64),
        ("ignore_index", ctypes.c_int64),
        ("filter_eps", ctypes.c_float),
        ("flags", ctypes.c_uint32),
    ]


class AdamwHparams(ctypes.Structure):
    """flce_adamw_hparams: one AdamW step's hyper-parameters (kept in device memory)."""
    _fields_ = [
        ("lr", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("weight_decay", ctypes.c_float),
        ("step", ctypes.c_int32),
    ]


def adamw_hparams_bytes(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int) -> bytes:
    """The struct's bytes, for a caller to copy into device memory."""
    return bytes(AdamwHparams(lr, beta1, beta2, eps, weight_decay, step))


def make_problem(n_rows: int, hidden: int, vocab: int, ignore_index: int = -100,
                 filter_eps: float = 0.0, flags: int = 0) -> FlceProblem:
    return FlceProblem(n_rows, hidden, vocab, ignore_index, filter_eps, flags)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libflce.so is not built ({LIB_PATH}); build it with lm_head_loss_gb300.build_lib.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    prob = ctypes.POINTER(FlceProblem)
    lib.flce_workspace_bytes.argtypes = [prob]
    lib.flce_workspace_bytes.restype = sz
    lib.flce_forward_workspace_bytes.argtypes = [prob]
    lib.flce_forward_workspace_bytes.restype = sz
    lib.flce_forward.argtypes = [prob, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward.restype = ctypes.c_int
    lib.flce_forward_backward.argtypes = [prob, vp, vp, vp, f32, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_backward.restype = ctypes.c_int
    lib.flce_count_valid.argtypes = [prob, vp, vp, vp]
    lib.flce_count_valid.restype = ctypes.c_int
    lib.flce_forward_backward_global.argtypes = [prob, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_backward_global.restype = ctypes.c_int
    lib.flce_forward_backward_adamw.argtypes = [prob, vp, vp, vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_backward_adamw.restype = ctypes.c_int
    lib.flce_adamw_step.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp]
    lib.flce_adamw_step.restype = ctypes.c_int
    lib.flce_get_device_status.argtypes = [vp, vp]
    lib.flce_get_device_status.restype = ctypes.c_int
    lib.flce_status_string.argtypes = [ctypes.c_int]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_get_filter_stats.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_double)]
    lib.flce_get_filter_stats.restype = ctypes.c_int
    lib.flce_get_vocab_order.argtypes = [prob, vp, vp, vp, vp]
    lib.flce_get_vocab_order.restype = ctypes.c_int
    lib.flce_forward_ex.argtypes = [prob, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_ex.restype = ctypes.c_int
    lib.flce_backward_ex.argtypes = [prob, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_backward_ex.restype = ctypes.c_int
    lib.flce_forward_static_scratch.argtypes = [prob, vp, vp, vp, vp, vp, vp]
    lib.flce_forward_static_scratch.restype = ctypes.c_int
    lib.flce_profile_set.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
    lib.flce_profile_set.restype = ctypes.c_int
    lib.flce_profile_count.argtypes = []
    lib.flce_profile_count.restype = ctypes.c_int32
    return lib


lib = _load()


def declared_symbols() -> list[str]:
    """Names of the functions include/flce.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:size_t|flce_status|int32_t|const char\*)\s+(flce_\w+)\s*\(", text, re.M)))


def _addr(x) -> int | None:
    """Device (or host) address of a tensor, an int, or None for NULL."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(ws) -> int:
    return ws.numel() * ws.element_size()


def flce_workspace_bytes(problem: FlceProblem | None) -> int:
    return int(lib.flce_workspace_bytes(ctypes.byref(problem) if problem is not None else None))


def flce_forward_workspace_bytes(problem: FlceProblem | None) -> int:
    return int(lib.flce_forward_workspace_bytes(ctypes.byref(problem) if problem is not None else None))


def flce_forward(problem, H, W, y, lse, loss, ws, ws_bytes: int | None = None, stream=None) -> Status:
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_forward(ctypes.byref(problem) if problem is not None else None, _addr(H), _addr(W),
                                   _addr(y), _addr(lse), _addr(loss), _addr(ws), nb, _stream(stream)))


def flce_forward_backward(problem, H, W, y, grad_loss: float, lse, loss, dH, dW, ws, ws_bytes: int | None = None,
                          stream=None) -> Status:
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_forward_backward(ctypes.byref(problem) if problem is not None else None, _addr(H),
                                            _addr(W), _addr(y), float(grad_loss), _addr(lse), _addr(loss),
                                            _addr(dH), _addr(dW), _addr(ws), nb, _stream(stream)))


def flce_count_valid(problem, y, count, stream=None) -> Status:
    """Number of valid targets of these rows into `count` (device int64 [1])."""
    return Status(lib.flce_count_valid(ctypes.byref(problem) if problem is not None else None, _addr(y),
                                       _addr(count), _stream(stream)))


def flce_forward_backward_global(problem, H, W, y, count_global, grad_loss: float, lse, loss, dH, dW, ws,
                                 ws_bytes: int | None = None, stream=None) -> Status:
    """flce_forward_backward with the mean over `count_global` (device int64
    [1], the valid count of every rank of a data-parallel step)."""
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_forward_backward_global(ctypes.byref(problem) if problem is not None else None, _addr(H),
                                                   _addr(W), _addr(y), _addr(count_global), float(grad_loss),
                                                   _addr(lse), _addr(loss), _addr(dH), _addr(dW), _addr(ws), nb,
                                                   _stream(stream)))


def flce_forward_backward_adamw(problem, H, W, y, grad_loss: float, lse, loss, dH, w_master, adam_m, adam_v, w_out,
                                hparams, ws, ws_bytes: int | None = None, stream=None) -> Status:
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_forward_backward_adamw(
        ctypes.byref(problem) if problem is not None else None, _addr(H), _addr(W), _addr(y), float(grad_loss),
        _addr(lse), _addr(loss), _addr(dH), _addr(w_master), _addr(adam_m), _addr(adam_v), _addr(w_out),
        _addr(hparams), _addr(ws), nb, _stream(stream)))


def flce_adamw_step(hparams, grad, w_master, adam_m, adam_v, w_out, n: int, ws, stream=None) -> Status:
    return Status(lib.flce_adamw_step(_addr(hparams), _addr(grad), _addr(w_master), _addr(adam_m), _addr(adam_v),
                                      _addr(w_out), int(n), _addr(ws), _stream(stream)))


def flce_forward_ex(problem, reduction: int, H, W, bias, y, lse, loss, ws, ws_bytes: int | None = None,
                    stream=None) -> Status:
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_forward_ex(ctypes.byref(problem) if problem is not None else None, int(reduction),
                                      _addr(H), _addr(W), _addr(bias), _addr(y), _addr(lse), _addr(loss), _addr(ws),
                                      nb, _stream(stream)))


def flce_backward_ex(problem, reduction: int, H, W, bias, y, lse, grad, dH, dW, dbias, ws,
                     ws_bytes: int | None = None, stream=None) -> Status:
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    return Status(lib.flce_backward_ex(ctypes.byref(problem) if problem is not None else None, int(reduction),
                                       _addr(H), _addr(W), _addr(bias), _addr(y), _addr(lse), _addr(grad),
                                       _addr(dH), _addr(dW), _addr(dbias), _addr(ws), nb, _stream(stream)))


def flce_forward_static_scratch(problem, H, W, y, lse, loss, stream=None) -> Status:
    """flce_forward for callers that cannot hand over a workspace (no device
    allocation at call time); its scratch is a fixed 16 MiB array inside the
    library."""
    return Status(lib.flce_forward_static_scratch(ctypes.byref(problem) if problem is not None else None, _addr(H),
                                                  _addr(W), _addr(y), _addr(lse), _addr(loss), _stream(stream)))


def flce_get_device_status(ws, stream=None) -> Status:
    return Status(lib.flce_get_device_status(_addr(ws), _stream(stream)))


def flce_status_string(status: int) -> str:
    return lib.flce_status_string(int(status)).decode()


def flce_get_filter_stats(ws, stream=None) -> float:
    out = ctypes.c_double(0.0)
    st = lib.flce_get_filter_stats(_addr(ws), _stream(stream), ctypes.byref(out))
    if st != 0:
        raise FlceError(st, "flce_get_filter_stats")
    return out.value


def flce_get_vocab_order(problem, ws, order, avg_logit=None, stream=None) -> Status:
    """Copy the sorted vocabulary order (int32 [V]) and, if given, the average
    logits (float [V]) of the last sorted backward out of the workspace."""
    return Status(lib.flce_get_vocab_order(ctypes.byref(problem) if problem is not None else None, _addr(ws),
                                           _addr(order), _addr(avg_logit), _stream(stream)))


KERNEL_KINDS = {0: "gemm_lse", 1: "gemm_dz", 2: "gemm_dw", 3: "gemm_dh", 4: "prep", 5: "combine",
                6: "finalize", 7: "filter_stats", 8: "gemm_bwd", 9: "dbias", 10: "set_scale",
                11: "vocab_keys", 12: "vocab_sort", 13: "vocab_gather", 14: "adamw_prep",
                15: "adamw_step", 16: "count"}


class LaunchProfiler:
    """Records CUDA-event pairs around every launch of the library
    (flce_profile_set); `summary()` gives per-kind launch counts and summed
    device milliseconds."""

    def __init__(self, capacity: int):
        import torch
        self.capacity = capacity
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.events:           # torch creates the CUDA event on its first record
            e.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.events])
        self._kinds = (ctypes.c_int32 * capacity)()

    def __enter__(self):
        st = lib.flce_profile_set(self._handles, self._kinds, self.capacity)
        if st != 0:
            raise FlceError(st, "flce_profile_set")
        return self

    def __exit__(self, *exc):
        self.count = int(lib.flce_profile_count())
        lib.flce_profile_set(None, None, 0)
        return False

    def launches(self) -> list:
        """(kind, device ms) of every recorded launch, in launch order."""
        import torch
        torch.cuda.synchronize()
        return [(KERNEL_KINDS.get(self._kinds[i], str(self._kinds[i])),
                 self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i in range(min(self.count, self.capacity))]

    def summary(self) -> dict:
        import torch
        torch.cuda.synchronize()
        out: dict = {}
        for i in range(min(self.count, self.capacity)):
            kind = KERNEL_KINDS.get(self._kinds[i], str(self._kinds[i]))
            ms = self.events[2 * i].elapsed_time(self.events[2 * i + 1])
            d = out.setdefault(kind, {"launches": 0, "ms": 0.0})
            d["launches"] += 1
            d["ms"] += ms
        return out
