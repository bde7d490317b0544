"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/flce.h declares, sizes its workspace, and rejects bad
arguments on the host before touching CUDA."""

import ctypes
import math
import subprocess

import pytest

import lm_head_loss_gb300 as flce
from lm_head_loss_gb300 import Status
from lm_head_loss_gb300.build_lib import LIB_PATH

FAKE = 1 << 20          # a 1 MiB-aligned non-null address: never dereferenced on these paths


def test_library_exports_every_declared_symbol():
    declared = flce.declared_symbols()
    assert set(declared) == {"flce_workspace_bytes", "flce_forward", "flce_forward_backward",
                             "flce_get_device_status", "flce_status_string", "flce_get_filter_stats",
                             "flce_profile_set", "flce_profile_count", "flce_forward_static_scratch",
                             "flce_forward_ex", "flce_backward_ex", "flce_forward_workspace_bytes",
                             "flce_get_vocab_order", "flce_forward_backward_adamw", "flce_adamw_step",
                             "flce_count_valid", "flce_forward_backward_global"}
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared:
        assert name in exported, name
        assert hasattr(flce.lib, name)


def test_status_strings():
    for s in Status:
        assert flce.flce_status_string(s) == "FLCE_" + s.name
    assert flce.flce_status_string(99) == "FLCE_UNKNOWN_STATUS"


def test_workspace_is_linear_in_rows_and_vocab_never_n_times_v():
    p = flce.make_problem(8192, 2048, 151552)
    ws = flce.flce_workspace_bytes(p)
    logits = 8192 * 151552 * 2
    assert 0 < ws < logits / 5
    # 16x the rows: O(N) growth (row chunks reuse the same buffers), plus one
    # vocabulary chunk's fp32 dW for the fused optimizer once there are
    # several row chunks.
    p_long = flce.make_problem(131072, 2048, 151552)
    ws_long = flce.flce_workspace_bytes(p_long)
    assert ws_long - ws <= 131072 * 4 + (131072 // 256) * 8 + 10240 * 2048 * 4 + 8192
    assert ws_long < 131072 * 151552 * 2 / 50
    # Tiny problems need little.
    assert flce.flce_workspace_bytes(flce.make_problem(1, 8, 1)) < 1 << 20


def test_compaction_workspace_is_linear_in_rows():
    base = flce.flce_workspace_bytes(flce.make_problem(8192, 2048, 151552))
    comp = flce.flce_workspace_bytes(flce.make_problem(8192, 2048, 151552, flags=flce.FLAG_COMPACT_IGNORED))
    assert 0 < comp - base <= 8192 * 2048 * 6 + 8192 * 28 + 8 * 1024


def test_forward_workspace_is_the_front_of_the_full_one():
    p = flce.make_problem(8192, 2048, 151552)
    fwd, full = flce.flce_forward_workspace_bytes(p), flce.flce_workspace_bytes(p)
    assert 0 < fwd < full / 4
    assert fwd < 8192 * 151552 * 2 / 50
    nb = fwd
    assert flce.flce_forward(p, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws_bytes=nb - 1, stream=0) == \
        Status.ERR_WORKSPACE_TOO_SMALL
    assert flce.flce_forward_backward(p, FAKE, FAKE, FAKE, 1.0, None, FAKE, FAKE, FAKE, FAKE, ws_bytes=nb,
                                      stream=0) == Status.ERR_WORKSPACE_TOO_SMALL
    assert flce.flce_forward_workspace_bytes(None) == 0


def test_sorted_vocabulary_workspace_and_getter_checks():
    base = flce.make_problem(8192, 2048, 151552)
    srt = flce.make_problem(8192, 2048, 151552, flags=flce.FLAG_SORT_VOCAB)
    grow = flce.flce_workspace_bytes(srt) - flce.flce_workspace_bytes(base)
    v, d, n = 151552, 2048, 8192
    assert v * d * 2 <= grow <= v * d * 2 + 29 * v + 8 * n + 1028 * d + 12 * 1024
    # The forward needs none of it.
    assert flce.flce_forward_workspace_bytes(srt) == flce.flce_forward_workspace_bytes(base)
    # Sorting and compaction together: the compaction buffers come after.
    both = flce.make_problem(8192, 2048, 151552, flags=flce.FLAG_SORT_VOCAB | flce.FLAG_COMPACT_IGNORED)
    comp = flce.make_problem(8192, 2048, 151552, flags=flce.FLAG_COMPACT_IGNORED)
    assert flce.flce_workspace_bytes(both) - flce.flce_workspace_bytes(comp) == grow
    st = flce.flce_get_vocab_order
    assert st(base, FAKE, FAKE, None, 0) == Status.ERR_INVALID_ARGUMENT      # flag not set
    assert st(srt, None, FAKE, None, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(srt, FAKE, None, None, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(srt, FAKE + 16, FAKE, None, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(srt, FAKE, FAKE + 2, None, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(None, FAKE, FAKE, None, 0) == Status.ERR_INVALID_ARGUMENT


def test_fused_adamw_argument_checks():
    assert ctypes.sizeof(flce.AdamwHparams) == 24
    assert flce.AdamwHparams.step.offset == 20
    good = flce.make_problem(16, 64, 100)
    nb = flce.flce_workspace_bytes(good)
    wbytes = 100 * 64 * 2
    W_ = FAKE
    out = FAKE + (1 << 24)

    def call(prob=good, w_out=out, hp=FAKE, dH=FAKE, master=FAKE, n=nb):
        return flce.flce_forward_backward_adamw(prob, FAKE, W_, FAKE, 1.0, None, FAKE, dH, master, FAKE, FAKE,
                                                w_out, hp, FAKE, ws_bytes=n, stream=0)
    assert call(hp=None) == Status.ERR_INVALID_ARGUMENT
    assert call(hp=FAKE + 4) == Status.ERR_INVALID_ARGUMENT
    assert call(master=None) == Status.ERR_INVALID_ARGUMENT
    assert call(dH=None) == Status.ERR_INVALID_ARGUMENT
    assert call(w_out=None) == Status.ERR_INVALID_ARGUMENT
    assert call(w_out=W_ + wbytes - 16) == Status.ERR_INVALID_ARGUMENT     # overlaps W
    assert call(master=FAKE + 8) == Status.ERR_UNSUPPORTED                 # not 16-byte aligned
    assert call(n=nb - 1) == Status.ERR_WORKSPACE_TOO_SMALL
    none = flce.make_problem(0, 64, 100)
    assert call(prob=none, n=flce.flce_workspace_bytes(none)) == Status.ERR_UNSUPPORTED


def test_adamw_step_argument_checks():
    st = flce.flce_adamw_step
    assert st(None, FAKE, FAKE, FAKE, FAKE, None, 10, FAKE, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(FAKE, FAKE, FAKE, FAKE, FAKE, None, -1, FAKE, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(FAKE, FAKE, FAKE, FAKE, FAKE, None, 10, None, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(FAKE, FAKE, FAKE, FAKE, FAKE, None, 10, FAKE + 64, 0) == Status.ERR_INVALID_ARGUMENT
    assert st(FAKE, FAKE + 4, FAKE, FAKE, FAKE, None, 10, FAKE, 0) == Status.ERR_UNSUPPORTED
    assert st(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 10, FAKE, 0) == Status.ERR_UNSUPPORTED


def test_workspace_bytes_rejects_bad_problems():
    assert flce.flce_workspace_bytes(None) == 0
    for args in [(-1, 8, 10), (4, 0, 10), (4, 8, 0), (4, 8, 1 << 31)]:
        assert flce.flce_workspace_bytes(flce.make_problem(*args)) == 0
    assert flce.flce_workspace_bytes(flce.make_problem(4, 8, 10, filter_eps=-1.0)) == 0
    assert flce.flce_workspace_bytes(flce.make_problem(4, 8, 10, filter_eps=math.inf)) == 0
    assert flce.flce_workspace_bytes(flce.make_problem(4, 8, 10, flags=0x80)) == 0
    assert flce.flce_workspace_bytes(flce.make_problem(4, 8, 10, flags=0x20)) == 0
    assert flce.flce_workspace_bytes(flce.make_problem(0, 8, 10)) > 0


def _fwd(prob, H=FAKE, W=FAKE, y=FAKE, lse=FAKE, loss=FAKE, ws=FAKE, nb=None):
    nb = flce.flce_workspace_bytes(prob) if nb is None and prob is not None else (nb or 0)
    return flce.flce_forward(prob, H, W, y, lse, loss, ws, ws_bytes=nb, stream=0)


def _fb(prob, H=FAKE, W=FAKE, y=FAKE, lse=None, loss=FAKE, dH=FAKE, dW=FAKE, ws=FAKE, nb=None, g=1.0):
    nb = flce.flce_workspace_bytes(prob) if nb is None and prob is not None else (nb or 0)
    return flce.flce_forward_backward(prob, H, W, y, g, lse, loss, dH, dW, ws, ws_bytes=nb, stream=0)


def test_host_argument_checks_return_before_any_launch():
    good = flce.make_problem(16, 64, 100)
    assert _fwd(None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, H=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, W=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, y=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, lse=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, loss=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, ws=None) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(good, ws=FAKE + 16) == Status.ERR_INVALID_ARGUMENT          # ws not 256-byte aligned
    assert _fwd(good, y=FAKE + 4) == Status.ERR_INVALID_ARGUMENT            # int64 targets misaligned
    assert _fwd(good, H=FAKE + 8) == Status.ERR_UNSUPPORTED                 # TMA needs 16-byte alignment
    assert _fwd(good, nb=flce.flce_forward_workspace_bytes(good) - 1) == Status.ERR_WORKSPACE_TOO_SMALL
    assert _fwd(flce.make_problem(16, 60, 100)) == Status.ERR_UNSUPPORTED   # D % 8 != 0
    assert _fwd(flce.make_problem(16, 64, 100, flags=0x20)) == Status.ERR_INVALID_ARGUMENT
    assert _fwd(flce.make_problem(16, 64, 100, filter_eps=float("nan"))) == Status.ERR_INVALID_ARGUMENT
    assert _fb(good, dW=None) == Status.ERR_INVALID_ARGUMENT
    assert _fb(good, dH=None) == Status.ERR_INVALID_ARGUMENT
    assert _fb(good, dH=FAKE + 4) == Status.ERR_UNSUPPORTED
    assert _fb(good, g=float("inf")) == Status.ERR_INVALID_ARGUMENT
    assert _fb(good, nb=1) == Status.ERR_WORKSPACE_TOO_SMALL


def test_general_entry_points_check_arguments():
    good = flce.make_problem(16, 64, 100)
    nb = flce.flce_workspace_bytes(good)
    assert flce.flce_forward_ex(good, 3, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, nb, 0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_forward_ex(good, 2, FAKE, FAKE, None, FAKE, None, FAKE, FAKE, nb, 0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_backward_ex(good, 0, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, nb,
                                 0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_backward_ex(good, 0, FAKE, FAKE, None, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, nb,
                                 0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_backward_ex(good, 0, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE + 4, None, FAKE, nb,
                                 0) == Status.ERR_UNSUPPORTED
    assert flce.flce_backward_ex(good, 9, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, nb,
                                 0) == Status.ERR_INVALID_ARGUMENT


def test_profile_hook_arguments():
    assert flce.lib.flce_profile_set(None, None, -1) == Status.ERR_INVALID_ARGUMENT
    assert flce.lib.flce_profile_set(None, None, 4) == Status.ERR_INVALID_ARGUMENT
    assert flce.lib.flce_profile_set(None, None, 0) == Status.OK
    assert flce.lib.flce_profile_count() == 0


def test_device_status_rejects_null_workspace():
    assert flce.flce_get_device_status(None, stream=0) == Status.ERR_INVALID_ARGUMENT
    with pytest.raises(flce.FlceError):
        flce.flce_get_filter_stats(None, stream=0)


def test_problem_struct_layout_matches_header():
    # int64 x4, float, uint32 -> 40 bytes, 8-byte aligned.
    assert ctypes.sizeof(flce.FlceProblem) == 40
    assert flce.FlceProblem.filter_eps.offset == 32 and flce.FlceProblem.flags.offset == 36


def test_api_refuses_cpu_tensors():
    import torch
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(5, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        flce.forward(H, W, y)


def test_data_parallel_step_refuses_cpu_tensors():
    # The step's buffers need a GPU; the check on the inputs comes first, so a
    # step object without them is enough to see CPU tensors refused.
    import torch
    step = object.__new__(flce.DataParallelStep)
    step.problem = flce.make_problem(4, 8, 5)
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(5, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        step(H, W, y)
    with pytest.raises(TypeError):
        step(H.float(), W, y)


def test_data_parallel_calls_reject_bad_arguments_on_the_host():
    # Rejected before any launch, so this runs without a GPU.
    p = flce.make_problem(64, 128, 1000)
    nb = flce.flce_workspace_bytes(p)
    assert flce.flce_count_valid(p, FAKE, None, stream=0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_count_valid(None, FAKE, FAKE, stream=0) == Status.ERR_INVALID_ARGUMENT
    assert flce.flce_count_valid(p, FAKE + 4, FAKE, stream=0) == Status.ERR_INVALID_ARGUMENT
    call = flce.flce_forward_backward_global
    assert call(p, FAKE, FAKE, FAKE, None, 1.0, None, FAKE, FAKE, FAKE, FAKE, ws_bytes=nb,
                stream=0) == Status.ERR_INVALID_ARGUMENT
    assert call(p, FAKE, FAKE, FAKE, FAKE + 4, 1.0, None, FAKE, FAKE, FAKE, FAKE, ws_bytes=nb,
                stream=0) == Status.ERR_INVALID_ARGUMENT
    assert call(p, FAKE, FAKE, FAKE, FAKE, 1.0, None, FAKE, FAKE, FAKE, FAKE, ws_bytes=nb - 1,
                stream=0) == Status.ERR_WORKSPACE_TOO_SMALL


def test_caller_output_buffers_are_checked_before_use():
    # forward_backward(out=...) hands these pointers to kernels that write the
    # full shapes; a short or mistyped buffer must be refused on the host.
    import torch
    from lm_head_loss_gb300.api import _check_out
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(5, 8, dtype=torch.bfloat16)
    good = (torch.zeros(()), torch.zeros(4), torch.zeros(4, 8), torch.zeros(5, 8))
    _check_out(good, H, W)
    bad = [(torch.zeros(()), torch.zeros(4), torch.zeros(4, 8), torch.zeros(4, 8)),       # dW too short
           (torch.zeros(()), torch.zeros(3), torch.zeros(4, 8), torch.zeros(5, 8)),       # lse too short
           (torch.zeros(()), torch.zeros(4), torch.zeros(4, 8).double(), torch.zeros(5, 8)),
           (torch.zeros(()), torch.zeros(4), torch.zeros(8, 4).t(), torch.zeros(5, 8)),   # not contiguous
           (torch.zeros(2), torch.zeros(4), torch.zeros(4, 8), torch.zeros(5, 8)),
           good[:3]]
    for out in bad:
        with pytest.raises(ValueError):
            _check_out(out, H, W)
