"""Host-only checks of the C ABI: the library loads without a GPU, exports every function
include/moe.h declares, and rejects bad arguments on the host before any launch.

Every call below fails host validation, so nothing is launched (on a GPU machine too): the
fake device addresses are never dereferenced."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from sparse_moe_ffn_router_gb300 import binding
from sparse_moe_ffn_router_gb300.binding import CWeights, Dims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FULL = (64, 2048, 256, 8, 512, 512)
A = 0x10000000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    return binding.load_library()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(names) == set(binding.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_workspace_size_and_taps(lib):
    n = lib.moe_workspace_size(ctypes.byref(Dims(*FULL)))
    assert n > 0 and n % 256 == 0
    # Y [T, K+1, H] fp32 dominates; it must fit
    assert n >= 64 * 9 * 2048 * 4
    assert lib.moe_workspace_size(ctypes.byref(Dims(0, 2048, 256, 8, 512, 512))) > 0
    for bad in [(1, 2000, 256, 8, 512, 512), (1, 2048, 257, 8, 512, 512), (1, 2048, 256, 9, 512, 512),
                (1, 2048, 4, 8, 512, 512), (1, 2048, 256, 8, 500, 512), (-1, 2048, 256, 8, 512, 512),
                (1, 2048, 256, 0, 512, 512), (1, 64, 8, 2, 64, 64)]:
        assert lib.moe_workspace_size(ctypes.byref(Dims(*bad))) == 0, bad
    off, nb = binding.moe_workspace_tap(FULL, 1)
    assert off % 256 == 0 and nb == 64 * 9 * 2048 * 4 and off + nb <= n
    with pytest.raises(binding.MoEError):
        binding.moe_workspace_tap(FULL, 99)


def _weights(**over):
    w = dict(router_w=A, router_b=None, gate_up=A, down=A, shared_gate_up=A, shared_down=A, shared_gate=A)
    w.update(over)
    return CWeights(*[w[f[0]] for f in CWeights._fields_])


def _forward(lib, dims=FULL, x=A + 0x100000, w=None, res=None, out=A + 0x200000, ws=A + 0x400000, wsb=None):
    d = Dims(*dims)
    if wsb is None:
        wsb = lib.moe_workspace_size(ctypes.byref(d))
    w = w or _weights()
    return lib.moe_forward(ctypes.byref(d), x, ctypes.byref(w), res, out, ws, wsb, None)


def test_forward_rejects_bad_arguments(lib):
    assert lib.moe_forward(None, A, None, None, A, A, 0, None) == 1
    assert _forward(lib, dims=(1, 2048, 256, 9, 512, 512)) == 2
    assert _forward(lib, x=None) == 1
    assert _forward(lib, w=_weights(down=None)) == 1
    assert _forward(lib, out=None) == 1
    assert _forward(lib, x=A + 8) == 3
    assert _forward(lib, w=_weights(gate_up=A + 2)) == 3
    assert _forward(lib, out=A + 0x200002) == 3
    assert _forward(lib, ws=A + 0x400004) == 3
    assert _forward(lib, wsb=1024) == 4
    # out overlapping x, and out partly overlapping residual
    assert _forward(lib, out=A + 0x100000 + 64 * 2048) == 1
    assert _forward(lib, res=A + 0x200000 + 4096) == 1


def test_zero_tokens_is_a_noop(lib):
    assert _forward(lib, dims=(0, 2048, 256, 8, 512, 512), x=None, out=None, ws=None, wsb=0) == 0


def test_route_and_rmsnorm_reject_bad_arguments(lib):
    d = Dims(*FULL)
    w = _weights()
    wsb = lib.moe_workspace_size(ctypes.byref(d))
    assert lib.moe_route(ctypes.byref(d), A, ctypes.byref(w), A, A, None, A, A, A, wsb, None) == 1
    assert lib.moe_route(ctypes.byref(d), A, ctypes.byref(w), None, A, A, A, A, A, wsb, None) == 1
    assert lib.moe_route(ctypes.byref(d), A, ctypes.byref(w), A + 4, A, A, A, A, A, wsb, None) == 3
    assert lib.moe_route(ctypes.byref(d), A, ctypes.byref(w), A, A, A, A, A, A, wsb - 256, None) == 4
    assert lib.moe_rmsnorm(None, A, None, ctypes.c_float(1e-6), A, None) == 1
    assert lib.moe_rmsnorm(ctypes.byref(Dims(4, 100, 1, 1, 64, 64)), A, None, ctypes.c_float(1e-6), A, None) == 2
    assert lib.moe_rmsnorm(ctypes.byref(d), A, None, ctypes.c_float(-1.0), A + 0x100000, None) == 1
    assert lib.moe_rmsnorm(ctypes.byref(d), A, None, ctypes.c_float(1e-6), A + 8, None) == 3
    assert lib.moe_rmsnorm(ctypes.byref(d), A, None, ctypes.c_float(1e-6), A + 64, None) == 1  # overlap
    assert lib.moe_last_device_error(None, None) == 1
    assert lib.moe_workspace_init(None, 16, None) == 1


def test_status_strings(lib):
    for s in range(8):
        assert lib.moe_status_string(s).decode().startswith(binding.MOE_STATUS[s])
    assert b"unknown" in lib.moe_status_string(42)


def test_binding_refuses_cpu_tensors():
    import torch
    with pytest.raises(ValueError, match="GPU only"):
        binding._ptr(torch.zeros(4))


def test_unknown_flag_bits_are_rejected_before_any_launch(lib):
    # MOE_FLAG_BF16_SCORES (1) is the only flag; every entry point that routes refuses others
    w = _weights()
    for flags in (2, 1 << 30, -1):
        dims = FULL + (flags,)
        d = Dims(*dims)
        assert _forward(lib, dims=dims) == 1
        wsb = lib.moe_workspace_size(ctypes.byref(d))
        assert wsb == lib.moe_workspace_size(ctypes.byref(Dims(*FULL)))  # the size ignores flags
        assert lib.moe_route(ctypes.byref(d), A, ctypes.byref(w), A, A, A, A, A, A, wsb, None) == 1
        assert lib.moe_router_stats(ctypes.byref(d), A, ctypes.byref(w), A, A, A, A, wsb, None) == 1
        assert lib.moe_route_noalloc(ctypes.byref(d), A, ctypes.byref(w), A, A, A, A, A, None) == 1
    # the defined flag passes host validation (the call then stops at a misaligned output)
    assert _forward(lib, dims=FULL + (binding.FLAG_BF16_SCORES,), out=A + 0x200002) == 3


def test_host_experts_shadow_size_and_host_checks(lib):
    T, H, E, K, I, Is = FULL
    assert binding.moe_expert_shadow_size(FULL) == E * (2 * I * H + H * I) * 2
    assert binding.moe_expert_shadow_size((1, 2048, 256, 9, 512, 512)) == 0  # K > 8
    d = Dims(*FULL)
    w = _weights()
    wsb = lib.moe_workspace_size(ctypes.byref(d))
    sb = binding.moe_expert_shadow_size(FULL)
    call = lambda shadow, nb: lib.moe_forward_host_experts(  # noqa: E731
        ctypes.byref(d), A + 0x100000, ctypes.byref(w), None, A + 0x200000, shadow, nb, A + 0x400000, wsb, None)
    assert call(None, sb) == 1
    assert call(A + 0x800008, sb) == 3
    assert call(A + 0x800000, sb - 16) == 4


def test_host_io_host_checks(lib):
    d = Dims(*FULL)
    w = _weights()
    wsb = lib.moe_workspace_size(ctypes.byref(d))
    act = FULL[0] * FULL[1] * 2
    call = lambda hx, hout, xd, od, nb=wsb: lib.moe_forward_host_io(  # noqa: E731
        ctypes.byref(d), hx, ctypes.byref(w), None, hout, xd, od, A + 0x400000, nb, None)
    xd, od = A + 0x100000, A + 0x200000
    assert call(None, A, xd, od) == 1  # no host x
    assert call(A, None, xd, od) == 1  # no host out
    assert call(A, A, xd, None) == 1  # no device staging for out
    assert call(A, A, xd + 8, od) == 3
    assert call(A, A, xd, od + 8) == 3
    assert call(A, A, xd, xd + act - 16) == 1  # staging buffers overlap
    assert call(A, A, xd, od, wsb - 256) == 4
    # T = 0 is a no-op before any pointer is looked at
    assert lib.moe_forward_host_io(ctypes.byref(Dims(0, 2048, 256, 8, 512, 512)), None, None, None, None, None,
                                   None, None, 0, None) == 0
    with pytest.raises(ValueError, match="the layer needs"):  # a host x shorter than [T, H] bf16
        binding.moe_forward_host_io(FULL, torch.empty(4, dtype=torch.bfloat16), None, None, None, None, None, None)


def test_prepared_host_io_checks_its_tensors():
    T, H = FULL[:2]
    cpu = lambda *shape: torch.empty(*shape, dtype=torch.bfloat16)  # noqa: E731
    W = binding.Weights(router_w=cpu(4), router_b=None, gate_up=cpu(4), down=cpu(4), shared_gate_up=cpu(4),
                        shared_down=cpu(4), shared_gate=cpu(4))
    with pytest.raises(ValueError, match=r"\[T, H\]"):  # staging shorter than [T, H] bf16
        binding.ForwardHostIO(FULL, W, cpu(T, H // 2), cpu(T, H), torch.empty(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="GPU only"):  # the weights and staging must be CUDA tensors
        binding.ForwardHostIO(FULL, W, cpu(T, H), cpu(T, H), torch.empty(16, dtype=torch.uint8))


def test_wait_limit_hook_validates_its_arguments(lib):
    """The testing aid for the bounded waits takes a limit of at most 10 s and a known signal;
    anything else is rejected on the host, and the defaults are restored."""
    assert lib.moe_test_set_wait(0, 3) == 1
    assert lib.moe_test_set_wait(0, -1) == 1
    assert lib.moe_test_set_wait(10_000_000_001, 0) == 1
    assert lib.moe_test_set_wait(2_000_000, 1) == 0
    assert lib.moe_test_set_wait(2_000_000, 2) == 0
    assert lib.moe_test_set_wait(0, 0) == 0
