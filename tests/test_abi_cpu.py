"""The C-ABI library builds for sm_103a, loads without a GPU and exports every function that
include/mm.h declares. Only calls that return before touching the device are made here."""
import ctypes
import subprocess

import pytest

from moe_ffn_expert_gb300 import _abi
from moe_ffn_expert_gb300 import build as mm_build


@pytest.fixture(scope="module", autouse=True)
def built():
    mm_build.build()


def test_exports_every_header_symbol():
    names = _abi.header_symbols()
    assert len(names) >= 10
    lib = ctypes.CDLL(_abi.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert set(names) <= exported


def test_workspace_size_and_limits():
    d = _abi.dims(16384, 2048, 768, 128, 8)
    n = _abi.mm_workspace_size(d)
    S, S_pad = 16384 * 8, 16384 * 8 + 128 * 127 + 128
    assert n > S_pad * 2048 * 2 * 3  # x_slot, o, dy_slot at least
    assert n < 4 * 2 ** 30
    assert _abi.mm_workspace_size(_abi.dims(16, 60, 32, 4, 2)) == 0      # H not a multiple of 8
    assert _abi.mm_workspace_size(_abi.dims(16, 64, 36, 4, 2)) == 0      # I not a multiple of 8
    assert _abi.mm_workspace_size(_abi.dims(16, 64, 32, 1025, 2)) == 0   # E > 1024
    assert _abi.mm_workspace_size(_abi.dims(16, 64, 32, 4, 17)) == 0     # K > 16
    assert _abi.mm_workspace_size(_abi.dims(-1, 64, 32, 4, 2)) == 0     # negative T
    assert _abi.mm_workspace_size(_abi.dims(0, 64, 32, 4, 2)) > 0       # an empty batch
    assert _abi.mm_workspace_size(_abi.dims(1, 8, 8, 1, 1)) > 0


def test_host_validation_without_device():
    d = _abi.dims(16, 64, 32, 4, 2)
    n = _abi.mm_workspace_size(d)
    # null workspace / too small / null tensors are rejected before any CUDA call
    assert _abi.mm_forward(d, 0, 0, 0, 0, 0, 0, 0, n, 0, 0) == _abi.MM_ERR_WORKSPACE
    assert _abi.mm_forward(d, 16, 16, 16, 16, 16, 16, 256, n - 1, 0, 0) == _abi.MM_ERR_WORKSPACE
    assert _abi.mm_forward(d, 0, 16, 16, 16, 16, 16, 256, n, 0, 0) == _abi.MM_ERR_INVALID_ARG
    assert _abi.mm_forward(d, 24, 16, 16, 16, 16, 16, 256, n, 0, 0) == _abi.MM_ERR_INVALID_ARG
    assert _abi.mm_forward(_abi.dims(16, 60, 32, 4, 2), 16, 16, 16, 16, 16, 16, 256, n, 0, 0) == _abi.MM_ERR_UNSUPPORTED
    both = _abi.MM_FLAG_FUSED_FORWARD_GEMMS | _abi.MM_FLAG_SEPARATE_FORWARD_GEMMS  # contradictory
    assert _abi.mm_forward(d, 16, 16, 16, 16, 16, 16, 256, n, 0, both) == _abi.MM_ERR_INVALID_ARG
    assert _abi.mm_backward(d, 0, 16, 16, 16, 16, 16, 256, n, 16, 16, 16, 16, 0, 0) == _abi.MM_ERR_INVALID_ARG
    assert _abi.mm_get_status(0, 0) == _abi.MM_ERR_WORKSPACE
    assert _abi.mm_status_string(_abi.MM_ERR_BAD_EXPERT_ID) == "expert id out of range"
    assert _abi.mm_abi_version() == 3
    assert _abi.mm_status_string(_abi.MM_ERR_TOKENS_PER_EXPERT) == \
        "tokens_per_expert does not match topk_ids"


def test_extended_entry_points_host_checks():
    d = _abi.dims(16, 64, 32, 4, 2)
    n = _abi.mm_workspace_size(d)
    # no options, or empty options: the plain layout
    assert _abi.mm_workspace_size_ex(d, None) == n
    assert _abi.mm_workspace_size_ex(d, _abi.options()) == n
    # a shared expert adds its own region; its size follows the same rules as I
    ns = _abi.mm_workspace_size_ex(d, _abi.options(_abi.shared_expert(48, 0, 0)))
    assert ns > n
    assert _abi.mm_workspace_size_ex(d, _abi.options(_abi.shared_expert(96, 0, 0))) > ns
    assert _abi.mm_workspace_size_ex(d, _abi.options(_abi.shared_expert(0, 0, 0))) == 0
    assert _abi.mm_workspace_size_ex(d, _abi.options(_abi.shared_expert(36, 0, 0))) == 0
    # shared-expert weights missing or misaligned; misaligned tokens_per_expert
    se_null = _abi.options(_abi.shared_expert(48, 0, 0))
    assert _abi.mm_forward_ex(d, se_null, 16, 16, 16, 16, 16, 16, 256, ns, 0, 0) == _abi.MM_ERR_INVALID_ARG
    se_odd = _abi.options(_abi.shared_expert(48, 16, 24))
    assert _abi.mm_forward_ex(d, se_odd, 16, 16, 16, 16, 16, 16, 256, ns, 0, 0) == _abi.MM_ERR_INVALID_ARG
    se_nograd = _abi.options(_abi.shared_expert(48, 16, 16))
    assert _abi.mm_backward_ex(d, se_nograd, 16, 16, 16, 16, 16, 16, 256, ns, 16, 16, 16, 16, 0,
                               0) == _abi.MM_ERR_INVALID_ARG
    # a shared expert needs the larger workspace
    assert _abi.mm_forward_ex(d, _abi.options(_abi.shared_expert(48, 16, 16)), 16, 16, 16, 16, 16,
                              16, 256, n, 0, 0) == _abi.MM_ERR_WORKSPACE
    assert _abi.mm_forward_ex(d, _abi.options(None, 18), 16, 16, 16, 16, 16, 16, 256, n, 0,
                              0) == _abi.MM_ERR_INVALID_ARG
    # an empty batch checks the shared expert's weights as a full one does
    d0 = _abi.dims(0, 64, 32, 4, 2)
    n0 = _abi.mm_workspace_size_ex(d0, _abi.options(_abi.shared_expert(48, 16, 16)))
    for up, down in ((24, 16), (16, 24), (0, 16)):
        opt = _abi.options(_abi.shared_expert(48, up, down, 16, 16))
        assert _abi.mm_backward_ex(d0, opt, 0, 0, 0, 0, 16, 16, 256, n0, 0, 0, 16, 16, 0,
                                   0) == _abi.MM_ERR_INVALID_ARG, (up, down)
        assert _abi.mm_forward_ex(d0, opt, 0, 0, 0, 16, 16, 0, 256, n0, 0,
                                  0) == _abi.MM_ERR_INVALID_ARG, (up, down)


def test_stage_table():
    names = [_abi._lib().mm_stage_name(i).decode() for i in range(_abi.MM_NUM_STAGES)]
    assert names[0] == "route_count" and names[-1] == "wgrad_reduce" and len(set(names)) == 17
    assert _abi.mm_timing_read() == {n: (0.0, 0) for n in names}


def test_python_constants_match_the_header():
    """Every MM_FLAG_* / MM_NUM_STAGES define and every status enumerator of include/mm.h has a
    twin of the same name and value in the Python binding."""
    import os
    import re
    text = open(os.path.join(os.path.dirname(_abi.__file__), os.pardir, "include", "mm.h")).read()
    found = {}
    for name, value in re.findall(r"#define\s+(MM_(?:FLAG_\w+|NUM_STAGES))\s+(0x[0-9a-fA-F]+|\d+)u?", text):
        found[name] = int(value, 0)
    for name, value in re.findall(r"\b(MM_(?:OK|ERR_\w+))\s*=\s*(\d+)", text):
        found[name] = int(value)
    assert len(found) >= 17
    for name, value in found.items():
        assert getattr(_abi, name) == value, name


def test_c_example_builds_against_the_header(tmp_path):
    """tests/c_abi/layer_step.c (a layer step through the C ABI alone) compiles with the host C
    compiler against include/mm.h and links against libmm.so; it runs in the GPU tests."""
    from c_abi_util import build_layer_step
    exe = build_layer_step(str(tmp_path))
    import os
    assert os.access(exe, os.X_OK)
