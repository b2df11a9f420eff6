"""ctypes binding of the C ABI declared in include/mm.h (libmm.so, built in-tree).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
Pointers are plain integers (device addresses, or host addresses where the header allows),
`stream` is a cudaStream_t as an integer (0 = legacy default stream).
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmm.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mm.h")

MM_OK = 0
MM_ERR_INVALID_ARG = 1
MM_ERR_UNSUPPORTED = 2
MM_ERR_WORKSPACE = 3
MM_ERR_CUDA = 4
MM_ERR_BAD_EXPERT_ID = 5
MM_ERR_TIMEOUT = 6
MM_ERR_TOKENS_PER_EXPERT = 7
MM_FLAG_VALIDATE_IDS = 0x1
MM_FLAG_TEST_STALL = 0x80000000
MM_FLAG_ACCUMULATE_WEIGHT_GRADS = 0x2
MM_FLAG_FP32_WEIGHT_GRADS = 0x4
MM_FLAG_FUSED_FORWARD_GEMMS = 0x8
MM_FLAG_FUSED_COMBINE = 0x10
MM_FLAG_FORWARD_ONLY = 0x20
MM_FLAG_SEPARATE_FORWARD_GEMMS = 0x40
MM_FLAG_SINGLE_CTA_TILES = 0x100
MM_NUM_STAGES = 17
MM_TRACE_CTA = 0
MM_TRACE_MAINLOOP = 1
MM_TRACE_EPILOGUE = 2
TRACE_RECORD_BYTES = 32  # sizeof(mm_trace_record); the buffer's header takes one record's bytes

STATUS_NAMES = {0: "MM_OK", 1: "MM_ERR_INVALID_ARG", 2: "MM_ERR_UNSUPPORTED", 3: "MM_ERR_WORKSPACE",
                4: "MM_ERR_CUDA", 5: "MM_ERR_BAD_EXPERT_ID", 6: "MM_ERR_TIMEOUT",
                7: "MM_ERR_TOKENS_PER_EXPERT"}


class MMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = _lib().mm_last_error_detail().decode() if status == MM_ERR_CUDA else ""
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({_lib().mm_status_string(status).decode()}){' ' + detail if detail else ''}")


class mm_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("K", ctypes.c_int64)]


class mm_shared_expert(ctypes.Structure):
    _fields_ = [("I", ctypes.c_int64), ("up_proj_weight", ctypes.c_void_p),
                ("down_proj_weight", ctypes.c_void_p), ("d_up_proj_weight", ctypes.c_void_p),
                ("d_down_proj_weight", ctypes.c_void_p)]


class mm_options(ctypes.Structure):
    _fields_ = [("shared", ctypes.POINTER(mm_shared_expert)),
                ("tokens_per_expert", ctypes.c_void_p)]


_P = ctypes.c_void_p
_LIB = None


def _lib():
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run `python -m moe_ffn_expert_gb300.build`)")
    lib = ctypes.CDLL(LIB_PATH)
    st = ctypes.c_int
    sig = {
        "mm_workspace_size": (ctypes.c_size_t, [mm_dims, ctypes.c_uint32]),
        "mm_forward": (st, [mm_dims, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_uint32]),
        "mm_backward": (st, [mm_dims, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P, _P, _P,
                             _P, ctypes.c_uint32]),
        "mm_workspace_size_ex": (ctypes.c_size_t, [mm_dims, ctypes.POINTER(mm_options),
                                                   ctypes.c_uint32]),
        "mm_forward_ex": (st, [mm_dims, ctypes.POINTER(mm_options), _P, _P, _P, _P, _P, _P,
                               _P, ctypes.c_size_t, _P, ctypes.c_uint32]),
        "mm_backward_ex": (st, [mm_dims, ctypes.POINTER(mm_options), _P, _P, _P, _P, _P, _P,
                                _P, ctypes.c_size_t, _P, _P, _P, _P, _P, ctypes.c_uint32]),
        "mm_get_status": (st, [_P, _P]),
        "mm_routing_export": (st, [mm_dims, _P, _P, _P, _P, _P]),
        "mm_status_string": (ctypes.c_char_p, [st]),
        "mm_abi_version": (ctypes.c_int, []),
        "mm_last_error_detail": (ctypes.c_char_p, []),
        "mm_timing_enable": (st, [ctypes.c_int]),
        "mm_timing_select": (st, [ctypes.c_uint32]),
        "mm_timing_read": (ctypes.c_int, [_P, _P, ctypes.c_int]),
        "mm_stage_name": (ctypes.c_char_p, [ctypes.c_int]),
        "mm_route_noalloc": (st, [mm_dims, _P, _P, _P, _P, _P]),
        "mm_trace_set": (st, [_P, ctypes.c_size_t]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def header_symbols() -> list[str]:
    """Function names declared in include/mm.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(mm_\w+)\s*\(", text, re.M)))


def dims(T, H, I, E, K) -> mm_dims:
    return mm_dims(int(T), int(H), int(I), int(E), int(K))


def mm_workspace_size(d: mm_dims, flags: int = 0) -> int:
    return int(_lib().mm_workspace_size(d, flags))


def mm_forward(d, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y, workspace,
               workspace_bytes, stream=0, flags=0) -> int:
    return int(_lib().mm_forward(d, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y,
                                 workspace, workspace_bytes, stream, flags))


def mm_backward(d, dy, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, workspace,
                workspace_bytes, dx, d_topk_weights, d_up_proj_weight, d_down_proj_weight,
                stream=0, flags=0) -> int:
    return int(_lib().mm_backward(d, dy, x, topk_ids, topk_weights, up_proj_weight,
                                  down_proj_weight, workspace, workspace_bytes, dx, d_topk_weights,
                                  d_up_proj_weight, d_down_proj_weight, stream, flags))


def shared_expert(I, up_proj_weight, down_proj_weight, d_up_proj_weight=0, d_down_proj_weight=0):
    return mm_shared_expert(int(I), up_proj_weight, down_proj_weight, d_up_proj_weight,
                            d_down_proj_weight)


def options(shared=None, tokens_per_expert=0) -> mm_options:
    """An mm_options; `shared` is an mm_shared_expert (kept alive by the returned object)."""
    o = mm_options(ctypes.pointer(shared) if shared is not None else None, tokens_per_expert or None)
    o._keep = shared
    return o


def _opt(opt):
    return ctypes.byref(opt) if opt is not None else None


def mm_workspace_size_ex(d: mm_dims, opt=None, flags: int = 0) -> int:
    return int(_lib().mm_workspace_size_ex(d, _opt(opt), flags))


def mm_forward_ex(d, opt, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y,
                  workspace, workspace_bytes, stream=0, flags=0) -> int:
    return int(_lib().mm_forward_ex(d, _opt(opt), x, topk_ids, topk_weights, up_proj_weight,
                                    down_proj_weight, y, workspace, workspace_bytes, stream, flags))


def mm_backward_ex(d, opt, dy, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                   workspace, workspace_bytes, dx, d_topk_weights, d_up_proj_weight,
                   d_down_proj_weight, stream=0, flags=0) -> int:
    return int(_lib().mm_backward_ex(d, _opt(opt), dy, x, topk_ids, topk_weights,
                                     up_proj_weight, down_proj_weight, workspace, workspace_bytes,
                                     dx, d_topk_weights, d_up_proj_weight, d_down_proj_weight,
                                     stream, flags))


def mm_get_status(workspace, stream=0) -> int:
    return int(_lib().mm_get_status(workspace, stream))


def mm_routing_export(d, workspace, counts, offsets, row_of_slot, stream=0) -> int:
    return int(_lib().mm_routing_export(d, workspace, counts, offsets, row_of_slot, stream))


def mm_route_noalloc(d, topk_ids, counts, offsets, row_of_slot, stream=0) -> int:
    return int(_lib().mm_route_noalloc(d, topk_ids, counts, offsets, row_of_slot, stream))


def mm_status_string(status: int) -> str:
    return _lib().mm_status_string(status).decode()


def mm_abi_version() -> int:
    return int(_lib().mm_abi_version())


def mm_timing_enable(on: bool) -> int:
    return int(_lib().mm_timing_enable(1 if on else 0))


def mm_timing_select(stage_mask: int) -> int:
    return int(_lib().mm_timing_select(stage_mask & 0xFFFFFFFF))


def stage_index(name: str) -> int:
    for i in range(MM_NUM_STAGES):
        if _lib().mm_stage_name(i).decode() == name:
            return i
    raise KeyError(name)


def mm_timing_read() -> dict:
    """{stage name: (milliseconds, launches)} since the last read."""
    ms = (ctypes.c_double * MM_NUM_STAGES)()
    cnt = (ctypes.c_int64 * MM_NUM_STAGES)()
    n = _lib().mm_timing_read(ctypes.cast(ms, _P), ctypes.cast(cnt, _P), MM_NUM_STAGES)
    return {_lib().mm_stage_name(i).decode(): (ms[i], cnt[i]) for i in range(n)}


def mm_trace_set(device_buffer, nbytes: int) -> int:
    """Sets (device_buffer = 0: clears) the trace buffer; see moe_ffn_expert_gb300.trace."""
    return int(_lib().mm_trace_set(device_buffer or None, int(nbytes)))


def check(status: int, where: str):
    if status != MM_OK:
        raise MMError(status, where)
