"""Python binding of libqre.so: the quantized routed-expert MoE layer for GB300.

Argument marshalling only.  Every function has the name of the C entry point it
calls (declared in ``include/qre.h``); every step of the layer runs in the
library's CUDA kernels.  Tensor arguments may be ``torch.Tensor`` (their
``data_ptr()`` is passed), plain integer addresses, or ``None`` for NULL.  The
stream defaults to torch's current CUDA stream.  A non-zero status raises
:class:`QreError` carrying the library's message.

There is no fallback: if ``libqre.so`` has not been built, importing works but
the first call raises, naming the build command.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqre.so")

QRE_OK = 0
QRE_ERR_INVALID_ARG = 1
QRE_ERR_UNSUPPORTED = 2
QRE_ERR_MISALIGNED = 3
QRE_ERR_WORKSPACE = 4
QRE_ERR_CUDA = 5
QRE_ERR_TIMEOUT = 6
QRE_ERR_DEVICE_CHECK = 7

QRE_DEV_TIMEOUT = 0x1
QRE_DEV_NULL_SLOT = 0x2
QRE_DEV_BAD_SCALE = 0x4
QRE_DEV_BAD_INDEX = 0x8
QRE_DEV_FP16_RANGE = 0x10

# Every symbol include/qre.h declares.
EXPORTS = (
    "qre_last_error", "qre_status_string", "qre_version", "qre_workspace_size", "qre_quantize",
    "qre_quantize_gate_up",
    "qre_route", "qre_dispatch", "qre_expert_ffn", "qre_combine", "qre_validate_slots",
    "qre_cache_update", "qre_cache_copy",
    "qre_read_device_status", "qre_clear_device_status", "qre_route_noalloc", "qre_debug_wait_test",
    "qre_expert_ffn_routed", "qre_expert_ffn_shared", "qre_shared_workspace_size", "qre_stage_experts",
    "qre_read_probe", "qre_set_host_unit_cost", "qre_route_dispatch",
)


class qre_layer_shape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("group", ctypes.c_int32)]


class qre_slot(ctypes.Structure):
    _fields_ = [("w_gate_up", ctypes.c_void_p), ("s_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("s_down", ctypes.c_void_p), ("tier", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class QreError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)}: {message}")


_STATUS_NAMES = {0: "QRE_OK", 1: "QRE_ERR_INVALID_ARG", 2: "QRE_ERR_UNSUPPORTED", 3: "QRE_ERR_MISALIGNED",
                 4: "QRE_ERR_WORKSPACE", 5: "QRE_ERR_CUDA", 6: "QRE_ERR_TIMEOUT", 7: "QRE_ERR_DEVICE_CHECK"}

_lib = None

_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_SHAPE = ctypes.POINTER(qre_layer_shape)
_SIGS = {
    "qre_last_error": ([], ctypes.c_char_p),
    "qre_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "qre_version": ([], ctypes.c_int32),
    "qre_workspace_size": ([_SHAPE, _I32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "qre_quantize": ([_I32, _I32, _I32, _VP, _VP, _VP, _VP], ctypes.c_int),
    "qre_quantize_gate_up": ([_I32, _I32, _I32, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "qre_route": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], ctypes.c_int),
    "qre_dispatch": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], ctypes.c_int),
    "qre_expert_ffn": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], ctypes.c_int),
    "qre_combine": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "qre_validate_slots": ([_SHAPE, ctypes.POINTER(qre_slot)], ctypes.c_int),
    "qre_cache_update": ([_SHAPE, _I32, ctypes.c_float, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP],
                         ctypes.c_int),
    "qre_cache_copy": ([_SHAPE, _VP, _VP, _VP, _VP, _I32, _VP], ctypes.c_int),
    "qre_read_device_status": ([_VP, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
    "qre_clear_device_status": ([_VP], ctypes.c_int),
    "qre_route_noalloc": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "qre_debug_wait_test": ([ctypes.c_uint64, ctypes.c_uint64], ctypes.c_int),
    "qre_expert_ffn_routed": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], ctypes.c_int),
    "qre_expert_ffn_shared": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _SZ, _VP], ctypes.c_int),
    "qre_shared_workspace_size": ([_SHAPE, _I32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "qre_stage_experts": ([_SHAPE, ctypes.POINTER(qre_slot), ctypes.POINTER(qre_slot), _I32, _VP, _VP,
                           ctypes.POINTER(ctypes.c_int32), _VP], ctypes.c_int),
    "qre_read_probe": ([_VP, _SZ, _VP, _VP], ctypes.c_int),
    "qre_set_host_unit_cost": ([_I32], ctypes.c_int),
    "qre_route_dispatch": ([_SHAPE, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP],
                           ctypes.c_int),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libqre.so (once) and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m quantized_routed_expert_03_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str) -> None:
    if status != QRE_OK:
        raise QreError(status, where, load_library().qre_last_error().decode())


def _nbytes(t, given):
    if given is not None:
        return given
    if t is None:
        return 0
    return t.numel() * t.element_size()


def make_shape(hidden: int, inter: int, n_experts: int, top_k: int, group: int) -> qre_layer_shape:
    return qre_layer_shape(hidden, inter, n_experts, top_k, group)


def qre_version() -> int:
    return load_library().qre_version()


def qre_status_string(status: int) -> str:
    return load_library().qre_status_string(status).decode()


def qre_last_error() -> str:
    return load_library().qre_last_error().decode()


def qre_workspace_size(shape: qre_layer_shape, T: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().qre_workspace_size(ctypes.byref(shape), T, ctypes.byref(out)), "qre_workspace_size")
    return out.value


def qre_quantize(n_rows, k_dim, group, w, packed, scales, stream=None) -> None:
    _check(load_library().qre_quantize(n_rows, k_dim, group, _ptr(w), _ptr(packed), _ptr(scales),
                                       _stream(stream)), "qre_quantize")


def qre_quantize_gate_up(inter, hidden, group, w_gate, w_up, packed, scales, stream=None) -> None:
    _check(load_library().qre_quantize_gate_up(inter, hidden, group, _ptr(w_gate), _ptr(w_up), _ptr(packed),
                                               _ptr(scales), _stream(stream)), "qre_quantize_gate_up")


def qre_route(shape, T, x_bf16, w_router, bias, topk_idx, topk_w, workspace, workspace_bytes=None,
              stream=None) -> None:
    _check(load_library().qre_route(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(w_router), _ptr(bias),
                                    _ptr(topk_idx), _ptr(topk_w), _ptr(workspace),
                                    _nbytes(workspace, workspace_bytes), _stream(stream)), "qre_route")


def qre_route_noalloc(shape, T, x_bf16, w_router, bias, topk_idx, topk_w, stream=None) -> None:
    """qre_route for callers that cannot allocate device memory: the logits scratch
    is a fixed array inside the library (T * n_experts <= 65,536)."""
    _check(load_library().qre_route_noalloc(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(w_router), _ptr(bias),
                                            _ptr(topk_idx), _ptr(topk_w), _stream(stream)), "qre_route_noalloc")


def qre_route_dispatch(shape, T, x_bf16, w_router, bias, topk_idx, topk_w, counts, offsets, perm, inv_perm, active,
                       n_active, workspace, workspace_bytes=None, stream=None) -> None:
    _check(load_library().qre_route_dispatch(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(w_router), _ptr(bias),
                                             _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(perm),
                                             _ptr(inv_perm), _ptr(active), _ptr(n_active), _ptr(workspace),
                                             _nbytes(workspace, workspace_bytes), _stream(stream)),
           "qre_route_dispatch")


def qre_dispatch(shape, T, topk_idx, counts, offsets, perm, inv_perm, active, n_active, workspace,
                 workspace_bytes=None, stream=None) -> None:
    _check(load_library().qre_dispatch(ctypes.byref(shape), T, _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                       _ptr(perm), _ptr(inv_perm), _ptr(active), _ptr(n_active),
                                       _ptr(workspace), _nbytes(workspace, workspace_bytes), _stream(stream)),
           "qre_dispatch")


def qre_expert_ffn(shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out, workspace,
                   workspace_bytes=None, stream=None) -> None:
    _check(load_library().qre_expert_ffn(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(slots), _ptr(offsets),
                                         _ptr(perm), _ptr(active), _ptr(n_active), _ptr(expert_out),
                                         _ptr(workspace), _nbytes(workspace, workspace_bytes), _stream(stream)),
           "qre_expert_ffn")


def qre_expert_ffn_routed(shape, T, x_bf16, slots, offsets, perm, active, n_active, expert_out, workspace,
                          workspace_bytes=None, stream=None) -> None:
    _check(load_library().qre_expert_ffn_routed(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(slots), _ptr(offsets),
                                                _ptr(perm), _ptr(active), _ptr(n_active), _ptr(expert_out),
                                                _ptr(workspace), _nbytes(workspace, workspace_bytes),
                                                _stream(stream)), "qre_expert_ffn_routed")


def qre_expert_ffn_shared(shape, T, x_bf16, slots, expert_out, workspace, workspace_bytes=None,
                          stream=None) -> None:
    _check(load_library().qre_expert_ffn_shared(ctypes.byref(shape), T, _ptr(x_bf16), _ptr(slots),
                                                _ptr(expert_out), _ptr(workspace),
                                                _nbytes(workspace, workspace_bytes), _stream(stream)),
           "qre_expert_ffn_shared")


def qre_shared_workspace_size(shape: qre_layer_shape, T: int) -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().qre_shared_workspace_size(ctypes.byref(shape), T, ctypes.byref(out)),
           "qre_shared_workspace_size")
    return out.value


def qre_combine(shape, T, expert_out, topk_w, inv_perm, y_f32, y_bf16, stream=None) -> None:
    _check(load_library().qre_combine(ctypes.byref(shape), T, _ptr(expert_out), _ptr(topk_w), _ptr(inv_perm),
                                       _ptr(y_f32), _ptr(y_bf16), _stream(stream)), "qre_combine")


def qre_cache_update(shape, n_slots, decay, active, n_active, scores, expert_slot, slot_expert, home, slot_mem,
                     table, copy_list, n_copies, max_copies, stream=None) -> None:
    _check(load_library().qre_cache_update(ctypes.byref(shape), n_slots, decay, _ptr(active), _ptr(n_active),
                                           _ptr(scores), _ptr(expert_slot), _ptr(slot_expert), _ptr(home),
                                           _ptr(slot_mem), _ptr(table), _ptr(copy_list), _ptr(n_copies),
                                           max_copies, _stream(stream)), "qre_cache_update")


def qre_cache_copy(shape, home, slot_mem, copy_list, n_copies, max_copies, stream=None) -> None:
    _check(load_library().qre_cache_copy(ctypes.byref(shape), _ptr(home), _ptr(slot_mem), _ptr(copy_list),
                                         _ptr(n_copies), max_copies, _stream(stream)), "qre_cache_copy")


def qre_stage_experts(shape, host_table, host_staging, host_out, table_out, stream=None) -> int:
    """Stages the host-resident experts of ``host_table`` (ctypes qre_slot array) into
    ``host_staging`` slots; ``host_out``: a host buffer of (E + 1) qre_slot (an int
    address or a tensor, kept alive until the stream passes the call); returns the
    number of experts staged."""
    n = ctypes.c_int32(0)
    _check(load_library().qre_stage_experts(ctypes.byref(shape), host_table, host_staging, len(host_staging),
                                            _ptr(host_out), _ptr(table_out), ctypes.byref(n), _stream(stream)),
           "qre_stage_experts")
    return n.value


def qre_read_probe(src, nbytes, sink, stream=None) -> None:
    """One streaming read of ``nbytes`` at ``src`` (device or host-mapped); time it with events."""
    _check(load_library().qre_read_probe(_ptr(src), nbytes, _ptr(sink), _stream(stream)), "qre_read_probe")


def qre_validate_slots(shape, host_slots) -> None:
    """host_slots: a ctypes array of qre_slot (n_experts + 1 entries) in host memory."""
    _check(load_library().qre_validate_slots(ctypes.byref(shape), host_slots), "qre_validate_slots")


def qre_debug_wait_test(wait_limit_ns: int, stall_ns: int) -> None:
    """Test hook: lower the kernels' wait limit and delay one warp of the expert
    FFN's first CTA, so that the give-up path runs (0, 0 restores the defaults)."""
    _check(load_library().qre_debug_wait_test(wait_limit_ns, stall_ns), "qre_debug_wait_test")


def qre_set_host_unit_cost(cost: int) -> None:
    """Process-wide: cut the decode kernels' work at equal cost with a host-mapped
    unit counted as ``cost`` (0 or 1: equal counts, the default)."""
    _check(load_library().qre_set_host_unit_cost(cost), "qre_set_host_unit_cost")


def qre_read_device_status(stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(load_library().qre_read_device_status(_stream(stream), ctypes.byref(out)), "qre_read_device_status")
    return out.value


def qre_clear_device_status(stream=None) -> None:
    _check(load_library().qre_clear_device_status(_stream(stream)), "qre_clear_device_status")


def slot_array(entries) -> ctypes.Array:
    """Host ctypes array of qre_slot from (w_gate_up, s_gate_up, w_down, s_down, tier) tuples of addresses."""
    arr = (qre_slot * len(entries))()
    for i, (wg, sg, wd, sd, tier) in enumerate(entries):
        arr[i] = qre_slot(_ptr(wg), _ptr(sg), _ptr(wd), _ptr(sd), tier, 0)
    return arr
