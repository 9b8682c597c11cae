"""Python binding of libmxfp4.so (the C ABI in include/mxfp4.h and include/q4k.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library.  Tensors are torch CUDA tensors (device memory and
streams are PyTorch's); the functions take the same names and arguments as the
C entry points, with `stream` defaulting to torch's current stream.  There is
no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "Mxfp4Error", "lib", "library_path", "mxfp4_nbytes", "mxfp4_device_faults",
    "mxfp4_set_launch_overlap", "mxfp4_dequant", "mxfp4_mv",
    "mxfp4_mm", "mxfp4_mm_fp32", "mxfp4_mm_bf16", "mxfp4_mm_bf16_workspace_bytes",
    "mxfp4_mm_bf16_ws", "mxfp4_matmat_host",
    "mxfp4_moe_workspace_bytes", "mxfp4_moe_gate_up", "mxfp4_moe_down",
    "mxfp4_moe_plan_errors", "mxfp4_moe_layer_noalloc", "mxfp4_moe_gate_up_ex",
    "mxfp4_moe_down_ex", "mxfp4_moe_cold_pairs", "mxfp4_moe_gate_up_seg", "mxfp4_moe_down_seg",
    "MOE_MODE_F32", "MOE_MODE_V41", "q4k_nbytes", "q4k_dequant", "q4k_mv", "q4k_mm",
    "mxfp4_status_string", "MM_SMALL_MAX", "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libmxfp4.so")
MM_SMALL_MAX = 64
MOE_MODE_F32 = 0
MOE_MODE_V41 = 1

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIG = {
    "mxfp4_status_string": (ctypes.c_char_p, [_I]),
    "mxfp4_last_cuda_error": (_I, []),
    "mxfp4_version": (_I, []),
    "mxfp4_set_launch_overlap": (_I, [_I]),
    "mxfp4_device_faults": (_I, [ctypes.POINTER(_I), _I]),
    "mxfp4_nbytes": (_SZ, [_I, _I]),
    "mxfp4_dequant": (_I, [_P, _I, _I, _P, _P]),
    "mxfp4_mv": (_I, [_P, _I, _I, _P, _P, _P]),
    "mxfp4_mm": (_I, [_P, _I, _I, _P, _I, _P, _P]),
    "mxfp4_mm_fp32": (_I, [_P, _I, _I, _P, _I, _P, _P]),
    "mxfp4_mm_bf16": (_I, [_P, _I, _I, _P, _I, _P, _P]),
    "mxfp4_mm_bf16_workspace_bytes": (_SZ, [_I, _I, _I]),
    "mxfp4_mm_bf16_ws": (_I, [_P, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "mxfp4_matmat_host": (_I, [_P, _I, _I, _P, _I, _P, _P, _P, _P]),
    "mxfp4_moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "mxfp4_moe_gate_up": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _SZ, _P]),
    "mxfp4_moe_down": (_I, [_P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "mxfp4_moe_plan_errors": (_I, [_P, _SZ, ctypes.POINTER(_I), _P]),
    "mxfp4_moe_layer_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P]),
    "mxfp4_moe_gate_up_ex": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _P, _P, _I, _P, _I,
                                  ctypes.c_float, _P, _P, _SZ, _P]),
    "mxfp4_moe_down_ex": (_I, [_P, _I, _I, _I, _P, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "mxfp4_moe_cold_pairs": (_I, [_P, _SZ, _I, _I, _I, ctypes.POINTER(_I), _P, _I, _P]),
    "mxfp4_moe_gate_up_seg": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _I, _P, _P, _I, _P, _I,
                                   ctypes.c_float, _P, _P, _SZ, _P]),
    "mxfp4_moe_down_seg": (_I, [_P, _I, _I, _I, _I, _P, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    # the second codec (include/q4k.h)
    "q4k_nbytes": (_SZ, [_I, _I]),
    "q4k_dequant": (_I, [_P, _I, _I, _P, _P]),
    "q4k_mv": (_I, [_P, _I, _I, _P, _P, _P]),
    "q4k_mm": (_I, [_P, _I, _I, _P, _I, _P, _P]),
}
EXPORTED_SYMBOLS = tuple(_SIG)
_lib = None


class Mxfp4Error(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn}: status {status} ({mxfp4_status_string(status)})"
        if cuda_error:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


def lib():
    """The loaded library; raises if it was not built (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing: build it with __graft_entry__.build() "
                "(there is no CPU fallback)")
        h = ctypes.CDLL(library_path)
        for name, (res, args) in _SIG.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def mxfp4_status_string(status: int) -> str:
    return lib().mxfp4_status_string(status).decode()


def _addr(t) -> int | None:
    """Device address of a tensor (or an int address / None passed through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        err = lib().mxfp4_last_cuda_error() if status == 3 else 0
        raise Mxfp4Error(fn, status, err)


def mxfp4_device_faults(reset: bool = False) -> int:
    v = ctypes.c_int(0)
    _check("mxfp4_device_faults", lib().mxfp4_device_faults(ctypes.byref(v), int(reset)))
    return v.value


def mxfp4_set_launch_overlap(enable: bool) -> None:
    """Programmatic dependent launch for mxfp4_mv / mxfp4_mm (see include/mxfp4.h):
    only when nothing still running in the stream writes the weight buffers."""
    _check("mxfp4_set_launch_overlap", lib().mxfp4_set_launch_overlap(int(bool(enable))))


def mxfp4_nbytes(rows: int, cols: int) -> int:
    return int(lib().mxfp4_nbytes(rows, cols))


def mxfp4_dequant(w, rows, cols, out, stream=None):
    _check("mxfp4_dequant", lib().mxfp4_dequant(_addr(w), rows, cols, _addr(out),
                                                _stream(stream)))


def mxfp4_mv(w, rows, cols, x, y, stream=None):
    _check("mxfp4_mv", lib().mxfp4_mv(_addr(w), rows, cols, _addr(x), _addr(y),
                                      _stream(stream)))


def mxfp4_mm(w, rows, cols, X, nb, Y, stream=None):
    _check("mxfp4_mm", lib().mxfp4_mm(_addr(w), rows, cols, _addr(X), nb, _addr(Y),
                                      _stream(stream)))


def mxfp4_mm_fp32(w, rows, cols, X, nb, Y, stream=None):
    _check("mxfp4_mm_fp32", lib().mxfp4_mm_fp32(_addr(w), rows, cols, _addr(X), nb,
                                                _addr(Y), _stream(stream)))


def mxfp4_mm_bf16(w, rows, cols, X, nb, Y, stream=None):
    _check("mxfp4_mm_bf16", lib().mxfp4_mm_bf16(_addr(w), rows, cols, _addr(X), nb,
                                                _addr(Y), _stream(stream)))


def mxfp4_mm_bf16_workspace_bytes(rows, cols, nb) -> int:
    return int(lib().mxfp4_mm_bf16_workspace_bytes(rows, cols, nb))


def mxfp4_mm_bf16_ws(w, rows, cols, X, nb, Y, workspace, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("mxfp4_mm_bf16_ws", lib().mxfp4_mm_bf16_ws(_addr(w), rows, cols, _addr(X), nb,
                                                      _addr(Y), _addr(workspace), ws_bytes,
                                                      _stream(stream)))


def mxfp4_matmat_host(w, rows, cols, X_host, nb, Y_host, x_dev, y_dev, stream=None):
    """X_host / Y_host: host tensors or numpy arrays (pinned memory copies
    asynchronously); synchronises the stream before returning."""
    def host_addr(a):
        if hasattr(a, "data_ptr"):
            return a.data_ptr()
        return a.ctypes.data
    _check("mxfp4_matmat_host", lib().mxfp4_matmat_host(
        _addr(w), rows, cols, host_addr(X_host), nb, host_addr(Y_host), _addr(x_dev),
        _addr(y_dev), _stream(stream)))


def mxfp4_moe_workspace_bytes(n_experts, n_tokens, top_k, hidden, inter) -> int:
    return int(lib().mxfp4_moe_workspace_bytes(n_experts, n_tokens, top_k, hidden, inter))


def mxfp4_moe_gate_up(gate_bank, up_bank, n_experts, hidden, inter, x, n_tokens, top_k,
                      expert_ids, act, workspace, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("mxfp4_moe_gate_up", lib().mxfp4_moe_gate_up(
        _addr(gate_bank), _addr(up_bank), n_experts, hidden, inter, _addr(x), n_tokens, top_k,
        _addr(expert_ids), _addr(act), _addr(workspace), ws_bytes, _stream(stream)))


def mxfp4_moe_down(down_bank, n_experts, hidden, inter, act, n_tokens, top_k, expert_ids,
                   route_w, y, workspace, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("mxfp4_moe_down", lib().mxfp4_moe_down(
        _addr(down_bank), n_experts, hidden, inter, _addr(act), n_tokens, top_k,
        _addr(expert_ids), _addr(route_w), _addr(y), _addr(workspace), ws_bytes,
        _stream(stream)))


def mxfp4_moe_plan_errors(workspace, ws_bytes=None, stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    n = ctypes.c_int(0)
    _check("mxfp4_moe_plan_errors", lib().mxfp4_moe_plan_errors(
        _addr(workspace), ws_bytes, ctypes.byref(n), _stream(stream)))
    return n.value


NOALLOC_SCRATCH_BYTES = 16 << 20


def mxfp4_moe_layer_noalloc(gate_bank, up_bank, down_bank, n_experts, hidden, inter, x,
                            n_tokens, top_k, expert_ids, route_w, y, stream=None):
    """The whole routed-expert layer with its scratch in the library's own
    fixed device array (no workspace argument, nothing allocated)."""
    _check("mxfp4_moe_layer_noalloc", lib().mxfp4_moe_layer_noalloc(
        _addr(gate_bank), _addr(up_bank), _addr(down_bank), n_experts, hidden, inter, _addr(x),
        n_tokens, top_k, _addr(expert_ids), _addr(route_w), _addr(y), _stream(stream)))


def mxfp4_moe_gate_up_ex(gate_bank, up_bank, n_slots, hidden, inter, x, n_tokens, top_k,
                         expert_ids, act, workspace, slot_of=None, n_experts=None, route_w=None,
                         mode=MOE_MODE_F32, swiglu_limit=0.0, ws_bytes=None, stream=None):
    """Gate/up pass with the global-bank options (see include/mxfp4.h)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    n_experts = n_slots if n_experts is None else n_experts
    _check("mxfp4_moe_gate_up_ex", lib().mxfp4_moe_gate_up_ex(
        _addr(gate_bank), _addr(up_bank), n_slots, hidden, inter, _addr(x), n_tokens, top_k,
        _addr(expert_ids), _addr(slot_of), n_experts, _addr(route_w), int(mode),
        float(swiglu_limit), _addr(act), _addr(workspace), ws_bytes, _stream(stream)))


def mxfp4_moe_down_ex(down_bank, n_slots, hidden, inter, act, n_tokens, top_k, y, workspace,
                      route_w=None, mode=MOE_MODE_F32, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check("mxfp4_moe_down_ex", lib().mxfp4_moe_down_ex(
        _addr(down_bank), n_slots, hidden, inter, _addr(act), n_tokens, top_k, _addr(route_w),
        int(mode), _addr(y), _addr(workspace), ws_bytes, _stream(stream)))


def mxfp4_moe_cold_pairs(workspace, n_slots, n_tokens, top_k, ws_bytes=None, stream=None):
    """The plan's cold pairs (increasing pair indices) as a list."""
    import numpy as np
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    cap = n_tokens * top_k
    buf = np.zeros(cap, dtype=np.int32)
    n = ctypes.c_int(0)
    _check("mxfp4_moe_cold_pairs", lib().mxfp4_moe_cold_pairs(
        _addr(workspace), ws_bytes, n_slots, n_tokens, top_k, ctypes.byref(n),
        buf.ctypes.data, cap, _stream(stream)))
    return buf[:n.value].tolist()


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[_addr(t) for t in tensors])
    return arr


def mxfp4_moe_gate_up_seg(gate_segments, up_segments, segment_slots, hidden, inter, x, n_tokens,
                          top_k, expert_ids, act, workspace, slot_of=None, n_experts=None,
                          route_w=None, mode=MOE_MODE_F32, swiglu_limit=0.0, ws_bytes=None,
                          stream=None):
    """Gate/up pass on a bank in segments (lists of device tensors, one per segment)."""
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    n_seg = len(gate_segments)
    n_experts = n_seg * segment_slots if n_experts is None else n_experts
    g, u = _ptr_array(gate_segments), _ptr_array(up_segments)
    _check("mxfp4_moe_gate_up_seg", lib().mxfp4_moe_gate_up_seg(
        ctypes.cast(g, _P), ctypes.cast(u, _P), n_seg, segment_slots, hidden, inter, _addr(x),
        n_tokens, top_k, _addr(expert_ids), _addr(slot_of), n_experts, _addr(route_w), int(mode),
        float(swiglu_limit), _addr(act), _addr(workspace), ws_bytes, _stream(stream)))


def mxfp4_moe_down_seg(down_segments, segment_slots, hidden, inter, act, n_tokens, top_k, y,
                       workspace, route_w=None, mode=MOE_MODE_F32, ws_bytes=None, stream=None):
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    d = _ptr_array(down_segments)
    _check("mxfp4_moe_down_seg", lib().mxfp4_moe_down_seg(
        ctypes.cast(d, _P), len(down_segments), segment_slots, hidden, inter, _addr(act), n_tokens,
        top_k, _addr(route_w), int(mode), _addr(y), _addr(workspace), ws_bytes, _stream(stream)))


# --- the second codec: GGUF Q4_K (include/q4k.h) --------------------------------

def q4k_nbytes(rows: int, cols: int) -> int:
    return int(lib().q4k_nbytes(rows, cols))


def q4k_dequant(w, rows, cols, out, stream=None):
    _check("q4k_dequant", lib().q4k_dequant(_addr(w), rows, cols, _addr(out),
                                            _stream(stream)))


def q4k_mv(w, rows, cols, x, y, stream=None):
    _check("q4k_mv", lib().q4k_mv(_addr(w), rows, cols, _addr(x), _addr(y), _stream(stream)))


def q4k_mm(w, rows, cols, X, nb, Y, stream=None):
    _check("q4k_mm", lib().q4k_mm(_addr(w), rows, cols, _addr(X), nb, _addr(Y),
                                  _stream(stream)))
