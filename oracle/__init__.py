"""CPU oracle for the MXFP4 path -- TEST INFRASTRUCTURE ONLY.

The oracle (``mxfp4_oracle.cpp``) is the plain, slow statement of what the GPU
library computes: scalar decode, double accumulation.  Only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may
load it; the product library never does, and the two share no code.

This module compiles the C++ source with the host compiler and wraps its
``extern "C"`` functions with ctypes + numpy.

Parity pins (tests/test_oracle_pins.py) tie every function to the source page
("cortiq-engine 0.8.40 src/gpu_wgpu/mxfp4.rs") through closed forms, an
independent encoder, library routines and brute force; no function here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.cpp")
_LIB = os.path.join(_HERE, "libmxfp4_oracle.so")
_lock = threading.Lock()
_lib = None


def build_command(out: str = _LIB) -> list[str]:
    # -ffp-contract=off: no fused multiply-add contraction, so x86-64 and
    # aarch64 hosts give bit-identical doubles.
    return ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", "-o", out, _SRC]


def build(force: bool = False) -> str:
    """Compile the oracle shared library in-tree (idempotent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mxfp4_oracle.h"))):
        subprocess.run(build_command(), check=True)
    return _LIB


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIG = {
    "mxo_e2m1": (ctypes.c_float, [ctypes.c_uint]),
    "mxo_e8m0": (ctypes.c_float, [ctypes.c_uint]),
    "mxo_nbytes_exact": (_SZ, [_I, _I]),
    "mxo_code_at": (ctypes.c_uint, [_P, _I, _I, _I, _I]),
    "mxo_scale_at": (ctypes.c_uint, [_P, _I, _I, _I, _I]),
    "mxo_weight_at": (ctypes.c_float, [_P, _I, _I, _I, _I]),
    "mxo_dequant": (None, [_P, _I, _I, _P]),
    "mxo_matmat": (None, [_P, _I, _I, _P, _I, _I, _I, _P, _P]),
    "mxo_matmat_samples": (None, [_P, _I, _I, _P, _P, _P, _I, _P, _P]),
    "mxo_bf16_rne": (ctypes.c_float, [ctypes.c_float]),
    "mxo_round_bf16": (None, [_P, _P, _SZ]),
    "mxo_silu": (ctypes.c_double, [ctypes.c_double]),
    "mxo_silu_grad": (ctypes.c_double, [ctypes.c_double]),
    "mxo_moe_gate_up": (None, [_P, _P, _SZ, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "mxo_moe_down": (None, [_P, _SZ, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P]),
    "mxo_moe_forward": (None, [_P, _P, _P, _SZ, _SZ, _I, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P]),
    "mxo_moe_plan": (_I, [_P, _I, _I, _P, _P]),
    "mxo_moe_forward_ex": (None, [_P, _P, _P, _SZ, _SZ, _I, _I, _I, _P, _I, _I, _P, _P, _I, _P,
                                  _I, ctypes.c_float, _P, _P, _P, _P]),
    "mxo_q4k_nbytes": (_SZ, [_I, _I]),
    "mxo_f16": (ctypes.c_float, [ctypes.c_uint]),
    "mxo_q4k_scale_min": (None, [_P, _I, _P, _P]),
    "mxo_q4k_weight_at": (ctypes.c_float, [_P, _I, _I, _I, _I]),
    "mxo_q4k_dequant": (None, [_P, _I, _I, _P]),
    "mxo_q4k_matmat": (None, [_P, _I, _I, _P, _I, _I, _I, _P, _P]),
}


def lib():
    """Load (building if needed) the oracle library."""
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            h = ctypes.CDLL(path)
            for name, (res, args) in _SIG.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


# --- scalar decode -----------------------------------------------------------

def e2m1(n: int) -> float:
    return float(np.float32(lib().mxo_e2m1(n)))


def e8m0(k: int) -> float:
    return float(np.float32(lib().mxo_e8m0(k)))


def nbytes_exact(rows: int, cols: int) -> int:
    return int(lib().mxo_nbytes_exact(rows, cols))


def code_at(w, rows, cols, r, c) -> int:
    w = _u8(w)
    return int(lib().mxo_code_at(_ptr(w), rows, cols, r, c))


def scale_at(w, rows, cols, r, g) -> int:
    w = _u8(w)
    return int(lib().mxo_scale_at(_ptr(w), rows, cols, r, g))


def dequant(w, rows: int, cols: int) -> np.ndarray:
    w = _u8(w)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().mxo_dequant(_ptr(w), rows, cols, _ptr(out))
    return out


def matmat(w, rows: int, cols: int, x, nb: int, r0: int = 0, r1: int | None = None):
    """(y, l1), both float64 [nb, r1-r0]."""
    r1 = rows if r1 is None else r1
    w, x = _u8(w), _f32(x)
    assert x.size >= nb * cols
    y = np.empty((nb, r1 - r0), dtype=np.float64)
    l1 = np.empty_like(y)
    lib().mxo_matmat(_ptr(w), rows, cols, _ptr(x), nb, r0, r1, _ptr(y), _ptr(l1))
    return y, l1


def matmat_samples(w, rows: int, cols: int, x, tok, row):
    w, x, tok, row = _u8(w), _f32(x), _i32(tok), _i32(row)
    n = tok.size
    y = np.empty(n, dtype=np.float64)
    l1 = np.empty(n, dtype=np.float64)
    lib().mxo_matmat_samples(_ptr(w), rows, cols, _ptr(x), _ptr(tok), _ptr(row), n,
                             _ptr(y), _ptr(l1))
    return y, l1


def bf16_rne(v: float) -> float:
    return float(np.float32(lib().mxo_bf16_rne(v)))


def round_bf16(a) -> np.ndarray:
    a = _f32(a)
    out = np.empty_like(a)
    lib().mxo_round_bf16(_ptr(a), _ptr(out), a.size)
    return out


def silu(g: float) -> float:
    return float(lib().mxo_silu(g))


def silu_grad(g: float) -> float:
    return float(lib().mxo_silu_grad(g))


# --- routed experts ----------------------------------------------------------

def moe_gate_up(gate_bank, up_bank, stride, n_experts, hidden, inter, x, n_tokens,
                top_k, ids):
    """dict of float64 [n_tokens*top_k, inter] arrays: g, u, l1g, l1u, act."""
    gate_bank, up_bank, x, ids = _u8(gate_bank), _u8(up_bank), _f32(x), _i32(ids)
    shape = (n_tokens * top_k, inter)
    out = {k: np.empty(shape, dtype=np.float64) for k in ("g", "u", "l1g", "l1u", "act")}
    lib().mxo_moe_gate_up(_ptr(gate_bank), _ptr(up_bank), stride, n_experts, hidden, inter,
                          _ptr(x), n_tokens, top_k, _ptr(ids), _ptr(out["g"]),
                          _ptr(out["u"]), _ptr(out["l1g"]), _ptr(out["l1u"]),
                          _ptr(out["act"]))
    return out


def moe_down(down_bank, stride, n_experts, hidden, inter, act, n_tokens, top_k, ids,
             route_w, want_pairs: bool = False):
    """dict: out, l1_out [n_tokens, hidden] (+ o_pairs, l1_pairs [P, hidden])."""
    down_bank, act, ids, route_w = _u8(down_bank), _f32(act), _i32(ids), _f32(route_w)
    P = n_tokens * top_k
    res = {"out": np.empty((n_tokens, hidden)), "l1_out": np.empty((n_tokens, hidden))}
    op = lp = None
    if want_pairs:
        res["o_pairs"] = op = np.empty((P, hidden))
        res["l1_pairs"] = lp = np.empty((P, hidden))
    lib().mxo_moe_down(_ptr(down_bank), stride, n_experts, hidden, inter, _ptr(act),
                       n_tokens, top_k, _ptr(ids), _ptr(route_w),
                       _ptr(op) if op is not None else None,
                       _ptr(lp) if lp is not None else None,
                       _ptr(res["out"]), _ptr(res["l1_out"]))
    return res


def moe_forward(gate_bank, up_bank, down_bank, gu_stride, down_stride, n_experts,
                hidden, inter, x, n_tokens, top_k, ids, route_w):
    """dict: out, bound_l1, bound_prop, each float64 [n_tokens, hidden]."""
    gate_bank, up_bank, down_bank = _u8(gate_bank), _u8(up_bank), _u8(down_bank)
    x, ids, route_w = _f32(x), _i32(ids), _f32(route_w)
    res = {k: np.empty((n_tokens, hidden)) for k in ("out", "bound_l1", "bound_prop")}
    lib().mxo_moe_forward(_ptr(gate_bank), _ptr(up_bank), _ptr(down_bank), gu_stride,
                          down_stride, n_experts, hidden, inter, _ptr(x), n_tokens, top_k,
                          _ptr(ids), _ptr(route_w), _ptr(res["out"]),
                          _ptr(res["bound_l1"]), _ptr(res["bound_prop"]))
    return res


def moe_plan(ids, n_experts: int):
    """(offsets [E+1], pair_of [P], n_invalid)."""
    ids = _i32(ids)
    offsets = np.empty(n_experts + 1, dtype=np.int32)
    pair_of = np.full(ids.size, -1, dtype=np.int32)
    bad = lib().mxo_moe_plan(_ptr(ids), ids.size, n_experts, _ptr(offsets), _ptr(pair_of))
    return offsets, pair_of, int(bad)


def moe_forward_ex(gate_bank, up_bank, down_bank, gu_stride, down_stride, n_slots, hidden,
                   inter, x, n_tokens, top_k, ids, route_w, slot_of=None, n_experts=None,
                   bf16_mode=False, limit=0.0):
    """The global-bank form of the layer (bf16 boundaries, SwiGLU limit, route
    weight folded into the act, expert -> slot table with cold experts).
    dict: out, bound [n_tokens, hidden] float64; cold (int32 pair indices)."""
    gate_bank, up_bank, down_bank = _u8(gate_bank), _u8(up_bank), _u8(down_bank)
    x, ids, route_w = _f32(x), _i32(ids), _f32(route_w)
    n_experts = n_slots if n_experts is None else n_experts
    so = None if slot_of is None else _i32(slot_of)
    res = {k: np.empty((n_tokens, hidden)) for k in ("out", "bound")}
    cold = np.empty(max(ids.size, 1), dtype=np.int32)
    n_cold = ctypes.c_int(0)
    lib().mxo_moe_forward_ex(_ptr(gate_bank), _ptr(up_bank), _ptr(down_bank), gu_stride,
                             down_stride, n_slots, hidden, inter, _ptr(x), n_tokens, top_k,
                             _ptr(ids), None if so is None else _ptr(so), n_experts,
                             _ptr(route_w), int(bool(bf16_mode)), float(limit),
                             _ptr(res["out"]), _ptr(res["bound"]), _ptr(cold),
                             ctypes.addressof(n_cold))
    res["cold"] = cold[:n_cold.value].copy()
    return res


# --- the second codec: GGUF Q4_K ------------------------------------------------

def q4k_nbytes(rows: int, cols: int) -> int:
    return int(lib().mxo_q4k_nbytes(rows, cols))


def f16(bits: int) -> float:
    return float(np.float32(lib().mxo_f16(bits)))


def q4k_scale_min(scales12, j: int) -> tuple[int, int]:
    q = _u8(scales12)
    assert q.size >= 12
    sc, m = np.zeros(1, dtype=np.uint32), np.zeros(1, dtype=np.uint32)
    lib().mxo_q4k_scale_min(_ptr(q), j, _ptr(sc), _ptr(m))
    return int(sc[0]), int(m[0])


def q4k_dequant(w, rows: int, cols: int) -> np.ndarray:
    w = _u8(w)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().mxo_q4k_dequant(_ptr(w), rows, cols, _ptr(out))
    return out


def q4k_matmat(w, rows: int, cols: int, x, nb: int, r0: int = 0, r1: int | None = None):
    """(y, l1), both float64 [nb, r1-r0]."""
    r1 = rows if r1 is None else r1
    w, x = _u8(w), _f32(x)
    assert x.size >= nb * cols
    y = np.empty((nb, r1 - r0), dtype=np.float64)
    l1 = np.empty_like(y)
    lib().mxo_q4k_matmat(_ptr(w), rows, cols, _ptr(x), nb, r0, r1, _ptr(y), _ptr(l1))
    return y, l1
