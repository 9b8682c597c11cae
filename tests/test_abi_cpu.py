"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/*.h declares, and refuses bad arguments with the documented
status codes before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mx():
    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_dequant_matmul_gb300 as m
    m.lib()
    return m


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            with open(os.path.join(inc, fn)) as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
            names |= set(re.findall(r"\b((?:mxfp4|q4k)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(mx):
    names = header_functions()
    assert len(names) >= 14, names
    h = ctypes.CDLL(mx.library_path)
    for n in names:
        assert hasattr(h, n), f"{n} declared in include/*.h but not exported"
    assert set(names) == set(mx.EXPORTED_SYMBOLS), "binding and header disagree"


def test_nbytes_closed_form(mx):
    # rows*cols*17/32 rounded up to 16 (the page's examples: (2304,5120) and (1,32))
    assert mx.mxfp4_nbytes(2304, 5120) == 2304 * 5120 * 17 // 32
    assert mx.mxfp4_nbytes(1, 32) == 32
    assert mx.mxfp4_nbytes(14336, 4096) == 31195136
    assert mx.mxfp4_nbytes(2880, 2880) == 4406400
    for bad in [(0, 32), (4, 48), (4, 0), (-1, 64), (4, 31)]:
        assert mx.mxfp4_nbytes(*bad) == 0


def test_status_strings(mx):
    for s in range(5):
        assert mx.mxfp4_status_string(s)
    assert mx.mxfp4_status_string(99) == "unknown status"
    assert mx.lib().mxfp4_version() == 100


A = 1 << 20      # a 16-byte-aligned fake address; never dereferenced
MIS = A + 4      # misaligned


@pytest.mark.parametrize("rows,cols,nb,want", [
    (0, 64, 1, 1), (8, 48, 1, 1), (8, 2270, 1, 1), (8, 64, 0, 1), (8, 64, -3, 1),
    (1 << 20, 1 << 27, 1, 1),
])
def test_product_refuses_bad_shapes(mx, rows, cols, nb, want):
    L = mx.lib()
    assert L.mxfp4_mm(A, rows, cols, A, nb, A, None) == want
    assert L.mxfp4_mm_fp32(A, rows, cols, A, nb, A, None) == want
    assert L.mxfp4_mm_bf16(A, rows, cols, A, nb, A, None) == want
    if nb == 1:
        assert L.mxfp4_mv(A, rows, cols, A, A, None) == want


def test_product_refuses_bad_pointers(mx):
    L = mx.lib()
    for w, x, y in [(None, A, A), (A, None, A), (A, A, None), (MIS, A, A), (A, MIS, A),
                    (A, A, MIS)]:
        assert L.mxfp4_mv(w, 8, 64, x, y, None) == 2
        assert L.mxfp4_mm(w, 8, 64, x, 4, y, None) == 2
    assert L.mxfp4_dequant(None, 8, 64, A, None) == 2
    assert L.mxfp4_dequant(A, 8, 64, MIS, None) == 2
    assert L.mxfp4_dequant(A, 8, 33, A, None) == 1
    assert L.mxfp4_matmat_host(A, 8, 64, None, 1, A, A, A, None) == 2


def test_moe_refusals(mx):
    L = mx.lib()
    ws = mx.mxfp4_moe_workspace_bytes(64, 32, 4, 2880, 2880)
    assert ws > 32 * 4 * 2880 * 4
    # workspace too small
    assert L.mxfp4_moe_gate_up(A, A, 64, 2880, 2880, A, 32, 4, A, A, A, ws - 1, None) == 4
    assert L.mxfp4_moe_down(A, 64, 2880, 2880, A, 32, 4, A, A, A, A, ws - 1, None) == 4
    # bad shapes / counts
    assert L.mxfp4_moe_gate_up(A, A, 64, 2880, 2881, A, 32, 4, A, A, A, ws, None) == 1
    assert L.mxfp4_moe_gate_up(A, A, 0, 2880, 2880, A, 32, 4, A, A, A, ws, None) == 1
    assert L.mxfp4_moe_gate_up(A, A, 64, 2880, 2880, A, 0, 4, A, A, A, ws, None) == 1
    assert L.mxfp4_moe_down(A, 64, 2880, 2880, A, 32, 0, A, A, A, A, ws, None) == 1
    # bad pointers
    assert L.mxfp4_moe_gate_up(None, A, 64, 2880, 2880, A, 32, 4, A, A, A, ws, None) == 2
    assert L.mxfp4_moe_gate_up(A, A, 64, 2880, 2880, A, 32, 4, A + 2, A, A, ws, None) == 2
    assert L.mxfp4_moe_down(A, 64, 2880, 2880, A, 32, 4, A, None, A, A, ws, None) == 2
    assert L.mxfp4_moe_down(A, 64, 2880, 2880, A, 32, 4, A, A, A, MIS, ws, None) == 2
    assert mx.mxfp4_moe_workspace_bytes(0, 32, 4, 2880, 2880) == 0


def test_binding_raises_without_a_fallback(mx):
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.mxfp4_mv(A, 0, 64, A, A, stream=0)
    assert e.value.status == 1


def test_product_path_does_not_touch_the_oracle():
    """The library and its binding never load, import or link the oracle."""
    pkg = os.path.join(ROOT, "mxfp4_dequant_matmul_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    text = f.read()
                assert "oracle" not in text.replace("Oracle", "oracle").split("\n#")[0] or \
                    "import oracle" not in text, fn
                assert "import oracle" not in text and "mxfp4_oracle" not in text, fn


def test_q4k_nbytes_and_refusals(mx):
    # 144 bytes per 256 elements; cols must be a multiple of 256
    assert mx.q4k_nbytes(14336, 4096) == 14336 * 16 * 144
    assert mx.q4k_nbytes(1, 256) == 144
    for bad in [(0, 256), (4, 128), (4, 320), (-1, 256)]:
        assert mx.q4k_nbytes(*bad) == 0
    L = mx.lib()
    assert L.q4k_mv(A, 8, 320, A, A, None) == 1      # cols not a multiple of 256
    assert L.q4k_mv(A, 0, 256, A, A, None) == 1
    assert L.q4k_mv(MIS, 8, 256, A, A, None) == 2    # misaligned weights
    assert L.q4k_mv(A, 8, 256, None, A, None) == 2
    assert L.q4k_mm(A, 8, 256, A, 0, A, None) == 1   # no tokens
    assert L.q4k_dequant(A, 8, 256, MIS, None) == 2


def test_moe_workspace_holds_the_fragment_blocks(mx):
    # the workspace grows by 16 + 128 * (cols / 32) bytes per vector: one block per
    # token's x (hidden columns) and one per pair's act row (inter columns), beside
    # the per-pair down outputs (4 * hidden bytes per pair); regions 256-aligned
    E, T, K = 64, 32, 4
    P = T * K
    base = mx.mxfp4_moe_workspace_bytes(E, T, K, 2880, 2880)
    more_inter = mx.mxfp4_moe_workspace_bytes(E, T, K, 2880, 5760)
    assert abs((more_inter - base) - P * 128 * (5760 - 2880) // 32) < 256
    more_hidden = mx.mxfp4_moe_workspace_bytes(E, T, K, 5760, 2880)
    per_hidden = P * 4 * (5760 - 2880) + T * 128 * (5760 - 2880) // 32
    assert abs((more_hidden - base) - per_hidden) < 512
    assert base >= P * 4 * 2880 + T * (16 + 90 * 128) + P * (16 + 90 * 128)
