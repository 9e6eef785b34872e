"""CPU-side checks of the C ABI: the library builds, loads, exports every
declared symbol, and rejects bad arguments on the host without launching."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def q4k():
    from q4_dequant_gemv_gb300 import _build
    _build.build()
    import q4_dequant_gemv_gb300 as m
    m.lib()
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "q4k.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b((?:q4k|q6k)_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_exported(q4k):
    names = _declared()
    assert "q4k_gemv" in names and "q4k_gemv_argmax" in names and "q4k_gemm_prefill" in names
    L = q4k.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(q4k.EXPORTS)


def test_abi_version_and_strings(q4k):
    assert q4k.lib().q4k_abi_version() == 1
    for s in range(5):
        assert len(q4k.status_string(s)) > 0
    assert q4k.status_string(99) == "unknown status"


P = ctypes.c_void_p


def _gemv(q4k, W, x, y, N, K, B):
    return q4k.raw_call("q4k_gemv", P(W), P(x), P(y), N, K, B, P(0))


def test_host_validation(q4k):
    """Argument errors come back before any device call (no GPU needed)."""
    ok = 0x10000  # aligned fake addresses; never dereferenced on these paths
    assert _gemv(q4k, 0, ok, ok, 64, 256, 1) == 1
    assert _gemv(q4k, ok, 0, ok, 64, 256, 1) == 1
    assert _gemv(q4k, ok, ok, 0, 64, 256, 1) == 1
    assert _gemv(q4k, ok, ok, ok, 64, 255, 1) == 1
    assert _gemv(q4k, ok, ok, ok, 64, 0, 1) == 1
    assert _gemv(q4k, ok, ok, ok, 64, 384, 1) == 1
    assert _gemv(q4k, ok, ok, ok, -1, 256, 1) == 1
    assert _gemv(q4k, ok, ok, ok, 64, 256, 0) == 1
    assert _gemv(q4k, ok, ok, ok, 64, 256, 17) == 1
    assert _gemv(q4k, ok, ok, ok, 2 ** 31, 256, 1) == 1
    assert _gemv(q4k, ok + 8, ok, ok, 64, 256, 1) == 2
    assert _gemv(q4k, ok, ok + 4, ok, 64, 256, 1) == 2
    am = lambda W, x, i, N, K, B: q4k.raw_call("q4k_gemv_argmax", P(W), P(x), P(i), N, K, B, P(0))
    assert am(ok, ok, ok, 0, 256, 1) == 1           # argmax of nothing is undefined
    assert am(ok, ok, 0, 8, 256, 1) == 1
    assert am(ok, ok, ok, 8, 256, 17) == 1
    dbg = q4k.raw_call("q4k_gemv_argmax_debug", P(ok), P(ok), P(ok), P(0), 8, 256, 1, P(0))
    assert dbg == 1
    assert _gemv(q4k, 0, ok, 0, 0, 256, 1) in (0, 3, 4)
    for fn in ("q4k_gemm_prefill", "q4k_gemm_prefill_exact"):
        pf = lambda W, X, Y, N, K, T: q4k.raw_call(fn, P(W), P(X), P(Y), N, K, T, P(0))
        assert pf(0, ok, ok, 64, 256, 32) == 1
        assert pf(0, 0, 0, 0, 256, 32) in (0, 3, 4)      # N == 0: no pointer is needed
        assert pf(ok, ok, ok, 64, 100, 32) == 1
        assert pf(ok, ok, ok, 64, 256, -1) == 1
        assert pf(ok, ok + 2, ok, 64, 256, 32) == 2


def test_no_device_reports_status(q4k):
    """A well-formed call on a machine without a usable GPU returns a status, not a crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    st = _gemv(q4k, 0x10000, 0x10000, 0x10000, 64, 256, 1)
    assert st in (3, 4)


def test_missing_library_fails_loudly(tmp_path):
    """Without libq4k.so the binding raises; there is no CPU fallback."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import q4_dequant_gemv_gb300 as q\n"
        "q.LIB_PATH = %r\n"
        "try:\n    q.lib()\nexcept RuntimeError as e:\n    print('raised', e)\n"
    ) % (ROOT, str(tmp_path / "nope.so"))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert "raised" in out.stdout


def test_product_does_not_touch_oracle():
    """The product package never imports or names the oracle."""
    pkg = os.path.join(ROOT, "q4_dequant_gemv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
    text = open(os.path.join(ROOT, "include", "q4k.h")).read()
    assert "oracle" not in text.lower()


def test_stream_read_host_validation(q4k):
    """The streaming probe rejects bad arguments before any device call."""
    L = q4k.lib()
    n = ctypes.c_int64(-1)
    ok = 0x10000
    assert L.q4k_stream_read(P(ok), 1 << 20, None, P(0)) == 1
    assert L.q4k_stream_read(P(ok), -1, ctypes.byref(n), P(0)) == 1
    assert n.value == 0
    assert L.q4k_stream_read(P(0), 1 << 20, ctypes.byref(n), P(0)) == 1
    assert L.q4k_stream_read(P(ok + 4), 1 << 20, ctypes.byref(n), P(0)) == 2


def test_split_receive_slots_fit():
    """The GEMV's split-K reduction (one row tile over `split` CTAs of a cluster):
    rank r owns tile rows [r*128/split, (r+1)*128/split) and receives one slot per
    source rank for each of them at offset src*(rows owned) + (row - first row).
    Every offset it writes or reads stays below the 144 rows of the buffer for
    every split up to 16 (the same formulas as the kernel's epilogue)."""
    k_rows, buf_rows = 128, 144
    for split in range(1, 17):
        top = 0
        for src in range(split):
            for row in range(k_rows):
                owner = (row * split + split - 1) // k_rows
                o0, o1 = owner * k_rows // split, (owner + 1) * k_rows // split
                assert o0 <= row < o1
                top = max(top, src * (o1 - o0) + (row - o0))
        for rank in range(split):
            rows = (rank + 1) * k_rows // split - rank * k_rows // split
            top = max(top, (split - 1) * rows + rows - 1)
        assert top < buf_rows, (split, top)


def test_q6k_host_validation(q4k):
    """q6k_gemv argument errors come back before any device call."""
    ok = 0x10000
    q6 = lambda W, x, y, N, K, B: q4k.raw_call("q6k_gemv", P(W), P(x), P(y), N, K, B, P(0))
    assert q6(0, ok, ok, 64, 256, 1) == 1
    assert q6(ok, 0, ok, 64, 256, 1) == 1
    assert q6(ok, ok, 0, 64, 256, 1) == 1
    assert q6(ok, ok, ok, 64, 300, 1) == 1
    assert q6(ok, ok, ok, -1, 256, 1) == 1
    assert q6(ok, ok, ok, 64, 256, 0) == 1
    assert q6(ok, ok, ok, 64, 256, 17) == 1
    assert q6(ok + 2, ok, ok, 64, 256, 1) == 2
    assert q6(ok, ok + 4, ok, 64, 256, 1) == 2
    assert q6(0, ok, 0, 0, 256, 1) in (0, 3, 4)      # N == 0: no weight or output pointer needed


def test_q6k_planar_host_validation(q4k):
    """q6k_repack_planar and q6k_gemv_planar argument errors come back before any
    device call (1 = INVALID_ARG, 2 = MISALIGNED)."""
    ok = 0x10000
    rp = lambda W, Wp, N, K: q4k.raw_call("q6k_repack_planar", P(W), P(Wp), N, K, P(0))
    gp = lambda Wp, x, y, N, K, B: q4k.raw_call("q6k_gemv_planar", P(Wp), P(x), P(y), N, K, B, P(0))
    assert rp(0, ok, 64, 256) == 1
    assert rp(ok, 0, 64, 256) == 1
    assert rp(ok, 0x100000, 64, 300) == 1
    assert rp(ok, 0x100000, -1, 256) == 1
    assert rp(ok + 2, 0x100000, 64, 256) == 2
    assert rp(ok, 0x100000 + 8, 64, 256) == 2
    assert gp(0, ok, ok, 64, 256, 1) == 1
    assert gp(ok, 0, ok, 64, 256, 1) == 1
    assert gp(ok, ok, 0, 64, 256, 1) == 1
    assert gp(ok, ok, ok, 64, 300, 1) == 1
    assert gp(ok, ok, ok, 64, 256, 0) == 1
    assert gp(ok, ok, ok, 64, 256, 17) == 1
    assert gp(ok + 2, ok, ok, 64, 256, 1) == 2
    assert gp(ok, ok + 4, ok, 64, 256, 1) == 2


def test_binding_refuses_host_tensors(q4k):
    """The Python entry points take device tensors only: host tensors raise
    before anything is computed (there is no CPU path)."""
    import torch
    W = torch.zeros((4, 144), dtype=torch.uint8)
    x = torch.zeros((1, 256), dtype=torch.float32)
    for call in (lambda: q4k.gemv(W, x), lambda: q4k.gemv_argmax(W, x),
                 lambda: q4k.q6k_gemv(torch.zeros((4, 210), dtype=torch.uint8), x),
                 lambda: q4k.gemm_prefill(W, torch.zeros((32, 256), dtype=torch.bfloat16))):
        with pytest.raises((ValueError, TypeError, RuntimeError)):
            call()


def test_q6k_planar_bytes_host_only(q4k):
    """The planar Q6_K size is a host computation: N * (nb*208 + 2*nb rounded up to 16)."""
    L = q4k.lib()
    assert L.q6k_planar_bytes(152064, 3584) == 152064 * (14 * 208 + 32)
    assert L.q6k_planar_bytes(3, 18944) == 3 * (74 * 208 + 160)
    assert L.q6k_planar_bytes(0, 256) == 0
    assert L.q6k_planar_bytes(5, 100) == -1 and L.q6k_planar_bytes(-1, 256) == -1
