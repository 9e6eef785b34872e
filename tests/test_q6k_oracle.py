"""Pins of the oracle's Q6_K decoding and GEMV against facts that do not come
from the oracle: the hand-derived field-to-weight map (tests/golden/q6k_bits.txt),
closed-form blocks, brute force through a library matmul, one-hot columns, and
planted mistakes."""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits():
    rows = []
    for line in open(os.path.join(GOLDEN, "q6k_bits.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _block(d_bits=0x3C00, sc=1, ql=0, qh=0):
    """210-byte block: every ql byte = ql, every qh byte = qh, every scale = sc (int8), d = d_bits."""
    b = np.zeros(210, np.uint8)
    b[0:128] = ql
    b[128:192] = qh
    b[192:208] = np.array([sc] * 16, np.int8).view(np.uint8)
    b[208] = d_bits & 0xFF
    b[209] = d_bits >> 8
    return b


@pytest.mark.parametrize("row", _bits(), ids=lambda r: "-".join(r))
def test_q6k_field_map(oracle_mod, row):
    base = np.full(256, -32.0)   # d = 1, sc = 1, q = 0
    b = _block()
    if row[0] == "ql":
        i, half, k = int(row[1]), row[2], int(row[3])
        b[i] = 0x01 if half == "lo" else 0x10
        want = base.copy()
        want[k] = -31.0
    elif row[0] == "qh":
        j, pair, k = int(row[1]), int(row[2]), int(row[3])
        b[128 + j] = 1 << (2 * pair)
        want = base.copy()
        want[k] = -16.0
    else:
        j, k0 = int(row[1]), int(row[2])
        b[192 + j] = 3
        want = base.copy()
        want[k0:k0 + 16] = -96.0
    assert np.array_equal(oracle_mod.q6k_dequant_block(b), want)


def test_q6k_closed_forms(oracle_mod):
    # every code 63, scale -2 (signed), d = 0.5 (fp16 0x3800): w = 0.5 * -2 * 31
    assert np.all(oracle_mod.q6k_dequant_block(_block(0x3800, -2, 0xFF, 0xFF)) == -31.0)
    # every code 32 (low nibbles 0, high bits 10): w = 0 whatever the scale
    assert np.all(oracle_mod.q6k_dequant_block(_block(0x3C00, 127, 0x00, 0xAA)) == 0.0)
    # scale -128, codes 0, d = 2^-24 (the smallest fp16 subnormal, 0x0001): w = 2^-24 * 128 * 32
    assert np.all(oracle_mod.q6k_dequant_block(_block(0x0001, -128, 0, 0)) == 2.0 ** -24 * 4096)
    # codes 47 (low nibble 15, high bits 10) with alternating scale signs
    b = _block(0x3C00, 1, 0xFF, 0xAA)
    b[192:208] = np.array([(-1) ** j * (j + 1) for j in range(16)], np.int8).view(np.uint8)
    w = oracle_mod.q6k_dequant_block(b)
    want = np.repeat([(-1) ** j * (j + 1) * 15.0 for j in range(16)], 16)
    assert np.array_equal(w, want)


@pytest.mark.parametrize("N,K,B", [(1, 256, 1), (5, 512, 2), (7, 1024, 3)])
def test_q6k_gemv_brute_force(oracle_mod, N, K, B):
    W = synth.q6k_weights(N, K, (N, K, 61))
    x = synth.normal_f32((B, K), (N, K, 62))
    D = oracle_mod.q6k_dequant_matrix(W, N, K)
    np.testing.assert_allclose(oracle_mod.q6k_gemv(W, x, N, K), x.astype(np.float64) @ D.T, rtol=1e-12, atol=1e-9)
    rows = np.array([N - 1, 0])
    np.testing.assert_allclose(oracle_mod.q6k_gemv_rows(W, x, N, K, rows), (x.astype(np.float64) @ D.T)[:, rows],
                               rtol=1e-12, atol=1e-9)


def test_q6k_gemv_one_hot(oracle_mod):
    N, K = 4, 512
    W = synth.q6k_weights(N, K, 63)
    D = oracle_mod.q6k_dequant_matrix(W, N, K)
    for k in (0, 77, 300, 511):
        x = np.zeros(K, np.float32)
        x[k] = 1.0
        assert np.array_equal(oracle_mod.q6k_gemv(W, x, N, K)[0], D[:, k])


def test_q6k_generator_marginals(oracle_mod):
    """Codes uniform on 0..63 and scales on all int8 values."""
    W = synth.q6k_weights(64, 4096, 64)
    blocks = W.reshape(-1, 210)
    d = blocks[:, 208].astype(np.uint16) | (blocks[:, 209].astype(np.uint16) << 8)
    dv = d.view(np.float16).astype(np.float64)
    assert dv.min() >= 2e-4 * 0.999 and dv.max() <= 2e-3 * 1.001
    sc = blocks[:, 192:208].view(np.int8)
    assert sc.min() == -128 and sc.max() == 127


def test_q6k_pins_catch_planted_mistakes(oracle_mod, tmp_path):
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "q4k_oracle.c")).read()
    mutants = {
        "qh shift": ("(qh[32 * h + l] >> (2 * c)) & 3", "(qh[32 * h + l] >> (2 * (c & 1))) & 3"),
        "offset 31": ("(double)(q - 32)", "(double)(q - 31)"),
        "scale per 32": ("(double)sc[k / 16]", "(double)sc[k / 32]"),
        "nibble half": ("(c < 2) ? (byte & 15) : (byte >> 4)", "(c & 1) ? (byte >> 4) : (byte & 15)"),
        "ql index": ("ql[64 * h + 32 * (c & 1) + l]", "ql[64 * h + l]"),
        "unsigned scales": ("const int8_t *sc = (const int8_t *)(blk + 192);",
                            "const uint8_t *sc = (const uint8_t *)(blk + 192);"),
    }
    rows = _bits()
    caught = {}
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"q6_{abs(hash(name))}.c"
        path.write_text(src.replace(a, b))
        so = str(path) + ".so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        lib.oracle_q6k_dequant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p]

        def deq(b):
            w = np.zeros(256)
            b = np.ascontiguousarray(b, np.uint8)
            lib.oracle_q6k_dequant_block(b.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p))
            return w

        bad = not np.all(deq(_block(0x3800, -2, 0xFF, 0xFF)) == -31.0)
        for row in rows:
            b = _block()
            if row[0] == "ql":
                b[int(row[1])] = 0x01 if row[2] == "lo" else 0x10
                want = np.full(256, -32.0)
                want[int(row[3])] = -31.0
            elif row[0] == "qh":
                b[128 + int(row[1])] = 1 << (2 * int(row[2]))
                want = np.full(256, -32.0)
                want[int(row[3])] = -16.0
            else:
                b[192 + int(row[1])] = 3
                want = np.full(256, -32.0)
                want[int(row[2]):int(row[2]) + 16] = -96.0
            bad |= not np.array_equal(deq(b), want)
        caught[name] = bad
    assert all(caught.values()), caught
