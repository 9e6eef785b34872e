"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: numpy's own IEEE decoders, the
hand-typed golden fixtures in tests/golden (layout reading written out by hand),
closed forms, brute force through a library matmul, or invariants of the
mathematics.  None of them re-types the oracle's formula.
"""
import math
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- fp16 / bf16
def test_fp16_decode_all_patterns(oracle_mod):
    """Every binary16 pattern decodes like numpy's float16 (independent decoder)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_fp16_named_values(oracle_mod):
    assert oracle_mod.fp16_to_double(0x3C00) == 1.0
    assert oracle_mod.fp16_to_double(0x0001) == 2.0 ** -24
    assert oracle_mod.fp16_to_double(0x7BFF) == 65504.0
    z = oracle_mod.fp16_to_double(0x8000)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert oracle_mod.fp16_to_double(0xC000) == -2.0


def test_bf16_decode_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle_mod.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_round_bf16_matches_integer_rounding(oracle_mod):
    """RNE to 8 significant bits, checked against round-half-even on integers."""
    g = np.random.default_rng(5)
    for _ in range(2000):
        v = float(g.standard_normal() * 10.0 ** g.integers(-5, 5))
        e = math.frexp(v)[1]
        scaled = v * 2.0 ** (8 - e)                      # |scaled| in [128, 256)
        ref = float(np.round(scaled)) * 2.0 ** (e - 8)   # numpy rounds half to even
        assert oracle_mod.round_bf16(v) == ref
    assert oracle_mod.round_bf16(1.0 + 2 ** -8) == 1.0               # tie -> even
    assert oracle_mod.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6   # tie -> even (up)


# ---------------------------------------------------------------- layout
def _scale_bits():
    rows = []
    with open(os.path.join(GOLDEN, "scale_bits.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            byte, bit, field, idx, val = line.split()
            rows.append((int(byte), int(bit), field, int(idx), int(val)))
    return rows


def test_scale_bits_single_bit(oracle_mod):
    """Each of the 96 bits of the scale bytes lands in the hand-typed field."""
    rows = _scale_bits()
    assert len(rows) == 96
    for byte, bit, field, idx, val in rows:
        s = np.zeros(12, np.uint8)
        s[byte] = 1 << bit
        sc, m = oracle_mod.unpack_scales(s)
        exp_sc = np.zeros(8, np.int32)
        exp_m = np.zeros(8, np.int32)
        (exp_sc if field == "sc" else exp_m)[idx] = val
        assert np.array_equal(sc, exp_sc), (byte, bit)
        assert np.array_equal(m, exp_m), (byte, bit)


def test_quant_nibbles_single(oracle_mod):
    """Low nibble of qs[32p+i] is weight 64p+i, high nibble is weight 64p+32+i."""
    for p in range(4):
        for i in (0, 7, 31):
            for hi in (0, 1):
                qs = np.zeros(128, np.uint8)
                qs[32 * p + i] = (5 << 4) if hi else 5
                q = oracle_mod.unpack_quants(qs)
                exp = np.zeros(256, np.int32)
                exp[64 * p + 32 * hi + i] = 5
                assert np.array_equal(q, exp)


def _golden_blocks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, rest = line.split(None, 1)
            rest = rest.strip()
            if key == "name":
                cur = {"name": rest}
                blocks.append(cur)
            elif key == "header":
                cur["header"] = bytes(int(h, 16) for h in rest.split())
            elif key == "d":
                a = rest.split()
                cur["d"], cur["dmin"] = float(a[0]), float(a[2])
            elif key in ("sc", "m"):
                cur[key] = [int(v) for v in rest.split()]
            else:
                cur[key] = rest
    return blocks


def _q_of(rule, k):
    j, i = divmod(k, 32)
    return int(eval(rule, {}, {"k": k, "i": i, "j": j}))


def _w_of(blk, k, q):
    j, i = divmod(k, 32)
    env = {"j": j, "i": i, "q": q, "sc_j": blk["sc"][j], "m_j": blk["m"][j]}
    return float(eval(blk["w"], {}, env))


@pytest.mark.parametrize("blk", _golden_blocks(), ids=lambda b: b["name"])
def test_golden_block(oracle_mod, blk):
    q = np.array([_q_of(blk["q"], k) for k in range(256)], np.int32)
    hdr = np.frombuffer(blk["header"], np.uint8)
    d_bits = int(hdr[0]) | (int(hdr[1]) << 8)
    m_bits = int(hdr[2]) | (int(hdr[3]) << 8)
    assert oracle_mod.fp16_to_double(d_bits) == blk["d"]
    assert oracle_mod.fp16_to_double(m_bits) == blk["dmin"]
    sc, m = oracle_mod.unpack_scales(hdr[4:16])
    assert list(sc) == blk["sc"] and list(m) == blk["m"]
    packed = oracle_mod.pack_block(d_bits, m_bits, blk["sc"], blk["m"], q)
    assert bytes(packed[:16]) == blk["header"]
    assert np.array_equal(oracle_mod.unpack_quants(packed[16:]), q)
    w = oracle_mod.dequant_block(packed)
    exp = np.array([_w_of(blk, k, q[k]) for k in range(256)])
    assert np.array_equal(w, exp)


def test_generator_marginals(oracle_mod):
    """Uniform bytes decode to uniform sc/m on 0..63 and q on 0..15 (input recipe)."""
    W = synth.q4k_weights(64, 4096, 11)
    blocks = W.reshape(-1, 144)
    sc_all, m_all, q_all = [], [], []
    for blk in blocks[:512]:
        sc, m = oracle_mod.unpack_scales(blk[4:16])
        sc_all.append(sc)
        m_all.append(m)
        q_all.append(oracle_mod.unpack_quants(blk[16:]))
    sc_all = np.concatenate(sc_all)
    m_all = np.concatenate(m_all)
    q_all = np.concatenate(q_all)
    assert sc_all.min() == 0 and sc_all.max() == 63 and m_all.max() == 63
    assert abs(sc_all.mean() - 31.5) < 1.0 and abs(m_all.mean() - 31.5) < 1.0
    assert abs(q_all.mean() - 7.5) < 0.1 and q_all.max() == 15
    d = blocks[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    assert d.min() >= 2e-4 * (1 - 2 ** -10) and d.max() <= 2e-3 * (1 + 2 ** -10)


# ---------------------------------------------------------------- gemv
def _tiny(N, K, seed):
    return synth.q4k_weights(N, K, (seed, 99)), synth.normal_f32((3, K), (seed, 98))


@pytest.mark.parametrize("N,K", [(1, 256), (5, 512), (8, 768)])
def test_gemv_brute_force(oracle_mod, N, K):
    """Oracle gemv == dense dequant followed by numpy's fp64 matmul."""
    W, x = _tiny(N, K, N * 7 + K)
    dense = oracle_mod.dequant_matrix(W, N, K)
    y = oracle_mod.gemv(W, x, N, K)
    ref = x.astype(np.float64) @ dense.T
    scale = np.abs(x.astype(np.float64)) @ np.abs(dense).T
    assert np.all(np.abs(y - ref) <= 1e-12 * scale + 1e-300)


def test_gemv_one_hot_column(oracle_mod):
    """x = e_k returns column k of the dequantized matrix exactly."""
    N, K = 6, 512
    W, _ = _tiny(N, K, 3)
    cols = [0, 1, 31, 32, 255, 256, 300, 511]
    x = np.zeros((len(cols), K), np.float32)
    for r, c in enumerate(cols):
        x[r, c] = 1.0
    y = oracle_mod.gemv(W, x, N, K)
    for r, c in enumerate(cols):
        blk = W[:, (c // 256) * 144:(c // 256 + 1) * 144]
        for n in range(N):
            # closed form of that single weight from its own fields
            hdr = blk[n]
            d = float(hdr[0:2].copy().view(np.float16)[0])
            dmin = float(hdr[2:4].copy().view(np.float16)[0])
            sc, m = oracle_mod.unpack_scales(hdr[4:16])
            q = oracle_mod.unpack_quants(hdr[16:144])
            kk = c % 256
            j = kk // 32
            assert y[r, n] == d * sc[j] * q[kk] - dmin * m[j]


def test_gemv_all_ones_row_sums(oracle_mod):
    """x = 1: y_n = sum over blocks and sub-blocks of d*sc_j*sum(q) - 32*dmin*m_j."""
    N, K = 4, 1024
    W, _ = _tiny(N, K, 4)
    y = oracle_mod.gemv(W, np.ones((1, K), np.float32), N, K)[0]
    for n in range(N):
        tot = 0.0
        for b in range(K // 256):
            blk = W[n, b * 144:(b + 1) * 144]
            d = float(blk[0:2].copy().view(np.float16)[0])
            dmin = float(blk[2:4].copy().view(np.float16)[0])
            sc, m = oracle_mod.unpack_scales(blk[4:16])
            q = oracle_mod.unpack_quants(blk[16:144])
            for j in range(8):
                tot += d * sc[j] * int(q[32 * j:32 * j + 32].sum()) - 32 * dmin * m[j]
        assert abs(y[n] - tot) <= 1e-12 * abs(tot) + 1e-12


def test_gemv_batch_invariance(oracle_mod):
    """A batch-B product equals B batch-1 products, bit for bit."""
    N, K = 9, 768
    W = synth.q4k_weights(N, K, 21)
    x = synth.normal_f32((5, K), 22)
    yb = oracle_mod.gemv(W, x, N, K)
    for b in range(5):
        assert np.array_equal(yb[b], oracle_mod.gemv(W, x[b], N, K)[0])


def test_gemv_threads_invariance(oracle_mod):
    N, K = 33, 512
    W = synth.q4k_weights(N, K, 23)
    x = synth.normal_f32((2, K), 24)
    assert np.array_equal(oracle_mod.gemv(W, x, N, K, threads=1), oracle_mod.gemv(W, x, N, K, threads=4))


def test_gemv_rows_subset(oracle_mod):
    N, K = 40, 512
    W = synth.q4k_weights(N, K, 25)
    x = synth.normal_f32((2, K), 26)
    rows = np.array([0, 3, 39, 17])
    assert np.array_equal(oracle_mod.gemv_rows(W, x, N, K, rows), oracle_mod.gemv(W, x, N, K)[:, rows])


def test_gemv_linearity(oracle_mod):
    """W.(a x1 + x2) == a W.x1 + W.x2 up to fp64 rounding (catches a dropped term)."""
    N, K = 7, 512
    W = synth.q4k_weights(N, K, 27)
    x1 = synth.normal_f32(K, 28).astype(np.float64)
    x2 = synth.normal_f32(K, 29).astype(np.float64)
    xs = (2.0 * x1 + x2).astype(np.float32)   # exact: both halves are fp32 values *2 and +
    lhs = oracle_mod.gemv(W, xs, N, K)[0]
    rhs = 2.0 * oracle_mod.gemv(W, x1.astype(np.float32), N, K)[0] + oracle_mod.gemv(W, x2.astype(np.float32), N, K)[0]
    # xs is 2*x1+x2 rounded to fp32, so compare against the exact sum's bound
    err_in = np.abs(xs.astype(np.float64) - (2.0 * x1 + x2))
    dense = oracle_mod.dequant_matrix(W, N, K)
    bound = np.abs(dense) @ err_in + 1e-9
    assert np.all(np.abs(lhs - rhs) <= bound)


# ---------------------------------------------------------------- argmax
def test_argmax_ties_lowest_index(oracle_mod):
    v = np.array([1.0, 3.0, -2.0, 3.0, 3.0], np.float32)
    assert oracle_mod.argmax(v) == 1
    v64 = np.array([5.0, 5.0], np.float64)
    assert oracle_mod.argmax(v64) == 0


def test_argmax_nan_and_zero(oracle_mod):
    assert oracle_mod.argmax(np.array([np.nan, -1.0, np.nan], np.float32)) == 1
    assert oracle_mod.argmax(np.array([np.nan, np.nan], np.float32)) == 0
    assert oracle_mod.argmax(np.array([-0.0, 0.0], np.float32)) == 0
    assert oracle_mod.argmax(np.array([-1.0, 0.0, -0.0], np.float32)) == 1
    assert oracle_mod.argmax(np.array([-np.inf, -np.inf], np.float32)) == 0


def test_argmax_matches_numpy(oracle_mod):
    g = np.random.default_rng(3)
    for _ in range(50):
        v = g.integers(-3, 3, size=int(g.integers(1, 40))).astype(np.float32)
        assert oracle_mod.argmax(v) == int(np.argmax(v))   # numpy returns the first maximum


def _planted_row(oracle_mod, x, K):
    """Row with d=1, dmin=0, sc=63, m=0, q=15 where x>0 else 0: y = 945*sum(x>0)."""
    nb = K // 256
    out = []
    for b in range(nb):
        q = np.where(x[b * 256:(b + 1) * 256] > 0, 15, 0)
        out.append(oracle_mod.pack_block(0x3C00, 0x0000, [63] * 8, [0] * 8, q))
    return np.concatenate(out)


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_argmax_planted_unique_max(oracle_mod, where):
    N, K = 300, 3584
    W = synth.q4k_weights(N, K, 31)
    x = synth.normal_f32(K, 32)
    r = {"first": 0, "middle": 137, "last": N - 1}[where]
    W2 = synth.plant_row(W, r, _planted_row(oracle_mod, x, K))
    y = oracle_mod.gemv(W2, x, N, K)[0]
    pos = x[x > 0].astype(np.float64).sum()
    assert y[r] == 945.0 * pos            # closed form, exact in fp64 (integers * fp32 sums)
    # every other row is bounded by max|w| * sum|x| with max|w| <= 2e-3*63*15 + 2e-3*63
    bound = (2e-3 * 63 * 15 + 2e-3 * 63) * (1 + 2 ** -10) * np.abs(x.astype(np.float64)).sum()
    others = np.delete(y, r)
    assert np.abs(others).max() <= bound < y[r]
    assert oracle_mod.argmax(y) == r


def test_argmax_two_identical_planted_rows(oracle_mod):
    N, K = 50, 512
    W = synth.q4k_weights(N, K, 33)
    x = synth.normal_f32(K, 34)
    row = _planted_row(oracle_mod, x, K)
    W2 = synth.plant_row(synth.plant_row(W, 11, row), 40, row)
    y = oracle_mod.gemv(W2, x, N, K)[0]
    assert y[11] == y[40] and oracle_mod.argmax(y) == 11


# ---------------------------------------------------------------- prefill
def test_prefill_brute_force(oracle_mod):
    N, K, T = 6, 512, 5
    W = synth.q4k_weights(N, K, 41)
    X = synth.normal_bf16_bits((T, K), 42)
    Y = oracle_mod.prefill(W, X, N, K)
    Xf = synth.bf16_bits_to_f32(X).astype(np.float64)
    dense = oracle_mod.dequant_matrix(W, N, K)
    ref = Xf @ dense.T
    scale = np.abs(Xf) @ np.abs(dense).T
    assert np.all(np.abs(Y - ref) <= 1e-12 * scale)


def test_prefill_rounded_weights_diagnostic(oracle_mod):
    """The bf16-weight variant differs from the exact one by at most 2^-9 relative per term."""
    N, K, T = 4, 512, 3
    W = synth.q4k_weights(N, K, 43)
    X = synth.normal_bf16_bits((T, K), 44)
    Y = oracle_mod.prefill(W, X, N, K)
    Yr = oracle_mod.prefill(W, X, N, K, round_w=True)
    Xf = np.abs(synth.bf16_bits_to_f32(X).astype(np.float64))
    dense = np.abs(oracle_mod.dequant_matrix(W, N, K))
    assert np.all(np.abs(Y - Yr) <= 2 ** -9 * (Xf @ dense.T) * 1.0001)
    assert not np.array_equal(Y, Yr)


# ---------------------------------------------------------------- planted mistakes
def test_pins_catch_planted_mistakes(oracle_mod, tmp_path):
    """Plant plausible mistakes into a copy of the oracle source; the pins above must notice.

    Each variant is compiled to its own library and exercised on the checks that
    should catch it (golden blocks, brute force, single-bit scales)."""
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "q4k_oracle.c")).read()
    mutants = {
        "min sign": ("- dmin * (double)m[j]", "+ dmin * (double)m[j]"),
        "high scale bits": ("((s[j - 4] >> 6) << 4)", "((s[j - 4] >> 6) << 3)"),
        "nibble order": ("q[64 * p + i] = qs[32 * p + i] & 15;", "q[64 * p + i] = qs[32 * p + i] >> 4;"),
        "min index": ("m[j] = s[j + 4] & 63;", "m[j] = s[j] & 63;"),
        "fp16 bias": ("e - 25", "e - 24"),
    }
    blk = _golden_blocks()[3]
    q = np.array([_q_of(blk["q"], k) for k in range(256)], np.int32)
    good = oracle_mod.pack_block(0x1400, 0xC000, blk["sc"], blk["m"], q)
    good[:16] = np.frombuffer(blk["header"], np.uint8)   # hand-typed header bytes
    exp = np.array([_w_of(blk, k, q[k]) for k in range(256)])
    caught = {}
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"m_{abs(hash(name))}.c"
        path.write_text(src.replace(a, b))
        so = str(path) + ".so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        lib.oracle_dequant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        w = np.zeros(256)
        lib.oracle_dequant_block(good.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p))
        caught[name] = not np.array_equal(w, exp)
    assert all(caught.values()), caught


# ---------------------------------------------------------------- Q8_K activations
def _q8k_golden():
    blocks, cur = [], None
    for line in open(os.path.join(GOLDEN, "q8k_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(None, 1)
        if key == "name":
            cur = {"name": rest}
            blocks.append(cur)
        elif key in ("x", "q"):
            cur[key] = [float(v) for v in rest.split()]
        elif key == "d":
            cur["d"] = rest
    return blocks


@pytest.mark.parametrize("blk", _q8k_golden(), ids=lambda b: b["name"])
def test_q8k_golden_blocks(oracle_mod, blk):
    """Hand-derived codes and scales (tests/golden/q8k_blocks.txt)."""
    x = np.zeros(256, np.float32)
    x[:len(blk["x"])] = blk["x"]
    q, d = oracle_mod.q8k_quantize(x, 256)
    assert list(q[:len(blk["q"])]) == [int(v) for v in blk["q"]]
    assert np.all(q[len(blk["q"]):] == 0)
    if "/" in blk["d"]:
        num, den = blk["d"].split("/")
        want = np.float32(num) / np.float32(den)   # IEEE single division (numpy)
    else:
        want = np.float32(blk["d"])
    assert d[0] == want


def test_q8k_invariants(oracle_mod):
    """|q| <= 127, the largest |x| maps to +-127 with its sign, every code is
    within half a step of x/d, and the signs agree."""
    g = np.random.default_rng(11)
    K = 256 * 8
    x = (g.standard_normal(K) * np.repeat(10.0 ** g.uniform(-20, 20, K // 256), 256)).astype(np.float32)
    q, d = oracle_mod.q8k_quantize(x, K)
    assert np.all(np.abs(q.astype(int)) <= 127)
    for b in range(K // 256):
        xb, qb = x[256 * b:256 * (b + 1)].astype(np.float64), q[256 * b:256 * (b + 1)].astype(np.float64)
        i = int(np.argmax(np.abs(xb)))
        assert qb[i] == 127 * np.sign(xb[i])
        assert np.all(np.abs(xb / np.float64(d[b]) - qb) <= 0.5 + 1e-5)
        assert np.all(qb * xb >= 0)


@pytest.mark.parametrize("e", [-90, -70, -3, 5, 60])
def test_q8k_power_of_two_scaling(oracle_mod, e):
    """Scaling a block by 2^e leaves every code unchanged and scales d by 2^e
    exactly -- including blocks whose max drops below 2^-64."""
    g = np.random.default_rng(12)
    x = g.standard_normal(512).astype(np.float32)
    q0, d0 = oracle_mod.q8k_quantize(x, 512)
    xs = (x.astype(np.float64) * 2.0 ** e).astype(np.float32)
    assert np.array_equal(xs.astype(np.float64), x.astype(np.float64) * 2.0 ** e)   # exact scaling
    q1, d1 = oracle_mod.q8k_quantize(xs, 512)
    assert np.array_equal(q0, q1)
    assert np.array_equal(d1.astype(np.float64), d0.astype(np.float64) * 2.0 ** e)


def test_q8k_product_brute_force(oracle_mod):
    """The Q4_K x Q8_K product equals the library matmul of the dequantized
    weights with the dequantized codes, and stays within the quantization
    bound sum_k |w| d/2 of the exact product with x."""
    N, K = 6, 768
    W = synth.q4k_weights(N, K, 13)
    x = synth.normal_f32((1, K), 14)[0]
    q, d = oracle_mod.q8k_quantize(x, K)
    xt = np.repeat(d.astype(np.float64), 256) * q.astype(np.float64)
    D = oracle_mod.dequant_matrix(W, N, K)
    y = oracle_mod.gemv_q8k(W, q, d, N, K)
    np.testing.assert_allclose(y, D @ xt, rtol=1e-12, atol=1e-12)
    exact = oracle_mod.gemv(W, x, N, K)[0]
    bound = np.abs(D) @ (np.repeat(d.astype(np.float64), 256) / 2) * (1 + 1e-6)
    assert np.all(np.abs(y - exact) <= bound)
    assert np.any(y != exact)


def test_q8k_pins_catch_planted_mistakes(oracle_mod, tmp_path):
    """Plausible mistakes planted into a copy of the quantizer are caught by
    the golden blocks or the scaling pin."""
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "q4k_oracle.c")).read()
    mutants = {
        "half away from zero": ("q[b * QK + i] = (int8_t)rintf(t);", "q[b * QK + i] = (int8_t)roundf(t);"),
        "128 levels": ("127.0f / (a * pre)", "128.0f / (a * pre)"),
        "scale 1/128": ("d[b] = a / 127.0f;", "d[b] = a / 128.0f;"),
        "signed max": ("const float v = fabsf(xb[i]);", "const float v = xb[i];"),
        "unscaled x": ("const float t = (xb[i] * pre) * inv;", "const float t = xb[i] * inv;"),
    }
    blocks = _q8k_golden()
    g = np.random.default_rng(15)
    xs = g.standard_normal(256).astype(np.float32)
    caught = {}
    for name, (a, b) in mutants.items():
        assert a in src, name
        path = tmp_path / f"q8_{abs(hash(name))}.c"
        path.write_text(src.replace(a, b))
        so = str(path) + ".so"
        subprocess.run(["gcc", "-O1", "-fPIC", "-shared", str(path), "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        lib.oracle_q8k_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]

        def quant(x):
            q = np.zeros(256, np.int8)
            d = np.zeros(1, np.float32)
            x = np.ascontiguousarray(x, np.float32)
            lib.oracle_q8k_quantize(x.ctypes.data_as(ctypes.c_void_p), 256, q.ctypes.data_as(ctypes.c_void_p),
                                    d.ctypes.data_as(ctypes.c_void_p))
            return q, d

        bad = False
        for blk in blocks:
            x = np.zeros(256, np.float32)
            x[:len(blk["x"])] = blk["x"]
            q, d = quant(x)
            bad |= list(q[:len(blk["q"])]) != [int(v) for v in blk["q"]]
            if "/" not in blk["d"]:
                bad |= d[0] != np.float32(blk["d"])
        q0, _ = quant(xs)
        q1, _ = quant((xs.astype(np.float64) * 2.0 ** -90).astype(np.float32))
        bad |= not np.array_equal(q0, q1)
        caught[name] = bad
    assert all(caught.values()), caught
