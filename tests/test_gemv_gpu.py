"""GPU parity of the decode GEMV (batch 1 .. 16) against the fp64 CPU oracle.

Every case draws its inputs from `synth` (seeded), runs the CUDA kernels
through the C ABI (via the thin binding) and compares element by element with
the oracle within the stated tolerances."""
import numpy as np
import pytest

import synth
from parity import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    import q4_dequant_gemv_gb300 as q4k
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    return q4k, oracle


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(q4k, W, x, **kw):
    y = q4k.gemv(_dev(W), _dev(x), **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy()


SMALL = [
    (1, 256, 1), (7, 256, 1), (33, 512, 1), (64, 768, 2), (100, 1280, 5), (200, 2048, 4),
    (129, 3584, 1), (65, 3584, 3), (250, 512, 8), (90, 1024, 9), (17, 2560, 16), (300, 4096, 5),
]


@pytest.mark.parametrize("N,K,B", SMALL)
def test_small_shapes(env, N, K, B):
    q4k, oracle = env
    W = synth.q4k_weights(N, K, (N, K, B))
    x = synth.normal_f32((B, K), (N, K, B, 1))
    y = _run(q4k, W, x)
    assert_close(y, oracle.gemv(W, x, N, K), x, K, f"N={N} K={K} B={B}")


@pytest.mark.parametrize("split", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("B", [1, 5])
def test_forced_split(env, split, B):
    q4k, oracle = env
    N, K = 150, 2304
    W = synth.q4k_weights(N, K, (17, split))
    x = synth.normal_f32((B, K), (18, split))
    y = _run(q4k, W, x, split_k=split)
    assert_close(y, oracle.gemv(W, x, N, K), x, K, f"split={split}")


def test_split_results_agree(env):
    """Split-K on/off only re-associates fp32 sums: results agree within tolerance
    and each configuration is deterministic run to run."""
    q4k, oracle = env
    N, K = 256, 3584
    W = synth.q4k_weights(N, K, 19)
    x = synth.normal_f32((1, K), 20)
    ys = {s: _run(q4k, W, x, split_k=s) for s in (1, 2, 7)}
    ref = oracle.gemv(W, x, N, K)
    for s, y in ys.items():
        assert_close(y, ref, x, K, f"split {s}")
        assert np.array_equal(y, _run(q4k, W, x, split_k=s))


def test_config0_4096(env):
    """4096 x 4096, batch 1 (16 super-blocks per row), every output."""
    q4k, oracle = env
    N = K = 4096
    W = synth.q4k_weights(N, K, (0, 0))
    x = synth.normal_f32((1, K), (0, 1))
    assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, "config0")


@pytest.mark.parametrize("B", [1, 2, 5, 9])
def test_qwen_layer0_all_matrices(env, B):
    """All seven Qwen2.5-7B-shaped matrices of layer 0, every output, batch 1/2/5/9."""
    q4k, oracle = env
    for name, N, K, W in synth.qwen_layer_weights(0):
        x = synth.normal_f32((B, K), (0, 2, B, N, K))
        assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, f"{name} B={B}")


def test_batch_rows_independent(env):
    """Row b of a batch-5 product matches the batch-1 product of x[b]."""
    q4k, oracle = env
    N, K = 320, 3584
    W = synth.q4k_weights(N, K, 23)
    x = synth.normal_f32((5, K), 24)
    y5 = _run(q4k, W, x)
    ref = oracle.gemv(W, x, N, K)
    for b in range(5):
        y1 = _run(q4k, W, x[b:b + 1])
        assert_close(y1, ref[b:b + 1], x[b:b + 1], K, f"b={b}")
        assert_close(y5[b:b + 1], ref[b:b + 1], x[b:b + 1], K, f"b={b}")


@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("scale", [1e-37, 1e-30, 1e-6, 1e6, 1e30])
def test_extreme_activation_scales(env, scale, B):
    """Any finite fp32 x works: batch 2 rescales by a power of two before the
    fp16 split, batch 1 quantizes against each super-block's own max|x|."""
    q4k, oracle = env
    N, K = 96, 1024
    W = synth.q4k_weights(N, K, 25)
    x = (synth.normal_f32((B, K), 26) * np.float32(scale)).astype(np.float32)
    assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, f"scale {scale} B={B}")


def _int8_parts(x):
    """The batch-1 integer path's representation of x, retaken in numpy fp32:
    per super-block a = max|x| (with x and a scaled by p = 2^64 below 2^-64, else
    p = 1), q = (p x) * (127 / (p a)), xh = rint(q), xl = rint((q - xh) * 254);
    returns x~ = ((p a) / 127 / 254)(254 xh + xl) / p in fp64."""
    K = x.size
    blocks = x.reshape(K // 256, 256).astype(np.float32)
    out = np.zeros((K // 256, 256), np.float64)
    for i, v in enumerate(blocks):
        a = np.float32(np.max(np.abs(v)))
        if a == 0:
            continue
        pre = np.float32(2.0 ** 64) if a < np.float32(2.0 ** -64) else np.float32(1)
        inv = np.float32(127) / np.float32(a * pre)
        q = (v * pre).astype(np.float32) * inv
        xh = np.rint(q)
        xl = np.rint((q - xh).astype(np.float32) * np.float32(254))
        u = np.float32(np.float32(np.float32(a * pre) / np.float32(127)) / np.float32(254))
        out[i] = np.float64(u) / np.float64(pre) * (254.0 * xh.astype(np.float64) + xl.astype(np.float64))
    return out.reshape(K)


@pytest.mark.parametrize("N,K,seed", [(300, 3584, 41), (129, 18944, 42), (640, 4096, 43)])
def test_batch1_integer_path_is_exact(env, N, K, seed):
    """Batch 1 runs integer dot products on int8 parts of x.  Given the same
    parts (retaken in numpy), the kernel's result must equal the fp64 product
    of the dequantized weights with them up to fp32 rounding of the
    per-super-block combine: |dy| <= 1e-5 sum_k |w||x~| (an integer overflow or a
    misplaced part would be off by far more)."""
    q4k, oracle = env
    W = synth.q4k_weights(N, K, (seed, 1))
    x = synth.normal_f32((1, K), (seed, 2))
    x[0, 5] = 40.0          # one super-block with a large max, so most parts are small
    x[0, 512:768] = 0.0     # an all-zero super-block
    xt = _int8_parts(x[0])
    D = oracle.dequant_matrix(W, N, K)
    ref = D @ xt
    bound = 1e-5 * (np.abs(D) @ np.abs(xt)) + 1e-30
    y = _run(q4k, W, x)[0]
    assert np.all(np.abs(y - ref) <= bound), f"max excess {np.max(np.abs(y - ref) - bound)}"
    # and the tensor-core path on the same input stays within the stated tolerance
    yt = _run(q4k, W, x, tensor_core=True)
    assert_close(yt[None, :] if yt.ndim == 1 else yt, oracle.gemv(W, x, N, K), x, K, "tensor-core batch 1")


def test_mixed_magnitudes_within_row(env):
    """One huge entry next to normal ones in the same chunk."""
    q4k, oracle = env
    N, K = 64, 1024
    W = synth.q4k_weights(N, K, 27)
    x = synth.normal_f32((1, K), 28)
    x[0, 300] = 3.0e4
    assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, "spike")


def test_zero_and_one_hot(env):
    q4k, oracle = env
    N, K = 70, 768
    W = synth.q4k_weights(N, K, 29)
    y0 = _run(q4k, W, np.zeros((1, K), np.float32))
    assert np.all(y0 == 0.0)
    dense = oracle.dequant_matrix(W, N, K)
    for c in (0, 31, 32, 255, 256, 767):
        e = np.zeros((1, K), np.float32)
        e[0, c] = 1.0
        y = _run(q4k, W, e)[0]
        np.testing.assert_allclose(y, dense[:, c], rtol=1e-6, atol=1e-7)


def test_all_ones_row_sums(env):
    q4k, oracle = env
    N, K = 40, 1024
    W = synth.q4k_weights(N, K, 30)
    x = np.ones((1, K), np.float32)
    assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, "ones")


def test_output_guards_untouched(env):
    """Writes stay inside y (sentinels around the output are intact)."""
    q4k, oracle = env
    N, K, B = 77, 512, 3
    W = _dev(synth.q4k_weights(N, K, 31))
    x = _dev(synth.normal_f32((B, K), 32))
    buf = torch.full((B * N + 2048,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[1024:1024 + B * N].view(B, N)
    q4k.gemv(W, x, y)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + B * N:] == 12345.0)


def test_n_zero_is_noop(env):
    q4k, _ = env
    W = torch.empty((0, 144), dtype=torch.uint8, device="cuda")
    x = torch.randn(1, 256, device="cuda")
    y = torch.empty((1, 0), device="cuda")
    q4k.gemv(W, x, y)


def test_pdl_and_streams_bitwise_equal(env):
    """The PDL launch path and a side stream give bitwise the same result."""
    q4k, oracle = env
    N, K = 512, 3584
    W = _dev(synth.q4k_weights(N, K, 33))
    x = _dev(synth.normal_f32((1, K), 34))
    y_ref = q4k.gemv(W, x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y_pdl = torch.empty_like(y_ref)
        for _ in range(3):
            q4k.gemv(W, x, y_pdl, pdl=True)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(y_ref, y_pdl)


def test_graph_capture_replay(env):
    """A chain of GEMVs captured in a CUDA graph replays to the eager results."""
    q4k, oracle = env
    mats = [(synth.q4k_weights(n, k, (35, i)), n, k) for i, (n, k) in enumerate([(512, 3584), (3584, 3584), (256, 1024)])]
    Ws = [_dev(w) for w, _, _ in mats]
    xs = [_dev(synth.normal_f32((1, k), (36, i))) for i, (_, _, k) in enumerate(mats)]
    ys = [torch.empty((1, n), device="cuda") for _, n, _ in mats]
    for W, x, y in zip(Ws, xs, ys):
        q4k.gemv(W, x, y)
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for W, x, y in zip(Ws, xs, ys):
                q4k.gemv(W, x, y, pdl=True)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, ys):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B", [1, 5])
def test_grouped_qkv_and_gate_up(env, B):
    """Fused dispatch (q/k/v in one launch, gate/up in one launch) against the oracle,
    and bitwise equal to per-matrix launches when the split is forced the same."""
    q4k, oracle = env
    layer = synth.qwen_layer_weights(5)
    mats = {name: (N, K, W) for name, N, K, W in layer}
    for names in (("q", "k", "v"), ("gate", "up")):
        K = mats[names[0]][1]
        x = synth.normal_f32((B, K), (77, B, K))
        Ws = [_dev(mats[n][2]) for n in names]
        xd = _dev(x)
        ys = q4k.gemv_grouped(Ws, xd)
        torch.cuda.synchronize()
        for n, y in zip(names, ys):
            N = mats[n][0]
            assert_close(y.cpu().numpy(), oracle.gemv(mats[n][2], x, N, K), x, K, f"grouped {n} B={B}")
        ys2 = q4k.gemv_grouped(Ws, xd, split_k=2)
        for W, y2 in zip(Ws, ys2):
            assert torch.equal(y2, q4k.gemv(W, xd, split_k=2))


def test_grouped_ragged_and_empty(env):
    q4k, oracle = env
    K = 1024
    shapes = [130, 0, 7, 300]
    Wn = [synth.q4k_weights(N, K, (78, i)) for i, N in enumerate(shapes)]
    x = synth.normal_f32((3, K), 79)
    ys = q4k.gemv_grouped([_dev(W) if W.size else torch.empty((0, 576), dtype=torch.uint8, device="cuda") for W in Wn],
                          _dev(x))
    torch.cuda.synchronize()
    for N, W, y in zip(shapes, Wn, ys):
        if N:
            assert_close(y.cpu().numpy(), oracle.gemv(W, x, N, K), x, K, f"grouped N={N}")


def test_device_error_flags_clear(env):
    q4k, _ = env
    torch.cuda.synchronize()
    assert q4k.device_error_flags() == 0


def test_auto_split_above_eight(env):
    """Few row tiles and a long K: the planner may split K over up to 16 CTAs
    (non-portable cluster sizes); results stay within the tolerance."""
    q4k, oracle = env
    N, K = 3584, 18944
    plan = q4k.gemv_plan(N, K, 1)
    assert 1 <= plan["split_k"] <= 16
    W = synth.q4k_weights(N, K, (96, 1))
    for B in (1, 3, 6):
        x = synth.normal_f32((B, K), (96, 2, B))
        assert_close(_run(q4k, W, x), oracle.gemv(W, x, N, K), x, K, f"down-shaped B={B} split {plan['split_k']}")
    N2 = 600
    W2 = W[:N2]
    x = synth.normal_f32((2, K), (96, 3))
    assert_close(_run(q4k, W2, x), oracle.gemv(W2, x, N2, K), x, K, "5 tiles, long K")


# ---------------------------------------------------------------- Q8_K activations (batch 1, on request)
def _q8k_input(K, seed):
    x = synth.normal_f32((1, K), (seed, 2))
    x[0, 0:256] *= np.float32(1e-30)        # a tiny block
    x[0, 256:512] = 0.0                     # an all-zero block
    x[0, 700] = 55.0                        # a block with one large entry
    x[0, 1024:1280] = np.float32(127.0) * np.round(x[0, 1024:1280])   # codes on exact integers
    return x


@pytest.mark.parametrize("N,K,seed", [(300, 3584, 51), (129, 18944, 52), (640, 4096, 53), (1, 1536, 54)])
def test_q8k_matches_oracle(env, N, K, seed):
    """Q4K_FLAG_Q8K_X: the kernel quantizes x with the oracle's rule (same fp32
    decisions) and multiplies exactly in integers; against the oracle's
    Q4_K x Q8_K product it may differ only by fp32 rounding of the
    per-block combine, and against the exact product by the quantization bound
    sum_k |w| d/2."""
    q4k, oracle = env
    W = synth.q4k_weights(N, K, (seed, 1))
    x = _q8k_input(K, seed)
    y = _run(q4k, W, x, q8k=True)[0]
    q, d = oracle.q8k_quantize(x[0], K)
    ref = oracle.gemv_q8k(W, q, d, N, K)
    D = oracle.dequant_matrix(W, N, K)
    xt = np.repeat(d.astype(np.float64), 256) * q.astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-5 * (np.abs(D) @ np.abs(xt)) + 1e-30)
    exact = oracle.gemv(W, x, N, K)[0]
    bound = (np.abs(D) @ (np.repeat(d.astype(np.float64), 256) / 2)) * (1 + 1e-4) + 1e-5 * (np.abs(D) @ np.abs(xt))
    assert np.all(np.abs(y - exact) <= bound)


def test_q8k_grouped_and_guards(env):
    q4k, oracle = env
    K = 3584
    Ws = [synth.q4k_weights(N, K, (55, N)) for N in (256, 129)]
    x = _q8k_input(K, 56)
    ys = q4k.gemv_grouped([_dev(W) for W in Ws], _dev(x), q8k=True)
    torch.cuda.synchronize()
    q, d = oracle.q8k_quantize(x[0], K)
    for W, yg in zip(Ws, ys):
        N = W.shape[0]
        ref = oracle.gemv_q8k(W, q, d, N, K)
        D = oracle.dequant_matrix(W, N, K)
        xt = np.repeat(d.astype(np.float64), 256) * q.astype(np.float64)
        assert np.all(np.abs(yg.cpu().numpy()[0] - ref) <= 1e-5 * (np.abs(D) @ np.abs(xt)) + 1e-30)
    W = _dev(Ws[0])
    with pytest.raises(q4k.Q4KError):
        q4k.gemv(W, _dev(synth.normal_f32((2, K), 57)), q8k=True)          # batch 1 only
    with pytest.raises(q4k.Q4KError):
        q4k.gemv(W, _dev(x), q8k=True, tensor_core=True)                   # one inner product at a time


# ---------------------------------------------------------------- 16-row tiles (batch 1)
ROWS16 = [
    (1, 256), (15, 512), (16, 1792), (17, 3584), (100, 1792), (333, 2048), (129, 8192), (4608, 3584),
    (5000, 1536),
]


@pytest.mark.parametrize("N,K", ROWS16)
def test_rows16_shapes(env, N, K):
    """The 16-row-tile kernel (one CTA per 16 rows over the whole K, the K split
    between its warps): ragged row counts, 1 to 32 super-blocks per row (a
    stage holds 7: full, partial and single-super-block stages), more tiles
    than resident CTAs (5000 rows: CTAs take two tiles), against the oracle;
    deterministic run to run."""
    q4k, oracle = env
    W = synth.q4k_weights(N, K, (61, N, K))
    x = synth.normal_f32((1, K), (62, N, K))
    x[0, :256] *= np.float32(1e-3)          # super-blocks of very different size
    y = _run(q4k, W, x, rows16=True)
    assert_close(y, oracle.gemv(W, x, N, K), x, K, f"rows16 N={N} K={K}")
    assert np.array_equal(y, _run(q4k, W, x, rows16=True))


def test_rows16_is_the_automatic_choice(env):
    """Batch 1 with too few 128-row tiles and K <= 8192 takes the 16-row kernel
    (the plan reports 16-row tiles and no split); a long K or a larger batch
    keeps the 128-row kernel; both agree within the tolerance."""
    q4k, oracle = env
    assert q4k.gemv_plan(4608, 3584, 1)["rows_per_tile"] == 16
    assert q4k.gemv_plan(3584, 3584, 1)["split_k"] == 1
    assert q4k.gemv_plan(3584, 18944, 1)["rows_per_tile"] == 128
    assert q4k.gemv_plan(4608, 3584, 2)["rows_per_tile"] == 128
    assert q4k.gemv_plan(37888, 3584, 1)["rows_per_tile"] == 128    # enough 128-row tiles
    N, K = 640, 4096
    W = synth.q4k_weights(N, K, 63)
    x = synth.normal_f32((1, K), 64)
    ref = oracle.gemv(W, x, N, K)
    y16, y128 = _run(q4k, W, x), _run(q4k, W, x, split_k=5)
    assert_close(y16, ref, x, K, "automatic (16-row)")
    assert_close(y128, ref, x, K, "forced split (128-row)")
    assert np.array_equal(y16, _run(q4k, W, x, rows16=True))


def test_rows16_grouped_q8k_and_guards(env):
    """Fused q/k/v-style launch with ragged and empty matrices on the 16-row
    kernel (batch 1), its Q8_K mode against the oracle's Q8_K product, the
    output guards, and the argument checks of the flag."""
    q4k, oracle = env
    K = 1024
    shapes = [130, 0, 7, 300]
    Wn = [synth.q4k_weights(N, K, (65, i)) for i, N in enumerate(shapes)]
    x = synth.normal_f32((1, K), 66)
    Wd = [_dev(W) if W.size else torch.empty((0, 576), dtype=torch.uint8, device="cuda") for W in Wn]
    ys = q4k.gemv_grouped(Wd, _dev(x), rows16=True)
    torch.cuda.synchronize()
    for N, W, y in zip(shapes, Wn, ys):
        if N:
            assert_close(y.cpu().numpy(), oracle.gemv(W, x, N, K), x, K, f"rows16 grouped N={N}")
    # Q8_K activations on the same kernel
    xq = _q8k_input(K, 67)
    q, d = oracle.q8k_quantize(xq[0], K)
    yq = _run(q4k, Wn[3], xq, q8k=True, rows16=True)[0]
    D = oracle.dequant_matrix(Wn[3], 300, K)
    xt = np.repeat(d.astype(np.float64), 256) * q.astype(np.float64)
    assert np.all(np.abs(yq - oracle.gemv_q8k(Wn[3], q, d, 300, K)) <= 1e-5 * (np.abs(D) @ np.abs(xt)) + 1e-30)
    # writes stay inside y
    N = 77
    buf = torch.full((N + 2048,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[1024:1024 + N].view(1, N)
    q4k.gemv(_dev(Wn[3][:N]), _dev(x), y, rows16=True)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + N:] == 12345.0)
    # the flag is batch 1, integer path, K <= 8192 only
    W = _dev(Wn[0])
    with pytest.raises(q4k.Q4KError):
        q4k.gemv(W, _dev(synth.normal_f32((2, K), 68)), rows16=True)
    with pytest.raises(q4k.Q4KError):
        q4k.gemv(W, _dev(x), rows16=True, tensor_core=True)
    Kl = 8448
    with pytest.raises(q4k.Q4KError):
        q4k.gemv(_dev(synth.q4k_weights(16, Kl, 69)), _dev(synth.normal_f32((1, Kl), 70)), rows16=True)


def test_pdl_ten_cta_clusters_bitwise_equal(env):
    """The down-projection shape (K split over clusters of more than 8 CTAs)
    launched with PDL, back to back on a side stream and captured in a graph,
    gives bitwise the results of plain launches, and stays within the
    tolerance of the oracle on sampled rows."""
    q4k, oracle = env
    N, K = 3584, 18944
    assert q4k.gemv_plan(N, K, 1)["split_k"] > 8
    W = synth.q4k_weights(N, K, (91, 1))
    Wd = _dev(W)
    xs = [_dev(synth.normal_f32((1, K), (92, i))) for i in range(3)]
    ref = [q4k.gemv(Wd, x) for x in xs]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ys = [torch.empty_like(r) for r in ref]
    with torch.cuda.stream(s):
        for x, y in zip(xs, ys):
            q4k.gemv(Wd, x, y, pdl=True, stream=s)
    s.synchronize()
    for a, b in zip(ref, ys):
        assert torch.equal(a, b)
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for x, y in zip(xs, ys):
                q4k.gemv(Wd, x, y, pdl=True, stream=s)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, ys):
        assert torch.equal(a, b)
    rows = np.array([0, 1, 127, 128, 1000, N - 1])
    x0 = xs[0].cpu().numpy()
    assert_close(ref[0].cpu().numpy()[:, rows], oracle.gemv_rows(W, x0, N, K, rows), x0, K, "down shape, PDL")
