"""GPU parity of the Q6_K decode GEMV against the fp64 CPU oracle (same
tolerances as the Q4_K GEMV)."""
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
    torch.cuda.set_device(0)
    return q4k, oracle


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(q4k, W, x):
    y = q4k.q6k_gemv(_dev(W), _dev(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


# (N, K, B): ragged row counts, every warps-per-row choice of the direct kernel (few rows -> up to 8
# warps per row), the staged path (8-row tiles through shared memory in K-slices of up to 16 blocks,
# batch <= 4) with and without a remainder of rows for the direct kernel, and shapes that only take
# the direct kernel (batch > 4, fewer than 8 rows)
SHAPES = [(1, 256, 1), (7, 512, 2), (129, 3584, 1), (300, 4096, 5), (512, 3584, 1), (1000, 2048, 16),
          (65, 18944, 3), (3584, 3584, 1), (37, 768, 9), (64, 1024, 3), (29, 2560, 4),
          # K-sliced stages: several slices per tile, a short last slice, batch 1 and 4
          (3584, 18944, 1), (40, 4608, 4), (16, 4352, 1),
          # batch 1 in 16-row tiles: a tail of 8 rows after whole tiles, one tile plus a tail;
          # batch 1 back on 8-row tiles: rows longer than a 48 KB slice, fewer than 16 rows
          (1000, 3584, 1), (24, 3584, 1), (136, 4096, 1), (12, 3584, 1)]


@pytest.mark.parametrize("N,K,B", SHAPES)
def test_q6k_shapes(env, N, K, B):
    q4k, oracle = env
    W = synth.q6k_weights(N, K, (N, K, 71))
    x = synth.normal_f32((B, K), (N, K, B, 72))
    assert_close(_run(q4k, W, x), oracle.q6k_gemv(W, x, N, K), x, K, f"q6k N={N} K={K} B={B}")


@pytest.mark.parametrize("B", [1, 5])
def test_q6k_lm_head_sampled(env, B):
    """A Q6_K LM head of Qwen2.5-7B's shape (152064 x 3584, 447 MB): sampled rows, every batch row."""
    q4k, oracle = env
    N, K = 152064, 3584
    W = synth.q6k_weights(N, K, (73, B))
    x = synth.normal_f32((B, K), (74, B))
    y = _run(q4k, W, x)
    rows = np.unique(np.concatenate([np.random.default_rng(B).integers(0, N, 64), [0, 1, 127, 128, N - 1]]))
    assert_close(y[:, rows], oracle.q6k_gemv_rows(W, x, N, K, rows), x, K, f"q6k lm head B={B}")


def test_q6k_deterministic_and_guards(env):
    q4k, oracle = env
    N, K = 200, 1024
    W = _dev(synth.q6k_weights(N, K, 75))
    x = _dev(synth.normal_f32((2, K), 76))
    y1 = q4k.q6k_gemv(W, x)
    y2 = q4k.q6k_gemv(W, x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    with pytest.raises(q4k.Q4KError):
        q4k.q6k_gemv(W, _dev(synth.normal_f32((17, K), 77)))          # batch above 16
    xm = torch.zeros(2 * K + 4, dtype=torch.float32, device="cuda")[1:2 * K + 1].view(2, K)
    with pytest.raises(q4k.Q4KError):
        q4k.q6k_gemv(W, xm)                                          # x not 16-byte aligned
    empty = q4k.q6k_gemv(torch.zeros((0, (K // 256) * 210), dtype=torch.uint8, device="cuda"), x)
    assert empty.shape == (2, 0)


# ---------------------------------------------------------------- planar form (q6k_repack_planar / q6k_gemv_planar)
def _planar(q4k, W, K):
    Wp = q4k.q6k_repack_planar(_dev(W), K)
    torch.cuda.synchronize()
    return Wp


def test_q6k_planar_layout(env):
    """The planar form holds each block's bytes 0..207 unchanged in the QS plane
    and the d bytes of the row's blocks, zero-padded to 16 bytes, in the D plane."""
    q4k, _ = env
    for N, K in ((5, 256), (37, 3584), (130, 2048), (3, 18944)):
        W = synth.q6k_weights(N, K, (81, N, K))
        nb = K // 256
        dp = -(-2 * nb // 16) * 16
        Wp = _planar(q4k, W, K).cpu().numpy()
        assert Wp.size == q4k.q6k_planar_bytes(N, K) == N * (nb * 208 + dp)
        blocks = W.reshape(N, nb, 210)
        assert np.array_equal(Wp[:N * nb * 208].reshape(N, nb, 208), blocks[:, :, :208])
        D = Wp[N * nb * 208:].reshape(N, dp)
        assert np.array_equal(D[:, :2 * nb].reshape(N, nb, 2), blocks[:, :, 208:210])
        assert not D[:, 2 * nb:].any()


# row tiles of 128 with a tail, one tile, K splits over clusters (few tiles), x in several chunks (long
# K), batch 1..16 (launches of up to four batch rows)
PLANAR = [(1, 256, 1), (7, 512, 1), (129, 3584, 1), (300, 4096, 3), (1000, 3584, 1), (24, 18944, 1),
          (3584, 18944, 1), (1500, 2304, 4), (200, 1024, 5), (136, 4096, 16), (2000, 3584, 2), (640, 11008, 4)]


@pytest.mark.parametrize("N,K,B", PLANAR)
def test_q6k_planar_shapes(env, N, K, B):
    q4k, oracle = env
    W = synth.q6k_weights(N, K, (N, K, 82))
    x = synth.normal_f32((B, K), (N, K, B, 83))
    x[:, :256] *= np.float32(1e-3)      # blocks of x of very different size
    Wp = _planar(q4k, W, K)
    y = q4k.q6k_gemv_planar(Wp, _dev(x), N)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.q6k_gemv(W, x, N, K), x, K, f"q6k planar N={N} K={K} B={B}")
    y2 = q4k.q6k_gemv_planar(Wp, _dev(x), N)
    assert torch.equal(y, y2)


def test_q6k_planar_lm_head_sampled(env):
    """The 152064 x 3584 LM head on the planar form at batch 1: sampled rows
    against the oracle, every row against the GGUF-form kernel."""
    q4k, oracle = env
    N, K = 152064, 3584
    W = synth.q6k_weights(N, K, (84, 1))
    x = synth.normal_f32((1, K), (85, 1))
    Wp = _planar(q4k, W, K)
    y = q4k.q6k_gemv_planar(Wp, _dev(x), N).cpu().numpy()
    rows = np.unique(np.concatenate([np.random.default_rng(3).integers(0, N, 64), [0, 1, 127, 128, N - 1]]))
    ref = oracle.q6k_gemv_rows(W, x, N, K, rows)
    assert_close(y[:, rows], ref, x, K, "q6k planar lm head")
    y_gguf = _run(q4k, W, x)
    scale = np.abs(y_gguf).max()
    assert np.abs(y - y_gguf).max() <= 2e-3 * scale


def test_q6k_planar_extremes_and_guards(env):
    q4k, oracle = env
    N, K = 260, 1536
    W = synth.q6k_weights(N, K, 86)
    x = synth.normal_f32((1, K), 87)
    x[0, 0:256] *= np.float32(1e-30)     # below 2^-64 relative scale
    x[0, 256:512] = 0.0                   # an all-zero block
    x[0, 700] = 3.0e4                     # one large entry
    Wp = _planar(q4k, W, K)
    y = q4k.q6k_gemv_planar(Wp, _dev(x), N)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.q6k_gemv(W, x, N, K), x, K, "q6k planar extremes")
    assert np.all(q4k.q6k_gemv_planar(Wp, _dev(np.zeros((1, K), np.float32)), N).cpu().numpy() == 0.0)
    # writes stay inside y
    buf = torch.full((N + 2048,), 12345.0, dtype=torch.float32, device="cuda")
    q4k.q6k_gemv_planar(Wp, _dev(x), N, buf[1024:1024 + N].view(1, N))
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 12345.0) and torch.all(buf[1024 + N:] == 12345.0)
    with pytest.raises(q4k.Q4KError):
        q4k.q6k_gemv_planar(Wp, _dev(synth.normal_f32((17, K), 88)), N)      # batch above 16
    xm = torch.zeros(K + 4, dtype=torch.float32, device="cuda")[1:K + 1].view(1, K)
    with pytest.raises(q4k.Q4KError):
        q4k.q6k_gemv_planar(Wp, xm, N)                                     # x not 16-byte aligned
    nbytes = q4k.q6k_planar_bytes(N, K)
    both = torch.zeros(W.size + nbytes + 16, dtype=torch.uint8, device="cuda")
    both[:W.size] = _dev(W.reshape(-1))
    with pytest.raises(q4k.Q4KError):                                      # W and Wp overlap
        q4k.q6k_repack_planar(both[:W.size].view(N, -1), K, both[16:16 + nbytes])
    empty = q4k.q6k_gemv_planar(torch.zeros(0, dtype=torch.uint8, device="cuda"), _dev(x), 0)
    assert empty.shape == (1, 0)


def test_q6k_planar_graph_capture(env):
    """Planar GEMVs captured in a CUDA graph on a side stream replay to the eager results."""
    q4k, _ = env
    mats = [(synth.q6k_weights(n, k, (89, i)), n, k) for i, (n, k) in enumerate([(640, 3584), (300, 18944)])]
    Wps = [q4k.q6k_repack_planar(_dev(w), k) for w, _, k in mats]
    xs = [_dev(synth.normal_f32((1, k), (90, i))) for i, (_, _, k) in enumerate(mats)]
    ys = [torch.empty((1, n), device="cuda") for _, n, _ in mats]
    for Wp, x, y, (_, n, _) in zip(Wps, xs, ys, mats):
        q4k.q6k_gemv_planar(Wp, x, n, y)
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for Wp, x, y, (_, n, _) in zip(Wps, xs, ys, mats):
                q4k.q6k_gemv_planar(Wp, x, n, y, stream=s)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, ys):
        assert torch.equal(a, b)
