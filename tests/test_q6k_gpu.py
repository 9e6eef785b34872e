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
