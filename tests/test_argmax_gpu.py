"""GPU parity of the fused LM-head + greedy argmax.

Bar: idx equals the oracle's scalar argmax over the logits the kernel itself
compared (bit-exact), and equals the oracle's argmax of its own fp64 logits
wherever the oracle's top-2 margin exceeds the absolute tolerance.  The planted
rows have closed-form answers."""
import numpy as np
import pytest

import synth
from parity import assert_close, tol_limits, top2_margin

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


def _argmax(q4k, W, x, want_logits=True):
    B = x.shape[0]
    N = W.shape[0]
    Wd, xd = _dev(W), _dev(x)
    idx = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    logits = torch.empty((B, N), dtype=torch.float32, device="cuda") if want_logits else None
    q4k.gemv_argmax(Wd, xd, idx, logits=logits)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (logits.cpu().numpy() if want_logits else None)


def _check(q4k, oracle, W, x, N, K, what):
    idx, lg = _argmax(q4k, W, x)
    ref = oracle.gemv(W, x, N, K)
    assert_close(lg, ref, x, K, what)
    lim = tol_limits(ref, x, K)
    for b in range(x.shape[0]):
        assert idx[b] == oracle.argmax(lg[b]), f"{what} b={b}: not the first max of the kernel's logits"
        if top2_margin(ref[b]) > lim[b]:
            assert idx[b] == oracle.argmax(ref[b]), f"{what} b={b}: differs from oracle argmax"
    # the plain entry point (no logits) gives the same indices
    idx2, _ = _argmax(q4k, W, x, want_logits=False)
    assert np.array_equal(idx, idx2)
    return idx, lg


@pytest.mark.parametrize("N,K,B", [(1, 256, 1), (7, 512, 2), (100, 1024, 1), (1000, 3584, 5), (4097, 2048, 3),
                                   (20000, 3584, 1), (300, 3584, 16)])
def test_argmax_shapes(env, N, K, B):
    q4k, oracle = env
    W = synth.q4k_weights(N, K, (N, K, 5))
    x = synth.normal_f32((B, K), (N, K, 6))
    _check(q4k, oracle, W, x, N, K, f"N={N} K={K} B={B}")


def test_logits_equal_gemv_output(env):
    """The argmax kernel's logits are bitwise the q4k_gemv output (same plan)."""
    q4k, oracle = env
    N, K = 5000, 3584
    W = synth.q4k_weights(N, K, 41)
    x = synth.normal_f32((2, K), 42)
    _, lg = _argmax(q4k, W, x)
    y = q4k.gemv(_dev(W), _dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(lg, y.cpu().numpy())


def _planted_row(oracle, x, K):
    nb = K // 256
    blocks = []
    for b in range(nb):
        q = np.where(x[b * 256:(b + 1) * 256] > 0, 15, 0)
        blocks.append(oracle.pack_block(0x3C00, 0x0000, [63] * 8, [0] * 8, q))
    return np.concatenate(blocks)


@pytest.mark.parametrize("where", [0, 1234, 152063])
def test_lm_head_planted_unique_max(env, where):
    """152064 x 3584 with a planted row whose value is 945 * sum(x>0) in closed form."""
    q4k, oracle = env
    N, K = 152064, 3584
    W = synth.q4k_weights(N, K, (3, 0))
    x = synth.normal_f32((1, K), (3, 1))
    W[where] = _planted_row(oracle, x[0], K)
    idx, lg = _argmax(q4k, W, x)
    assert idx[0] == where
    exact = 945.0 * x[0][x[0] > 0].astype(np.float64).sum()
    assert abs(lg[0, where] - exact) <= 2e-3 * exact


def test_planted_ties_lowest_index(env):
    q4k, oracle = env
    N, K = 3000, 1024
    W = synth.q4k_weights(N, K, 43)
    x = synth.normal_f32((2, K), 44)
    row = _planted_row(oracle, x[0], K)
    for r in (2999, 64, 1500, 65):
        W[r] = row
    idx, lg = _argmax(q4k, W, x)
    assert idx[0] == 64
    assert lg[0, 64] == lg[0, 65] == lg[0, 1500] == lg[0, 2999]


def test_identical_rows_give_zero(env):
    q4k, oracle = env
    N, K = 500, 512
    one = synth.q4k_weights(1, K, 45)
    W = np.repeat(one, N, axis=0)
    x = synth.normal_f32((1, K), 46)
    idx, _ = _argmax(q4k, W, x)
    assert idx[0] == 0


@pytest.mark.parametrize("B", [1, 5])
def test_lm_head_full(env, B):
    """LM head 152064 x 3584, batch 1 and 5: every logit against the oracle."""
    q4k, oracle = env
    N, K = 152064, 3584
    W = synth.q4k_weights(N, K, (3, 0))
    x = synth.normal_f32((B, K), (3, 2, B))
    _check(q4k, oracle, W, x, N, K, f"lm_head B={B}")


def test_graph_capture_argmax(env):
    """The argmax (with its stream-ordered scratch) replays inside a CUDA graph."""
    q4k, oracle = env
    N, K = 4096, 3584
    W = _dev(synth.q4k_weights(N, K, 47))
    x = _dev(synth.normal_f32((1, K), 48))
    idx = torch.empty(1, dtype=torch.int32, device="cuda")
    q4k.gemv_argmax(W, x, idx)
    torch.cuda.synchronize()
    eager = idx.clone()
    idx.fill_(-1)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            q4k.gemv_argmax(W, x, idx)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, idx)
    assert q4k.device_error_flags() == 0
