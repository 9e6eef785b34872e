"""GPU parity of chains (q4k_chain_*): a sequence of GEMV steps in one
persistent launch, checked against the fp64 CPU oracle step by step, including
steps that read an earlier step's output."""
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


def _layer_steps(B, layer=0):
    """Qwen2.5-7B-shaped layer as four steps (q/k/v, o, gate/up, down), each with its own x."""
    mats = {name: (N, K, W) for name, N, K, W in synth.qwen_layer_weights(layer)}
    plan = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
    host, dev = [], []
    for si, names in enumerate(plan):
        K = mats[names[0]][1]
        x = synth.normal_f32((B, K), (90, layer, si, B))
        xd = _dev(x)
        groups = []
        for n in names:
            N, _, W = mats[n]
            groups.append((_dev(W), torch.empty((B, N), device="cuda")))
        host.append((x, [(mats[n][2], mats[n][0]) for n in names]))
        dev.append((xd, groups))
    return host, dev


@pytest.mark.parametrize("B", [1, 5, 9])
def test_layer_chain_matches_oracle(env, B):
    q4k, oracle = env
    host, dev = _layer_steps(B)
    ch = q4k.Chain(dev, B)
    ch.run()
    torch.cuda.synchronize()
    for (x, hg), (_, dg) in zip(host, dev):
        K = x.shape[1]
        for (W, N), (_, y) in zip(hg, dg):
            assert_close(y.cpu().numpy(), oracle.gemv(W, x, N, K), x, K, f"chain N={N} K={K} B={B}")
    assert q4k.device_error_flags() == 0
    ch.close()


@pytest.mark.parametrize("B", [1, 3])
def test_dependent_steps(env, B):
    """Each step reads the previous step's output: y1 = W1 x0, y2 = W2 y1, y3 = W3 y2."""
    q4k, oracle = env
    dims = [(512, 3584), (256, 512), (1280, 256), (300, 1280)]   # (N, K); K of step i = N of step i-1
    Ws = [synth.q4k_weights(N, K, (91, i)) for i, (N, K) in enumerate(dims)]
    x0 = synth.normal_f32((B, dims[0][1]), (92, B))
    xd = _dev(x0)
    ys = [torch.empty((B, N), device="cuda") for N, _ in dims]
    steps = []
    for i, (N, K) in enumerate(dims):
        steps.append((xd if i == 0 else ys[i - 1], [(_dev(Ws[i]), ys[i])]))
    ch = q4k.Chain(steps, B)
    ch.run()
    torch.cuda.synchronize()
    prev = x0
    for i, (N, K) in enumerate(dims):
        got = ys[i].cpu().numpy()
        # the step must have used the final values of its input
        assert_close(got, oracle.gemv(Ws[i], prev, N, K), prev, K, f"step {i}")
        prev = got.astype(np.float32)
    ch.close()


def test_rerun_deterministic_and_follows_inputs(env):
    q4k, oracle = env
    B = 2
    host, dev = _layer_steps(B, layer=3)
    ch = q4k.Chain(dev, B)
    ch.run()
    first = [y.clone() for _, g in dev for _, y in g]
    ch.run()
    torch.cuda.synchronize()
    again = [y for _, g in dev for _, y in g]
    for a, b in zip(first, again):
        assert torch.equal(a, b)
    # new x contents in the same buffers: the next run uses them
    x_new = synth.normal_f32(tuple(dev[3][0].shape), (93,))
    dev[3][0].copy_(torch.from_numpy(x_new))
    ch.run()
    torch.cuda.synchronize()
    W, N = host[3][1][0]
    K = x_new.shape[1]
    assert_close(dev[3][1][0][1].cpu().numpy(), oracle.gemv(W, x_new, N, K), x_new, K, "rerun")
    ch.close()


def test_chain_matches_per_step_launches(env):
    """Same steps as separate grouped launches: equal within the tolerance."""
    q4k, oracle = env
    B = 1
    host, dev = _layer_steps(B, layer=1)
    ch = q4k.Chain(dev, B)
    ch.run()
    torch.cuda.synchronize()
    for (x, hg), (xd, dg) in zip(host, dev):
        K = x.shape[1]
        ys = q4k.gemv_grouped([W for W, _ in dg], xd)
        torch.cuda.synchronize()
        for (W, N), (_, y), y2 in zip(hg, dg, ys):
            ref = oracle.gemv(W, x, N, K)
            assert_close(y.cpu().numpy(), ref, x, K, "chain")
            assert_close(y2.cpu().numpy(), ref, x, K, "grouped")
    ch.close()


def test_graph_capture(env):
    q4k, _ = env
    B = 1
    host, dev = _layer_steps(B, layer=2)
    ch = q4k.Chain(dev, B)
    ch.run()
    torch.cuda.synchronize()
    eager = [y.clone() for _, g in dev for _, y in g]
    for _, g in dev:
        for _, y in g:
            y.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ch.run(stream=s)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    s.synchronize()
    for a, (_, gr) in zip(eager, [(None, y) for _, gg in dev for _, y in gg]):
        assert torch.equal(a, gr)
    ch.close()


def test_empty_groups_and_small_steps(env):
    q4k, oracle = env
    B = 4
    K = 1024
    Ws = [synth.q4k_weights(N, K, (94, i)) for i, N in enumerate([7, 130, 300])]
    x = synth.normal_f32((B, K), 95)
    xd = _dev(x)
    ys = [torch.empty((B, W.shape[0]), device="cuda") for W in Ws]
    empty_W = torch.empty((0, K // 256 * 144), dtype=torch.uint8, device="cuda")
    empty_y = torch.empty((B, 0), device="cuda")
    steps = [(xd, [(_dev(Ws[0]), ys[0]), (empty_W, empty_y), (_dev(Ws[1]), ys[1])]),
             (xd, [(empty_W, empty_y)]),
             (xd, [(_dev(Ws[2]), ys[2])])]
    ch = q4k.Chain(steps, B)
    ch.run()
    torch.cuda.synchronize()
    for W, y in zip(Ws, ys):
        assert_close(y.cpu().numpy(), oracle.gemv(W, x, W.shape[0], K), x, K, f"N={W.shape[0]}")
    assert q4k.device_error_flags() == 0
    ch.close()
