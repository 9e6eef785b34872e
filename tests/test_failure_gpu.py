"""Failure path of the bounded device waits, made to run out on purpose without
any fault: a GEMV launched with the test-only stall flag, whose first weight
copy in every CTA is awaited for 16 bytes more than it brings, with a 1 ms
bound.  The kernel must return by itself, set the sticky error bit and leave
the context usable; after q4k_device_error_clear() the next launch is correct."""
import time

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


@pytest.mark.parametrize("N,K,B,split", [(700, 1024, 1, 0), (3584, 3584, 1, 0), (300, 2048, 5, 0), (150, 2304, 1, 3),
                                         (3584, 18944, 1, 0)])
def test_wait_runs_out_then_recovers(env, N, K, B, split):
    q4k, oracle = env
    torch.cuda.synchronize()
    q4k.device_error_clear()
    assert q4k.device_error_flags() == 0
    W = synth.q4k_weights(N, K, (97, N, K))
    x = synth.normal_f32((B, K), (98, N, B))
    Wd = torch.from_numpy(W).cuda()
    xd = torch.from_numpy(x).cuda()
    y = torch.full((B, N), 7.0, device="cuda")
    t0 = time.time()
    q4k.gemv(Wd, xd, y, split_k=split, wait_limit_us=1000, test_stall=True)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert q4k.device_error_flags() & 1, "the stalled wait did not flag an error"
    # an aborted kernel writes no outputs
    assert torch.all(y == 7.0)
    # the context is still usable and the flag clears on request
    q4k.device_error_clear()
    assert q4k.device_error_flags() == 0
    q4k.gemv(Wd, xd, y, split_k=split)
    torch.cuda.synchronize()
    assert q4k.device_error_flags() == 0
    assert_close(y.cpu().numpy(), oracle.gemv(W, x, N, K), x, K, f"after recovery N={N} K={K} B={B}")


def test_error_clear_without_errors(env):
    q4k, _ = env
    q4k.device_error_clear()
    assert q4k.device_error_flags() == 0
