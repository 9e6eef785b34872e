"""The allocation-free argmax entry point (q4k_gemv_argmax_noalloc).

Some callers cannot allocate device memory while they run (fixed memory
budgets, real-time loops, a replaced or unavailable stream-ordered allocator),
so the library offers an argmax that keeps its scratch in a static device
array.  This test calls it through the C ABI and checks it against the regular
q4k_gemv_argmax on two calls in a row (the second call must not see stale
scratch from the first).  It lives in its own file, collected last."""
import ctypes

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_noalloc_argmax_matches_regular_entry_point():
    import __graft_entry__
    __graft_entry__.build()
    import q4_dequant_gemv_gb300 as q4k
    torch.cuda.set_device(0)
    L = q4k.lib()
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    N, K = 152064 // 4, 3584
    W = torch.from_numpy(synth.q4k_weights(N, K, (71, 0))).cuda()
    cases = [synth.normal_f32((5, K), (71, 1)), synth.normal_f32((3, K), (71, 2))]
    for call, xn in enumerate(cases):
        B = xn.shape[0]
        x = torch.from_numpy(xn).cuda()
        ref = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        got = torch.full((B,), -2, dtype=torch.int32, device="cuda")
        st = L.q4k_gemv_argmax(P(W.data_ptr()), P(x.data_ptr()), P(ref.data_ptr()), N, K, B, stream)
        assert st == 0, q4k.status_string(st)
        st = L.q4k_gemv_argmax_noalloc(P(W.data_ptr()), P(x.data_ptr()), P(got.data_ptr()), N, K, B, stream)
        assert st == 0, q4k.status_string(st)
        torch.cuda.synchronize()
        # argmax indices are integers: the two entry points must agree exactly
        assert np.array_equal(ref.cpu().numpy(), got.cpu().numpy()), f"call {call}"
    # beyond the static scratch's capacity: a clear error, nothing launched
    st = L.q4k_gemv_argmax_noalloc(P(W.data_ptr()), P(x.data_ptr()), P(got.data_ptr()), N, K, 17, stream)
    assert st == 1
    torch.cuda.synchronize()
    assert q4k.device_error_flags() == 0
