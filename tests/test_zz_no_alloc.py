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
from parity import assert_close, tol_limits, top2_margin

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
    import oracle
    oracle.build()
    N, K = 152064 // 4, 3584
    W_host = synth.q4k_weights(N, K, (71, 0)).copy()
    cases = [synth.normal_f32((5, K), (71, 1)), synth.normal_f32((3, K), (71, 2))]
    # give the first batch row a clear winner: scaling d and dmin of its
    # oracle argmax row by 4 scales that logit by exactly 4
    j = oracle.argmax(oracle.gemv(W_host, cases[0][:1], N, K)[0])
    hdr = W_host.reshape(N, K // 256, 144)[j, :, 0:4].copy().view(np.float16) * np.float16(4.0)
    W_host.reshape(N, K // 256, 144)[j, :, 0:4] = hdr.view(np.uint8)
    W = torch.from_numpy(W_host).cuda()
    checked = 0
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
        # and both are the scalar argmax (lowest index on ties) of the very
        # logits the kernel compared, scanned by the CPU oracle
        logits = torch.empty((B, N), dtype=torch.float32, device="cuda")
        dbg = torch.full((B,), -3, dtype=torch.int32, device="cuda")
        st = L.q4k_gemv_argmax_debug(P(W.data_ptr()), P(x.data_ptr()), P(dbg.data_ptr()), P(logits.data_ptr()),
                                     N, K, B, stream)
        assert st == 0, q4k.status_string(st)
        torch.cuda.synchronize()
        lg = logits.cpu().numpy()
        got_np = got.cpu().numpy()
        assert np.array_equal(dbg.cpu().numpy(), got_np)
        for b in range(B):
            assert got_np[b] == oracle.argmax(lg[b]), f"call {call} row {b}: not the scan of the kernel's logits"
        # the logits are within the stated tolerance of the oracle's, and the
        # index is the oracle's own argmax wherever its top-2 margin exceeds
        # twice that tolerance
        y_ref = oracle.gemv(W_host, xn, N, K)
        assert_close(lg, y_ref, xn, K, f"noalloc logits, call {call}")
        for b in range(B):
            tol = tol_limits(y_ref[b:b + 1], xn[b:b + 1], K)[0]
            # each of the two leading logits may be off by tol
            if top2_margin(y_ref[b]) > 2 * tol:
                assert got_np[b] == oracle.argmax(y_ref[b]), f"call {call} row {b}: differs from the oracle"
                checked += 1
    assert checked >= 1
    # beyond the static scratch's capacity: a clear error, nothing launched
    st = L.q4k_gemv_argmax_noalloc(P(W.data_ptr()), P(x.data_ptr()), P(got.data_ptr()), N, K, 17, stream)
    assert st == 1
    torch.cuda.synchronize()
    assert q4k.device_error_flags() == 0
