// q4k_prefill.cu -- prefill entry point (the tcgen05 kernel follows in this file).
#include <cstdint>

#include "q4k_internal.h"

namespace q4k {

static q4k_status validate_prefill(const void *W, const void *X, const float *Y, int64_t N, int64_t K, int64_t T)
{
    if (!W || !X || !Y) return Q4K_ERR_INVALID_ARG;
    if (N < 0 || N > 0x7FFFFFFFll || T < 0 || T > 0x7FFFFFFFll) return Q4K_ERR_INVALID_ARG;
    if (K <= 0 || (K % 256) != 0 || K / 256 >= (1ll << 24)) return Q4K_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) & 15u) || (reinterpret_cast<uintptr_t>(X) & 15u)) return Q4K_ERR_MISALIGNED;
    return Q4K_OK;
}

q4k_status prefill_impl(const void *W, const void *X, float *Y, int64_t N, int64_t K, int64_t T, void *stream)
{
    (void)stream;
    q4k_status st = validate_prefill(W, X, Y, N, K, T);
    if (st != Q4K_OK) return st;
    st = check_device(nullptr);
    if (st != Q4K_OK) return st;
    if (N == 0 || T == 0) return Q4K_OK;
    return Q4K_ERR_UNSUPPORTED_DEVICE;  // tensor-core kernel not wired yet
}

}  // namespace q4k
