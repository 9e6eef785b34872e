// q4k_api.cu -- the extern "C" entry points declared in include/q4k.h.
#include <cuda_runtime.h>

#include "../../include/q4k.h"
#include "q4k_internal.h"

extern "C" {

const char *q4k_status_string(q4k_status s)
{
    switch (s) {
        case Q4K_OK: return "ok";
        case Q4K_ERR_INVALID_ARG: return "invalid argument (null pointer, size, K % 256 or batch out of range)";
        case Q4K_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case Q4K_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300, sm_103a)";
        case Q4K_ERR_CUDA: return "CUDA error during launch";
        default: return "unknown status";
    }
}

int q4k_abi_version(void) { return Q4K_ABI_VERSION; }

q4k_status q4k_gemv(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream)
{
    return q4k::gemv_impl(W, x, y, N, K, batch, stream, nullptr);
}

q4k_status q6k_gemv(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream)
{
    return q4k::q6k_gemv_impl(W, x, y, N, K, batch, stream);
}

int64_t q6k_planar_bytes(int64_t N, int64_t K) { return q4k::q6k_planar_bytes_impl(N, K); }

q4k_status q6k_repack_planar(const void *W, void *Wp, int64_t N, int64_t K, void *stream)
{
    return q4k::q6k_repack_planar_impl(W, Wp, N, K, stream);
}

q4k_status q6k_gemv_planar(const void *Wp, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream)
{
    return q4k::q6k_gemv_planar_impl(Wp, x, y, N, K, batch, stream);
}

q4k_status q4k_gemv_ex(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream,
                       const q4k_launch_opts *opts)
{
    return q4k::gemv_impl(W, x, y, N, K, batch, stream, opts);
}

q4k_status q4k_gemv_grouped(const q4k_gemv_group *groups, int ngroups, const float *x, int64_t K, int batch,
                            void *stream, const q4k_launch_opts *opts)
{
    return q4k::gemv_grouped_impl(groups, ngroups, x, K, batch, stream, opts);
}

q4k_status q4k_gemv_argmax(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K, int batch,
                           void *stream)
{
    return q4k::gemv_argmax_impl(W, x, idx, nullptr, N, K, batch, stream, nullptr, nullptr, nullptr);
}

q4k_status q4k_gemv_argmax_debug(const void *W, const float *x, int32_t *idx, float *logits, int64_t N, int64_t K,
                                 int batch, void *stream)
{
    if (!logits) return Q4K_ERR_INVALID_ARG;
    return q4k::gemv_argmax_impl(W, x, idx, logits, N, K, batch, stream, nullptr, nullptr, nullptr);
}

q4k_status q4k_gemv_argmax_noalloc(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K, int batch,
                                   void *stream)
{
    return q4k::gemv_argmax_noalloc_impl(W, x, idx, N, K, batch, stream);
}

q4k_status q4k_gemm_prefill(const void *W, const void *X_bf16, float *Y, int64_t N, int64_t K, int64_t T,
                            void *stream)
{
    return q4k::prefill_impl(W, X_bf16, Y, N, K, T, stream, false);
}

q4k_status q4k_gemm_prefill_exact(const void *W, const void *X_bf16, float *Y, int64_t N, int64_t K, int64_t T,
                                  void *stream)
{
    return q4k::prefill_impl(W, X_bf16, Y, N, K, T, stream, true);
}

q4k_status q4k_stream_read(const void *buf, int64_t bytes, int64_t *bytes_read, void *stream)
{
    return q4k::stream_read_impl(buf, bytes, bytes_read, stream);
}

q4k_status q4k_gemv_plan(int64_t N, int64_t K, int batch, int out[4])
{
    return q4k::gemv_plan_impl(N, K, batch, out);
}

/* Sticky device-side error bits (bit 0: a bounded wait inside a kernel timed
 * out and the kernel wound down early).  Synchronous; 0 means no error. */
unsigned int q4k_device_error_flags(void)
{
    return q4k::read_device_error() | q4k::read_prefill_error() | q4k::read_q6k_error() | q4k::read_q6p_error() |
           q4k::read_probe_error();
}

q4k_status q4k_device_error_clear(void)
{
    const bool ok = q4k::clear_device_error() & q4k::clear_prefill_error() & q4k::clear_q6k_error() &
                    q4k::clear_q6p_error() & q4k::clear_probe_error();
    return ok ? Q4K_OK : Q4K_ERR_CUDA;
}

}  // extern "C"
