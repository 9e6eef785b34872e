// q4k_internal.h -- declarations shared by the translation units of the library.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>

#include "../../include/q4k.h"

namespace q4k {

q4k_status check_device(int *sms_out);
q4k_status gemv_impl(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream,
                     const q4k_launch_opts *opts);
// scratch_keys == nullptr: take 8*16 + 16 bytes from the stream-ordered allocator.
q4k_status gemv_argmax_impl(const void *W, const float *x, int32_t *idx, float *logits, int64_t N, int64_t K,
                            int batch, void *stream, unsigned long long *scratch_keys, unsigned int *scratch_ticket,
                            const q4k_launch_opts *opts);
q4k_status gemv_plan_impl(int64_t N, int64_t K, int batch, int out[4]);
q4k_status gemv_grouped_impl(const q4k_gemv_group *groups, int ngroups, const float *x, int64_t K, int batch,
                             void *stream, const q4k_launch_opts *opts);
q4k_status gemv_argmax_noalloc_impl(const void *W, const float *x, int32_t *idx, int64_t N, int64_t K, int batch,
                                    void *stream);
q4k_status q6k_gemv_impl(const void *W, const float *x, float *y, int64_t N, int64_t K, int batch, void *stream);
int64_t q6k_planar_bytes_impl(int64_t N, int64_t K);
q4k_status q6k_repack_planar_impl(const void *W, void *Wp, int64_t N, int64_t K, void *stream);
q4k_status q6k_gemv_planar_impl(const void *Wp, const float *x, float *y, int64_t N, int64_t K, int batch,
                                void *stream);
q4k_status prefill_impl(const void *W, const void *X, float *Y, int64_t N, int64_t K, int64_t T, void *stream,
                        bool exact);
unsigned int read_device_error();
unsigned int read_prefill_error();
unsigned int read_q6k_error();
unsigned int read_q6p_error();
unsigned int read_probe_error();
q4k_status stream_read_impl(const void *buf, int64_t bytes, int64_t *bytes_read, void *stream);
// Reset the sticky device-side error flag of each translation unit (false on a CUDA error).
bool clear_device_error();
bool clear_prefill_error();
bool clear_q6k_error();
bool clear_q6p_error();
bool clear_probe_error();
// cuTensorMapEncodeTiled from the CUDA driver API (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace q4k
