// Internal to libgdnspec: the kernel parameter block shared by the decode /
// recurrent-prefill translation unit (gdnspec.cu, which also holds every C
// entry point and its argument checks) and the tensor-core chunked prefill
// (gdnprefill_chunked.cu).  Not installed; the public interface is
// include/gdnspec.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdnspec.h"

namespace gdn_internal {

// Filled on the host from one validated call; passed by value to the kernels.
struct Params {
    CUtensorMap pool_map;            // decode: the state pool as [slots * H_v * K rows][V], box 128 x 16
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* a;
    const __nv_bfloat16* b;
    const __nv_bfloat16* z;
    const float* A_log;
    const __nv_bfloat16* dt_bias;
    const __nv_bfloat16* norm_w;
    void* pool;
    const int32_t* idx;
    const int32_t* num_acc;
    const int32_t* cu;
    const int32_t* sti;
    const int32_t* read_slots;   // prefill: start slot per sequence (-1: zero state)
    const int32_t* write_slots;  // prefill: final-state slot per sequence (-1: none)
    __nv_bfloat16* out;
    int32_t* status;
    int64_t q_stride, k_stride, v_stride, a_stride, b_stride, z_stride, out_stride;
    int64_t num_slots;
    int32_t batch, num_tokens, H_k, H_v, stride, max_T, group;
    int32_t flags;                   // decode: GDN_PRE_* (inputs read before the dependency wait)
    uint32_t wait_limit;             // chunked prefill: polls per tensor-core wait (0: the default)
    float scale, eps;
    // short causal convolution in front of the step (gdn_spec_decode_conv only)
    const __nv_bfloat16* x;          // pre-convolution rows, channels q | k | v
    const __nv_bfloat16* conv_w;     // [conv_dim][width]
    const __nv_bfloat16* conv_b;     // [conv_dim] or null
    __nv_bfloat16* conv_pool;        // [num_conv_slots][state_len][conv_dim]
    const int32_t* conv_in;
    const int32_t* conv_out;
    int64_t x_stride, num_conv_slots;
    int32_t conv_dim, conv_width, conv_state_len;
};

// Process-wide bound on the chunked prefill's tensor-core waits (0: the default).
extern uint32_t g_wait_limit;

// Launch the chunked prefill kernel: one CTA per (sequence, v-head) unit, or a
// 2-CTA cluster per unit when the units are fewer than half the SMs.
cudaError_t launch_prefill_chunked(const Params& p, int64_t units, gdn_dtype state_dtype, cudaStream_t stream);

}  // namespace gdn_internal
