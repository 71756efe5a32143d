// kda_internal.cuh -- definitions shared by libkda's translation units.
//
// Parameter blocks passed by value to the kernels, small device helpers for the
// two storage dtypes, and the host-side error / launch bookkeeping.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// ---------------------------------------------------------------------------
// host bookkeeping (kda_abi.cu)

void set_error(const char *fmt, ...);
void note_launch(int n = 1);
// Turns a pending CUDA error into KDA_ERR_CUDA with a message naming `what`.
kda_status check_launch(const char *what);

// ---------------------------------------------------------------------------
// parameter blocks

// One (sequence, head) problem set, shared by the recurrent and chunked paths.
struct SeqParams {
    const void *q, *k, *v;       // [rows, H, K], [rows, H, K], [rows, H, V]
    const float *g, *beta;       // [rows, H, K], [rows, H]
    const float *s0;             // [N, H, K, V] or null
    float *sT;                   // [N, H, K, V] or null
    void *o;                     // [rows, H, V] or null
    float *states;               // [rows, H, K, V] or null (recurrent path only)
    const int32_t *cu_seqlens;   // [N + 1] device or null (dense: sequence n = rows [n T, n T + T))
    const int32_t *cu_host;      // host copy of cu_seqlens or null (host-side scheduling only)
    const void *gate;            // [rows, H, V] or null
    const float *norm_w;         // [V]
    void *y;                     // [rows, H * V]
    int N, T, H;                 // sequences, tokens per sequence (dense) / packed tokens (varlen), heads
    float scale, eps;
    int l2norm;                  // 0 / 1
    int qkv_bf16, o_bf16, gate_bf16;  // storage dtypes (1 = bf16, 0 = fp32)
};

// Token range of sequence n, clamped to [0, T] so a bad cu_seqlens cannot
// send a kernel out of bounds.
__device__ __forceinline__ void seq_range(const SeqParams &p, int n, int &bos, int &len) {
    if (p.cu_seqlens) {
        int a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
        a = a < 0 ? 0 : (a > p.T ? p.T : a);
        b = b < a ? a : (b > p.T ? p.T : b);
        bos = a;
        len = b - a;
    } else {
        bos = n * p.T;
        len = p.T;
    }
}

__device__ __forceinline__ float ld_in(const void *base, size_t idx, int is_bf16) {
    if (is_bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
    return reinterpret_cast<const float *>(base)[idx];
}

__device__ __forceinline__ void st_out(void *base, size_t idx, float x, int is_bf16) {
    if (is_bf16)
        reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
    else
        reinterpret_cast<float *>(base)[idx] = x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---------------------------------------------------------------------------
// launchers (one per translation unit); each returns KDA_OK or an error status

kda_status launch_recurrent(const SeqParams &p, int K, int V, cudaStream_t st);
kda_status launch_chunk_fp32(const SeqParams &p, int K, int V, int chunk, const int *order,
                             cudaStream_t st);
kda_status launch_chunk_tc(const SeqParams &p, int K, int V, int chunk, cudaStream_t st);
kda_status launch_gated_rmsnorm(const void *o, int o_bf16, const void *gate, int gate_bf16,
                                const float *w, float eps, void *y, int y_bf16, int64_t rows,
                                int H, int V, cudaStream_t st);
kda_status launch_short_conv(const void *x, int x_bf16, const float *w, const float *bias, const float *s0,
                             float *sT, void *y, int y_bf16, const int32_t *cu, int N, int64_t rows, int T,
                             int D, int W, int act, cudaStream_t st);
bool chunk_tc_supported(int K, int V, int chunk);
// cuTensorMapEncodeTiled from the driver (no link against libcuda), or null.
void *tensor_map_encoder();
// Streaming multiprocessors of the current device.
int sm_count();

}  // namespace kda
