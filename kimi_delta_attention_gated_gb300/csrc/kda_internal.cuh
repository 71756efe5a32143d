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

// Bound (in polls) on the first-line waits on copies from global memory (decode step,
// short convolution, the fused chunked prefill): kDefaultWaitPolls unless
// kda_set_wait_limit changed it.  The waits that drain copies still in flight before a
// CTA exits, and the waits on the tensor core, always keep the default.
constexpr uint32_t kDefaultWaitPolls = 1u << 26;
uint32_t wait_polls();

// The current device, or 0 if it cannot be read.
int current_device();

// A one-time setup done once per device (devices 0-63; above that it runs every time):
// kernel attributes such as the dynamic shared-memory limit belong to one device.
struct DeviceOnce {
    unsigned long long bits = 0;  // guarded by the caller's idempotent setup: a race repeats it
    bool done(int dev) const { return dev >= 0 && dev < 64 && ((bits >> dev) & 1ull); }
    void set(int dev) {
        if (dev >= 0 && dev < 64) __atomic_fetch_or(&bits, 1ull << dev, __ATOMIC_RELAXED);
    }
};

// Device-side timeout counters of each translation unit, read and cleared on `st`
// (after it has drained) for the current device; each returns the count it took, or -1
// with the error message set when CUDA fails.
int take_chunk_tc_timeouts(cudaStream_t st);
int take_chunk_prep_timeouts(cudaStream_t st);
int take_chunk_chain_timeouts(cudaStream_t st);
int take_oproj_timeouts(cudaStream_t st);
int take_decode_timeouts(cudaStream_t st);
int take_short_conv_timeouts(cudaStream_t st);
// Chunks of the concurrent form that took the pre-pass's operands, read and cleared on
// `st` after it has drained; -1 with the error message set when CUDA fails.
long long take_chunk_blob_chunks(cudaStream_t st);

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
    int K;                       // key dim (indexes dt_bias)
    float scale, eps;
    int l2norm;                  // 0 / 1
    int qkv_bf16, o_bf16, gate_bf16;  // storage dtypes (1 = bf16, 0 = fp32)
    // Gates from their logits (then g / beta are not read):
    //   g = max(g_lower, -exp(A_log[h]) * softplus(g_logits + dt_bias[h][c])), beta = sigmoid(beta_logits)
    const void *g_logits;        // [rows, H, K] or null
    const float *A_log;          // [H]
    const float *dt_bias;        // [H, K] or null
    const void *beta_logits;     // [rows, H] or null
    float g_lower;               // -inf: no floor
    int g_logits_bf16, beta_logits_bf16;
    uint32_t polls;              // bound on the streaming kernels' first-line waits (wait_polls())
    // Short convolutions fused ahead of the decode step (decode kernel only; then q, k, v
    // above are the raw projections).  Filter f (0 = q, 1 = k, 2 = v): weights cw[f]
    // [H * 128, conv_w], history cs_in[f] [N, conv_w - 1, H * 128] (oldest first; all
    // three null: zero history), new history cs_out[f] of the same shape.  conv_w = 0: off.
    const float *cw[3];
    const float *cs_in[3];
    float *cs_out[3];
    int conv_w;
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

// sigmoid with the fast exponential and the fast reciprocal (a few ulp)
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// log(1 + t) for t in [0, 1] with full relative accuracy at small t (the decay logits sit
// near -4, where log(1 + t) formed from a rounded 1 + t and the fast logarithm loses up to
// 1e-3 of it): with s = t / (2 + t) in [0, 1/3], log(1 + t) = log((1 + s) / (1 - s)) =
// 2 (s + s^3/3 + s^5/5 + ...), the series of the inverse hyperbolic tangent, summed here
// through s^13 (the rest is below 1.5e-7 of the sum).  One fast divide and eight FMAs.
__device__ __forceinline__ float log1p_unit(float t) {
    const float s = __fdividef(t, 2.f + t), s2 = s * s;
    float p = 1.f / 13.f;
    p = fmaf(p, s2, 1.f / 11.f);
    p = fmaf(p, s2, 1.f / 9.f);
    p = fmaf(p, s2, 1.f / 7.f);
    p = fmaf(p, s2, 1.f / 5.f);
    p = fmaf(p, s2, 1.f / 3.f);
    p = fmaf(p, s2, 1.f);
    return 2.f * s * p;
}

// softplus(x) = log(1 + e^x) as max(x, 0) + log1p(e^-|x|): as accurate as the fast
// exponential, a few fp32 ulps relative.
__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1p_unit(__expf(-fabsf(x))); }

// g of one key channel from its logit z (bias not yet added); a_h = exp(A_log[h]).
__device__ __forceinline__ float gate_of_logit(float x, float a_h, float lower) { return fmaxf(lower, -a_h * softplus_f(x)); }

__device__ __forceinline__ float beta_of_logit(float b) { return __fdividef(1.f, 1.f + __expf(-b)); }

// g[idx] of head h, key channel c: given directly or from its logit.
__device__ __forceinline__ float load_g(const SeqParams &p, size_t idx, int h, int c) {
    if (!p.g_logits) return p.g[idx];
    const float x = ld_in(p.g_logits, idx, p.g_logits_bf16) + (p.dt_bias ? __ldg(p.dt_bias + (size_t)h * p.K + c) : 0.f);
    return gate_of_logit(x, __expf(__ldg(p.A_log + h)), p.g_lower);
}

// beta[idx]: given directly or the sigmoid of its logit.
__device__ __forceinline__ float load_beta(const SeqParams &p, size_t idx) {
    if (!p.beta_logits) return p.beta[idx];
    return beta_of_logit(ld_in(p.beta_logits, idx, p.beta_logits_bf16));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// kda_chunk_fwd's validation and dispatch, with the name `fn` in its error messages.
kda_status chunk_fwd_entry(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                           const float *g, const float *beta, const float *initial_state, float *final_state, void *o,
                           kda_dtype o_dtype, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                           int B, int T, int H, int K, int V, int chunk, float scale, int use_qk_l2norm,
                           const void *gate, kda_dtype gate_dtype, const float *norm_w, float eps, void *y,
                           void *workspace, size_t workspace_bytes, int mode, void *stream);

// The decay / write-strength logits of the *_logits entry points.
struct GateLogits {
    const void *z;
    int z_dtype;
    const float *A_log, *dt_bias;
    float lower;
    const void *b;
    int b_dtype;
};

// kda_chunk_fwd (gl null) or kda_chunk_fwd_logits (gl given) on device pointers, with
// every check of those entry points and `fn` in the error messages.
kda_status chunk_call(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                      const float *g, const float *beta, const GateLogits *gl, const float *initial_state,
                      float *final_state, void *o, kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk,
                      float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w,
                      float eps, void *y, int mode, void *stream);

// ---------------------------------------------------------------------------
// launchers (one per translation unit); each returns KDA_OK or an error status

kda_status launch_recurrent(const SeqParams &p, int K, int V, cudaStream_t st);
kda_status launch_chunk_fp32(const SeqParams &p, int K, int V, int chunk, const int *order,
                             cudaStream_t st);
// ws: a workspace of chunk_workspace_bytes with zeroed flags and progress words, whose
// blobs the pre-pass fills while this kernel runs (the concurrent form), or null.
kda_status launch_chunk_tc(const SeqParams &p, int K, int V, int chunk, cudaStream_t st, const void *ws = nullptr);
// The concurrent form: the fused kernel on `st` at the highest launch priority, the
// pre-pass beside it on a stream of the call, on the SMs the fused kernel leaves idle.
kda_status launch_chunk_concurrent(const SeqParams &p, void *ws, cudaStream_t st);
// The split tensor-core prefill: the state-independent pre-pass writes every chunk's
// operand images into ws (chunk_workspace_bytes long), then the chain kernel runs the
// state through the chunks.  Both need K = V = 128, chunk = 64, bf16 q/k/v.
size_t chunk_workspace_bytes(int64_t rows, int N, int H);
// The pre-pass alongside the fused kernel (the concurrent form): `grid` CTAs, flags set as
// blobs complete, items skipped within `lead` chunks of their fused CTA's progress.
struct PrepConcurrent {
    int grid;
    int lead;
};
kda_status launch_chunk_prep(const SeqParams &p, void *ws, cudaStream_t st, const PrepConcurrent *cc = nullptr);
// The pre-pass kernels' one-time setup on the current device (this also loads them: done
// before the fused kernel starts, so that loading cannot hold the pre-pass back until the
// fused kernel has finished).
kda_status configure_chunk_prep();
kda_status launch_chunk_chain(const SeqParams &p, const void *ws, cudaStream_t st);
kda_status launch_gated_rmsnorm(const void *o, int o_bf16, const void *gate, int gate_bf16,
                                const float *w, float eps, void *y, int y_bf16, int64_t rows,
                                int H, int V, cudaStream_t st);
kda_status launch_short_conv(const void *x, int x_bf16, const float *w, const float *bias, const float *s0,
                             float *sT, void *y, int y_bf16, const int32_t *cu, int N, int64_t rows, int T,
                             int D, int W, int act, cudaStream_t st);
kda_status launch_o_proj(const void *y, const void *w, void *out, int out_bf16, int64_t M, int K, int N,
                         cudaStream_t st);
bool o_proj_supported(int K, int N);
bool chunk_tc_supported(int K, int V, int chunk);
// cuTensorMapEncodeTiled from the driver (no link against libcuda), or null.
void *tensor_map_encoder();
// Streaming multiprocessors of the current device.
int sm_count();

}  // namespace kda
