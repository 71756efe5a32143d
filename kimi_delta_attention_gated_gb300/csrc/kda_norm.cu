// kda_norm.cu -- head-wise sigmoid-gated RMSNorm.
//
// Page: Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters"
// (the gated RMSNorm holds head_dim = 128 weights, one vector shared by all 96
// heads) and "Code" (o_norm(o, gate) with activation 'sigmoid', then the heads
// are flattened).  y = o / sqrt(mean_v(o^2) + eps) * w * sigmoid(gate).
//
// HBM-bound elementwise pass: one warp per (token, head) row of V values, each
// lane holding V/32 consecutive values so every access is one coalesced
// transaction per warp; a grid-stride loop over rows sized to the SM count.
// o and y may be the same buffer (each element is read before it is written by
// the same lane).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int V>
__global__ void __launch_bounds__(kThreads) gated_rmsnorm_kernel(const void *o, int o_bf16,
                                                                 const void *gate, int gate_bf16,
                                                                 const float *w, float eps, void *y,
                                                                 int y_bf16, int64_t nrows) {
    constexpr int VPL = V / 32;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    float wv[VPL];
#pragma unroll
    for (int c = 0; c < VPL; ++c) wv[c] = w[lane * VPL + c];
    for (int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < nrows; r += warps) {
        const size_t base = (size_t)r * V + lane * VPL;
        float x[VPL], gt[VPL];
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
            x[c] = ld_in(o, base + c, o_bf16);
            gt[c] = ld_in(gate, base + c, gate_bf16);
            ss = fmaf(x[c], x[c], ss);
        }
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)V + eps);
#pragma unroll
        for (int c = 0; c < VPL; ++c) st_out(y, base + c, x[c] * inv * wv[c] * sigmoidf_(gt[c]), y_bf16);
    }
}

}  // namespace

int sm_count() {
    static int counts[64] = {0};  // per device; a race only repeats the query
    const int dev = current_device();
    if (dev >= 0 && dev < 64 && counts[dev] > 0) return counts[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 1;
    }
    if (dev >= 0 && dev < 64) counts[dev] = n;
    return n;
}

kda_status launch_gated_rmsnorm(const void *o, int o_bf16, const void *gate, int gate_bf16,
                                const float *w, float eps, void *y, int y_bf16, int64_t rows,
                                int H, int V, cudaStream_t st) {
    const int64_t nrows = rows * (int64_t)H;
    if (nrows == 0) return KDA_OK;
    const int64_t need = (nrows + (kThreads / 32) - 1) / (kThreads / 32);
    const int64_t cap = (int64_t)sm_count() * 8;
    const int grid = (int)(need < cap ? need : cap);
#define KDA_CASE(VV)                                                                          \
    if (V == VV) {                                                                            \
        gated_rmsnorm_kernel<VV><<<grid, kThreads, 0, st>>>(o, o_bf16, gate, gate_bf16, w, eps, \
                                                            y, y_bf16, nrows);                \
        note_launch();                                                                        \
        return check_launch("gated_rmsnorm_kernel");                                          \
    }
    KDA_CASE(128)
    KDA_CASE(64)
    KDA_CASE(32)
#undef KDA_CASE
    set_error("gated_rmsnorm: V=%d not built (V in {32, 64, 128})", V);
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
