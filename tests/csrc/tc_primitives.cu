// tc_primitives.cu -- GPU unit test of the tensor-core building blocks in
// kda_tc_ptx.cuh: one CTA computes D = A * B^T (M = 128) with tcgen05.mma from
// the operand layouts the KDA prefill kernel uses, and writes D to global memory
// for comparison with a host matmul.
//
// Cases:
//   0  A K-major smem (K = 128, two column blocks), B K-major smem (N = 64)
//   1  A MN-major smem (K = 64), B K-major smem (N = 64)
//   2  A K-major smem (K = 64), B MN-major smem (N = 128)
//   3  A in TMEM (packed bf16 pairs, K = 64), B K-major smem (N = 64)
//   4  case 0 with the second half of K accumulated with B negated
//   5  A in TMEM (K = 64), B MN-major smem (N = 128)
//   6  failure detection: a bounded wait on an mbarrier that nothing arrives on must
//      give up, report it (err = 2) and leave the kernel and the context usable
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_tc_ptx.cuh"

using namespace kda::tc;

namespace {

constexpr uint32_t kPolls = 1u << 24;

__global__ void __launch_bounds__(128) probe_kernel(int which, const __nv_bfloat16 *A, const __nv_bfloat16 *B,
                                                    float *D, int *err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned operand tiles
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sa = base;               // 32 KB
    uint8_t *sb = base + 32768;       // 32 KB
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int tid = threadIdx.x, warp = tid >> 5;

    const bool a_mn = which == 1;
    const bool b_mn = which == 2 || which == 5;
    const bool a_tmem = which == 3 || which == 5;
    const int K = (which == 0 || which == 4) ? 128 : 64;
    const int N = (which == 2 || which == 5) ? 128 : 64;

    // stage A (logical A[m][k], 128 x K) and B (logical B[n][k], N x K)
    for (int e = tid; e < 128 * K; e += 128) {
        const int m = e / K, k = e % K;
        const __nv_bfloat16 x = A[m * 128 + k];
        const uint32_t off = a_mn ? sw128_off(k, m, K) : sw128_off(m, k, 128);
        *reinterpret_cast<__nv_bfloat16 *>(sa + off) = x;
    }
    for (int e = tid; e < N * K; e += 128) {
        const int n = e / K, k = e % K;
        const __nv_bfloat16 x = B[n * 128 + k];
        const uint32_t off = b_mn ? sw128_off(k, n, K) : sw128_off(n, k, N);
        *reinterpret_cast<__nv_bfloat16 *>(sb + off) = x;
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tbase, 256);
        tmem_relinquish();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t t0 = tbase;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    if (a_tmem) {  // thread m packs its row into TMEM columns [128, 128 + K/2)
        const int m = tid;
        uint32_t r[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int k = half * 32 + 2 * c;
                r[c] = pack_bf16(__bfloat162float(A[m * 128 + k]), __bfloat162float(A[m * 128 + k + 1]));
            }
            tmem_st16(t0 + lane_base + 128 + half * 16, r);
        }
        tmem_wait_st();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (which == 6) {  // no MMA is issued and nothing arrives: the wait must run out
        if (tid == 0 && !mbar_wait(&bar, 0, 4096)) atomicExch(err, 2);
        fence_before_sync();
        __syncthreads();
        if (warp == 0) tmem_dealloc(t0, 256);
        return;
    }
    if (tid == 0) {
        const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
        for (int s = 0; s < K / 16; ++s) {
            const bool neg = which == 4 && s >= 4;
            const uint32_t idesc = idesc_bf16(128, N, a_mn, b_mn, false, neg);
            uint64_t bd;
            if (b_mn)
                bd = sdesc(b0 + s * 2048, 64 * 128, 1024);
            else
                bd = sdesc(b0 + (s / 4) * N * 128 + (s % 4) * 32, 16, 1024);
            if (a_tmem) {
                mma_ts(t0, t0 + 128 + s * 8, bd, idesc, s > 0);
            } else {
                uint64_t ad;
                if (a_mn)
                    ad = sdesc(a0 + s * 2048, 64 * 128, 1024);
                else
                    ad = sdesc(a0 + (s / 4) * 128 * 128 + (s % 4) * 32, 16, 1024);
                mma_ss(t0, ad, bd, idesc, s > 0);
            }
        }
        mma_commit(&bar);
    }
    __syncwarp();
    bool ok = mbar_wait(&bar, 0, kPolls);
    fence_after_sync();
    if (!ok) {
        if (tid == 0) atomicExch(err, 1);
    } else {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(t0 + lane_base + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) D[tid * N + c0 + c] = __uint_as_float(r[c]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(t0, 256);
}

}  // namespace

extern "C" int tc_probe(int which, const void *A, const void *B, float *D, int *err, void *stream) {
    const int smem = 65536 + 1024;
    cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(which, (const __nv_bfloat16 *)A,
                                                         (const __nv_bfloat16 *)B, D, err);
    return (int)cudaGetLastError();
}
