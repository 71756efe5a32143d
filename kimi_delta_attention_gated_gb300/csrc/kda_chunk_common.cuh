// kda_chunk_common.cuh -- pieces shared by the chunked-prefill kernels on the tensor
// cores: the fused one-kernel form (kda_chunk_tc.cu) and the split form, whose
// state-independent pre-pass (kda_chunk_prep.cu) feeds the per-head chain kernel
// (kda_chunk_chain.cu) through a caller-provided workspace.
//
// Chunk algebra (derived from the recurrence, exact in real arithmetic).  For one
// (sequence, head) and a chunk of C = 64 tokens entering with state S [K x V]:
//   G_i = sum_{s<=i} g_s (inclusive, per key channel), gamma = G_{C-1}
//   Kd = k^ exp(G), Qd = q^ exp(G), Km = k^ exp(-G), Kg = k^ exp(gamma - G)
//   A = strict_lower(diag(beta) Kd Km^T),  P = lower(Qd Km^T)          (grams)
//   T = (I + A)^-1                                                    (UT transform)
//   R = V - Kd S,  D = T diag(beta) R
//   O = Qd S + P D,  S' = Diag(exp gamma) S + Kg^T D
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "kda_tc_ptx.cuh"

namespace kda {
namespace chunk {

using namespace tc;

constexpr int C = 64;                  // tokens per chunk
constexpr int DK = 128;                // key dim
constexpr int DV = 128;                // value dim
constexpr float kRangeMax = 80.f;      // Km = k^ exp(-G) stays finite while max_c(-gamma) <= this
constexpr uint32_t kPolls = 1u << 26;  // bound on every mbarrier wait
constexpr int AP = 68;                 // fp32 pitch of the A and T matrices in shared memory

// One chunk's state-independent operands, as the split form hands them from the pre-pass
// to the chain kernel: four 64 x 64 bf16 tiles in the 128-byte-swizzled K-major layout
// the tensor core reads (byte images of the shared-memory tiles), 8 KB each:
//   [0, 8K) T diag(beta) hi, [8K, 16K) its lo part, [16K, 24K) P hi, [24K, 32K) P lo.
constexpr uint32_t kBlobBytes = 32768;

// Blob slot of chunk c of sequence n (first token bos): floor(bos / C) + n + c.  Slots of
// different (sequence, chunk) pairs never coincide and stay below ceil(rows / C) + N, the
// slot count of a workspace.  The blob of (slot, head h) is at (slot * H + h) * kBlobBytes.
__host__ __device__ __forceinline__ int64_t blob_slot(int64_t bos, int n, int c) { return bos / C + n + c; }

__host__ __device__ __forceinline__ int64_t blob_slots(int64_t rows, int N) { return (rows + C - 1) / C + N; }

// Workspace layout: the blobs, then (256-byte aligned) one ready flag per blob and one
// progress word per (sequence, head).  The split form uses the blobs only; the concurrent
// form also the flags (set by the pre-pass once a blob is complete) and the progress
// words (how many chunks each fused CTA has begun), both zeroed before each call.
struct WorkspaceLayout {
    size_t flags, progress, bytes;
    __host__ __device__ WorkspaceLayout(int64_t rows, int N, int H) {
        const size_t blobs = (size_t)blob_slots(rows, N) * H;
        flags = blobs * kBlobBytes;
        progress = flags + ((blobs * 4 + 255) & ~(size_t)255);
        bytes = progress + (((size_t)N * H * 4 + 255) & ~(size_t)255);
    }
};

// Global-memory accesses of the concurrent form's flags and progress words (GPU scope).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's global accesses across the generic and the asynchronous proxy
// (bulk copies): a blob written by bulk stores before its flag, read by bulk loads after.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Writes 8 consecutive columns (col % 8 == 0) of one row as hi/lo.
__device__ __forceinline__ void st_tile8(uint32_t hi_base, uint32_t lo_base, uint32_t rows, uint32_t row,
                                         uint32_t col, const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split2(x[2 * e], x[2 * e + 1], h[e], l[e]);
    const uint32_t off = sw128_off(row, col, rows);
    st_shared_v4(hi_base + off, h[0], h[1], h[2], h[3]);
    st_shared_v4(lo_base + off, l[0], l[1], l[2], l[3]);
}

// Kg^T rows c..c+3 (one per key channel) at columns j0..j0+3 (4 tokens) of the
// [P ; Kg^T] tiles, hi and lo: x[t][e] is token j0 + t, channel c + e, c = 4 * lane.
// Store e of a lane writes channel c + ((e + rot) & 3) with rot = (lane >> 1) & 3, so the
// 32 rows of one store cover all 8 swizzle phases (4 wavefronts instead of 16).
__device__ __forceinline__ void st_kgt(uint32_t hi_base, uint32_t lo_base, int c, int j0, const float (&x)[4][4]) {
    const int rot = (c >> 3) & 3;
    float y[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float a[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = (rot & 1) ? x[t][(e + 1) & 3] : x[t][e];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[t][e] = (rot & 2) ? a[(e + 2) & 3] : a[e];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        uint32_t h0, l0, h1, l1;
        split2(y[0][e], y[1][e], h0, l0);
        split2(y[2][e], y[3][e], h1, l1);
        const uint32_t off = sw128_off(64 + c + ((e + rot) & 3), j0, 192);
        st_shared_v2(hi_base + off, h0, h1);
        st_shared_v2(lo_base + off, l0, l1);
    }
}

// SWIZZLE_128B shared-memory descriptor (the same fields as sdesc) of the operand at byte
// offset off from the 1024-aligned shared base whose address / 16 is sb16: the address
// field is sb16 + off / 16 (below 2^14, shared addresses being below 2^18 bytes), so with
// compile-time off, lbo and sbo the whole descriptor is one add and a constant high word.
__device__ __forceinline__ uint64_t sdesc_at(uint32_t sb16, uint32_t off, uint32_t lbo, uint32_t sbo) {
    const uint32_t lo = (sb16 + (off >> 4)) | ((lbo >> 4) << 16);
    const uint32_t hi = ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
    return ((uint64_t)hi << 32) | lo;
}

// hi*hi, hi*lo, lo*hi: (A part, B part) of the three products of a split operand pair
__device__ __forceinline__ int combo_a(int cb) { return cb == 2 ? 1 : 0; }
__device__ __forceinline__ int combo_b(int cb) { return cb == 1 ? 1 : 0; }

}  // namespace chunk
}  // namespace kda
