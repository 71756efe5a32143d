// kda_oproj.cu -- the layer's output projection of the gated-norm output, on the tensor cores.
//
// Page: Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters"
// (output projection 88,080,384 weights = 12288 inputs x 7168 outputs) and "Code"
// (o = o_proj(o) after o_norm and the heads flattened to heads * head_dim).
//
//   out[r][n] = sum_c y[r][c] * w_o[n][c]      (nn.Linear, no bias)
//
// A dense GEMM with bf16 operands and fp32 accumulation, written for tcgen05.  Each tile
// is 128 output features (the MMA M dimension: the rows of w_o, so the accumulator's
// TMEM lane is the feature) by BN rows of y (the MMA N dimension: tokens); both operands
// are K-major, as nn.Linear stores them, and arrive by TMA in 64-wide K slices with the
// 128-byte swizzle.  Warp-specialised persistent CTAs, one per SM:
//   warp 0    TMA producer: a ring of stages, each the w_o slice and the y slice
//   warp 1    MMA issuer: four 128 x BN x 16 products per stage into one of two TMEM
//             accumulators, a commit per stage releases it to the producer
//   warps 2-5 epilogue: TMEM -> registers -> out, then the accumulator goes back to
//             the MMA warp, so a tile's epilogue overlaps the next tile's products
// Tiles are visited in groups of 8 feature tiles across every token tile, so the CTAs
// running at one time share their w_o and y slices through L2.  BN = 256 when there are
// enough tiles to fill the GPU (prompts), else 128 (the decode batch: 256 rows give 112
// tiles over 7168 features, each streaming its 3 MB slice of w_o once).
#include <cuda.h>
#include <string.h>

#include "kda_chunk_common.cuh"
#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;
using chunk::sdesc_at;

constexpr int BM = 128;                // output features per tile
constexpr int BK = 64;                 // K per stage: one 128-byte swizzle row of bf16
constexpr int kWarps = 6;              // 0: TMA, 1: MMA, 2-5: epilogue
constexpr int kFeatureGroup = 8;       // feature tiles per raster group
constexpr uint32_t kPolls = 1u << 26;  // bound on every mbarrier wait

// Set by a CTA whose bounded wait gave up; its remaining output tiles hold NaN.
__device__ int g_oproj_timeouts = 0;

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr uint32_t A_BYTES = BM * BK * 2;  // w_o slice, 16 KB
    static constexpr uint32_t B_BYTES = BN * BK * 2;  // y slice
    static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t BARS = STAGES * STAGE;  // full[S], empty[S], acc_full[2], acc_empty[2], drain
    static constexpr uint32_t SMEM = BARS + (2 * STAGES + 5) * 8 + 16 + 1024;  // + tmem slot, abort flag
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};
static_assert(Cfg<256>::SMEM <= 232448 && Cfg<128>::SMEM <= 232448, "shared memory budget");

struct GemmArgs {
    void *out;
    int out_bf16;
    int M, N, K;
    int n_ft, n_tt, n_tiles;  // feature tiles, token tiles, all tiles
};

// Feature and token tile of tile id: groups of kFeatureGroup feature tiles, the feature
// index fastest inside a group, then every token tile, then the next group.
__device__ __forceinline__ void tile_coords(int id, int n_ft, int n_tt, int &f, int &t) {
    const int per_group = kFeatureGroup * n_tt;
    const int g = id / per_group, r = id % per_group;
    const int f0 = g * kFeatureGroup, gsz = min(kFeatureGroup, n_ft - f0);
    f = f0 + r % gsz;
    t = r / gsz;
}

template <int BN>
__global__ void __launch_bounds__(kWarps * 32, 1)
    oproj_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_y,
                 const __grid_constant__ GemmArgs a) {
    using L = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm), sb16 = sb >> 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint64_t *empty = full + L::STAGES;
    uint64_t *acc_full = empty + L::STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);  // a warp's bounded wait gave up
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = a.K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::TMEM_COLS);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    int failed = 0;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer
            uint32_t it = 0;
            for (int id = blockIdx.x; id < a.n_tiles && !failed; id += gridDim.x) {
                int f, t;
                tile_coords(id, a.n_ft, a.n_tt, f, t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % L::STAGES, use = it / L::STAGES;
                    // the stage's previous use must have been read by its MMAs
                    if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1, kPolls)) {
                        failed = 1;
                        *abort_flag = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(full + s, L::STAGE);
                    tma_load_2d(sb + s * L::STAGE, &tmap_w, full + s, kb * BK, f * BM);
                    tma_load_2d(sb + s * L::STAGE + L::A_BYTES, &tmap_y, full + s, kb * BK, t * BN);
                }
            }
            // every load issued lands before the CTA may exit: wait for each stage's last use
            const uint32_t n_issued = it;
            for (uint32_t s = 0; s < (uint32_t)L::STAGES && s < n_issued; ++s) {
                const uint32_t last = n_issued - 1 - ((n_issued - 1 + L::STAGES - s) % L::STAGES);
                mbar_wait(full + s, (last / L::STAGES) & 1, kPolls);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---- MMA issuer
            const uint32_t idesc = idesc_bf16(BM, BN, false, false);
            uint32_t it = 0, tc = 0;
            for (int id = blockIdx.x; id < a.n_tiles && !failed; id += gridDim.x, ++tc) {
                const uint32_t acc = tc & 1, use = tc >> 1;
                if (use > 0 && !mbar_wait(acc_empty + acc, (use - 1) & 1, kPolls)) {  // the epilogue has read it
                    failed = 1;
                    *abort_flag = 1;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tb + acc * BN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const uint32_t s = it % L::STAGES;
                    if (!mbar_wait(full + s, (it / L::STAGES) & 1, kPolls)) {
                        failed = 1;
                        *abort_flag = 1;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t sa = s * L::STAGE, sbb = sa + L::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_ss(d, sdesc_at(sb16, sa + k * 32, 16, 1024), sdesc_at(sb16, sbb + k * 32, 16, 1024), idesc,
                               (kb | k) ? 1u : 0u);
                    mma_commit(empty + s);  // the stage is free once these products have read it
                }
                if (failed) break;
                mma_commit(acc_full + acc);
            }
            // nothing issued may still run when the accumulators are freed
            mma_commit(drain);
            mbar_wait(drain, 0, kPolls);
        }
    } else {  // ---- epilogue, warps 2-5: TMEM lane quarter warp % 4
        const int q = warp & 3, m = q * 32 + lane;
        const uint32_t lane_base = tb + ((uint32_t)(q * 32) << 16);
        uint32_t tc = 0;
        for (int id = blockIdx.x; id < a.n_tiles; id += gridDim.x, ++tc) {
            int f, t;
            tile_coords(id, a.n_ft, a.n_tt, f, t);
            const uint32_t acc = tc & 1, use = tc >> 1;
            const bool ok = !failed && !*abort_flag && mbar_wait(acc_full + acc, use & 1, kPolls);
            if (!ok) failed = 1;
            fence_after_sync();
            const int feat = f * BM + m;
            const int t0 = t * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r0[16], r1[16];
                if (ok) {
                    tmem_ld16(lane_base + acc * BN + c0, r0);
                    tmem_ld16(lane_base + acc * BN + c0 + 16, r1);
                    tmem_wait_ld();
                }
                const int nrow = min(32, a.M - (t0 + c0));
                if (a.out_bf16) {
                    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(a.out) + (size_t)(t0 + c0) * a.N + feat;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < nrow)
                            o[(size_t)j * a.N] = __float2bfloat16_rn(
                                ok ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) : __int_as_float(0x7fc00000));
                } else {
                    float *o = reinterpret_cast<float *>(a.out) + (size_t)(t0 + c0) * a.N + feat;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < nrow) o[(size_t)j * a.N] = ok ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) : __int_as_float(0x7fc00000);
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(acc_empty + acc);
        }
    }
    fence_before_sync();
    if (__syncthreads_or(failed) && threadIdx.x == 0) atomicAdd(&g_oproj_timeouts, 1);
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tb, L::TMEM_COLS);
}

// Cluster helpers for the split-K form: this CTA's rank in its cluster, a shared-memory
// address mapped into another CTA of the cluster, a store there, and the cluster barrier
// (every thread of both CTAs passes each one exactly once).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The decode batch (at most 256 rows, few feature tiles): one 128-feature x 256-row tile per
// pair of CTAs in a cluster, each pair member running half of K, so that twice as many SMs
// run the products.  Rank 1 adds its fp32 accumulator into rank 0's shared memory (the
// stage buffers are idle by then) between two cluster barriers; rank 0 sums and writes.
__global__ void __launch_bounds__(kWarps * 32, 1)
    oproj_splitk_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_y,
                        const __grid_constant__ GemmArgs a) {
    constexpr int BN = 256;
    using L = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm), sb16 = sb >> 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint64_t *empty = full + L::STAGES;
    uint64_t *acc_full = empty + L::STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int f = blockIdx.x >> 1;  // feature tile of the pair
    const int KB = a.K / BK, kb0 = (int)rank * (KB / 2), kb1 = kb0 + KB / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    int failed = 0;

    if (warp == 0 && lane == 0) {  // ---- TMA producer
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const uint32_t s = it % L::STAGES, use = it / L::STAGES;
            if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1, kPolls)) {
                failed = 1;
                break;
            }
            mbar_arrive_expect_tx(full + s, L::STAGE);
            tma_load_2d(sb + s * L::STAGE, &tmap_w, full + s, kb * BK, f * BM);
            tma_load_2d(sb + s * L::STAGE + L::A_BYTES, &tmap_y, full + s, kb * BK, 0);
        }
        const uint32_t n_issued = it;
        for (uint32_t s = 0; s < (uint32_t)L::STAGES && s < n_issued; ++s) {
            const uint32_t last = n_issued - 1 - ((n_issued - 1 + L::STAGES - s) % L::STAGES);
            mbar_wait(full + s, (last / L::STAGES) & 1, kPolls);
        }
    } else if (warp == 1 && lane == 0) {  // ---- MMA issuer
        const uint32_t idesc = idesc_bf16(BM, BN, false, false);
        uint32_t it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const uint32_t s = it % L::STAGES;
            if (!mbar_wait(full + s, (it / L::STAGES) & 1, kPolls)) {
                failed = 1;
                break;
            }
            fence_after_sync();
            const uint32_t sa = s * L::STAGE, sbb = sa + L::A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
                mma_ss(tb, sdesc_at(sb16, sa + k * 32, 16, 1024), sdesc_at(sb16, sbb + k * 32, 16, 1024), idesc,
                       (it | k) ? 1u : 0u);
            mma_commit(empty + s);
        }
        mma_commit(acc_full);  // also an arrival after a failure: nothing issued may still run
    }
    __syncwarp();  // the producer and MMA warps reconverge before the cluster barriers
    // every MMA of this CTA has completed once acc_full does
    const int q = warp & 3, m = q * 32 + lane;
    const uint32_t lane_base = tb + ((uint32_t)(q * 32) << 16);
    if (warp >= 2 && !mbar_wait(acc_full, 0, kPolls)) failed = 1;
    fence_after_sync();
    cluster_sync();  // both halves' products done: rank 0's stage buffers are idle
    // rank 1's partial sums in rank 0's shared memory: [128 lanes][kPartPitch] fp32 (130 KB), a
    // lane's 256 columns contiguous, rows padded so that 16-byte accesses of consecutive lanes
    // fall in different banks
    constexpr int kPartPitch = BN + 4;
    static_assert(128 * kPartPitch * 4 <= L::STAGES * L::STAGE, "the partial sums fit in the stage buffers");
    const float *part = reinterpret_cast<const float *>(sm) + m * kPartPitch;
    if (warp >= 2 && rank == 1) {
        const uint32_t remote = map_to_rank(sb, 0) + (uint32_t)(m * kPartPitch * 4);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(lane_base + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; j += 4) st_cluster_v4(remote + (uint32_t)((c0 + j) * 4), r[j], r[j + 1], r[j + 2], r[j + 3]);
        }
    }
    cluster_sync();  // rank 1's partial sums are in rank 0's shared memory
    if (warp >= 2 && rank == 0) {
        const int feat = f * BM + m;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(lane_base + c0, r);
            tmem_wait_ld();
            const int nrow = min(16, a.M - c0);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (j >= nrow) continue;
                const float v = failed ? __int_as_float(0x7fc00000) : __uint_as_float(r[j]) + part[c0 + j];
                if (a.out_bf16)
                    reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)(c0 + j) * a.N + feat] = __float2bfloat16_rn(v);
                else
                    reinterpret_cast<float *>(a.out)[(size_t)(c0 + j) * a.N + feat] = v;
            }
        }
    }
    fence_before_sync();
    if (__syncthreads_or(failed) && threadIdx.x == 0) atomicAdd(&g_oproj_timeouts, 1);
    fence_after_sync();
    if (warp == 1) tmem_dealloc(tb, BN);
}

// ---------------------------------------------------------------------------
// Pair form: two CTAs of a cluster run one 256-feature x 256-row tile as 2-SM products
// (tcgen05 cta_group::2).  Each CTA stages 128 w_o rows and 128 y rows of every 64-wide K
// slice (32 KB, against 48 KB for a 128 x 256 tile on one SM), and the even CTA's MMA
// thread issues M = 256, N = 256 products that read both CTAs' halves: features
// [0, 128) of the tile land in the even CTA's TMEM, [128, 256) in the odd CTA's, each with
// all 256 rows.  Both CTAs' loads complete on the even CTA's full barrier; its commits
// arrive at the same barrier offset in both CTAs (multicast); the odd CTA's epilogue
// warps arrive remotely on the even CTA's acc_empty.  SPLIT = 2 (the decode batch, one
// tile per cluster of four): ranks 0-1 run the first half of K and ranks 2-3 the second;
// rank r + 2 adds its fp32 accumulator into rank r's shared memory before rank r writes.

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the barrier at `bar`'s offset in every CTA of `mask` once the pair's
// products issued so far by this thread complete.
__device__ __forceinline__ void mma_pair_commit(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
// A 2-D tile into this CTA's shared memory, completing on the pair's barrier at the
// shared::cluster address `bar` (which may be in the other CTA of the pair).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// NSUB = 1: a 256-feature x 256-row tile.  NSUB = 2 (long prompts): 256 features x 512
// rows, two N = 256 products per K step on the same w_o slice, so an SM takes 48 KB per
// 8 products instead of 32 KB per 4: 42 instead of 56 bytes per cycle of tensor work at
// the bf16 rate, and about the same bytes in flight (4 stages of 48 KB against 6-7 of
// 32 KB) cover a third more load latency.  Its 512 TMEM columns hold one accumulator, so
// a tile's epilogue no longer overlaps the next tile's products.  NSUB = 1 takes a seventh
// stage (224 KB), which the shared memory just holds.
template <int NSUB>
struct PairCfg {
    static constexpr int BN = 256 * NSUB;              // rows of y per tile (128 of each 256 staged per CTA)
    static constexpr int STAGES = NSUB == 1 ? 7 : 4;
    static constexpr uint32_t A_BYTES = 128 * BK * 2;  // this CTA's 128 w_o rows
    static constexpr uint32_t B_BYTES = 128 * BK * 2;  // this CTA's 128 y rows of each 256-row sub-tile
    static constexpr uint32_t STAGE = A_BYTES + NSUB * B_BYTES;
    static constexpr uint32_t BARS = STAGES * STAGE;   // full[S], empty[S], acc_full[2], acc_empty[2], drain
    static constexpr uint32_t SMEM = BARS + (2 * STAGES + 5) * 8 + 16 + 1024;
};
static_assert(PairCfg<1>::SMEM <= 232448 && PairCfg<2>::SMEM <= 232448, "shared memory budget");

// Tile id -> (256-feature tile, row tile): groups of 14 feature tiles (3584 features)
// across every row tile, so the pairs running together share w_o and y through L2.  With
// 256-row tiles, the 76 pairs' tiles in flight cover 14 feature tiles by about 5.4 row
// tiles, about 120 MB of operands (the L2 holds 129 MB), and y is read from DRAM twice per
// call at 7168 features.  Measured at 8192 x 12288 -> 7168 on one GPU: 0.767 ms with 14,
// 0.776 with 7, 0.790 with 4, 0.815 with 28; with 512-row tiles 0.716 ms with 14, 0.718
// with 10, 0.720 with 28, 0.733 with 7.
__device__ __forceinline__ void pair_tile_coords(int id, int n_ft, int n_tt, int &f, int &t) {
    constexpr int G = 14;
    const int per_group = G * n_tt;
    const int g = id / per_group, r = id % per_group;
    const int f0 = g * G, gsz = min(G, n_ft - f0);
    f = f0 + r % gsz;
    t = r / gsz;
}

template <int SPLIT, int NSUB>
__global__ void __launch_bounds__(kWarps * 32, 1)
    oproj_pair_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_y,
                      const __grid_constant__ GemmArgs a) {
    static_assert(SPLIT == 1 || NSUB == 1, "the split-K form runs 256-row tiles");
    using L = PairCfg<NSUB>;
    constexpr int BN = L::BN;
    constexpr uint32_t NACC = SPLIT == 1 && NSUB == 1 ? 2 : 1;  // accumulator buffers (BN TMEM columns each)
    constexpr uint32_t TMEM_COLS = NACC * BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm), sb16 = sb >> 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::BARS);
    uint64_t *empty = full + L::STAGES;
    uint64_t *acc_full = empty + L::STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), pr = rank & 1u, leader = rank & ~1u;
    const uint16_t pair_mask = (uint16_t)(3u << leader);
    // the tiles of this pair: SPLIT 1 walks tiles with the pair count as stride; SPLIT 2
    // has one tile per cluster and a K half per pair
    const int KB = a.K / BK;
    const int kb0 = SPLIT == 1 ? 0 : (int)(rank >> 1) * (KB / 2), kb1 = SPLIT == 1 ? KB : kb0 + KB / 2;
    const int pair_id = SPLIT == 1 ? (int)(blockIdx.x >> 1) : (int)(blockIdx.x >> 2);
    const int pair_stride = SPLIT == 1 ? (int)(gridDim.x >> 1) : a.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, 8);  // one arrival per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    fence_before_sync();
    __syncwarp();
    cluster_sync();  // every barrier of the cluster is initialised before any remote use
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    const uint32_t full_leader = map_to_rank(smem_u32(full), leader);
    const uint32_t acc_empty_leader = map_to_rank(smem_u32(acc_empty), leader);
    int failed = 0;

    if (warp == 0) {
        if (lane == 0) {  // ---- TMA producer (both CTAs): this CTA's halves of each stage
            uint32_t it = 0;
            for (int id = pair_id; id < a.n_tiles && !failed; id += pair_stride) {
                int f, t;
                if (SPLIT == 1)
                    pair_tile_coords(id, a.n_ft, a.n_tt, f, t);
                else
                    f = id, t = 0;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % L::STAGES, use = it / L::STAGES;
                    if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1, kPolls)) {
                        failed = 1;
                        *abort_flag = 1;
                        break;
                    }
                    if (pr == 0) mbar_arrive_expect_tx(full + s, 2 * L::STAGE);  // both CTAs' bytes
                    tma_load_2d_pair(sb + s * L::STAGE, &tmap_w, full_leader + s * 8, kb * BK, f * 256 + (int)pr * 128);
#pragma unroll
                    for (int u = 0; u < NSUB; ++u)  // rows past M (or a whole sub-tile) arrive as zeros
                        tma_load_2d_pair(sb + s * L::STAGE + L::A_BYTES + u * L::B_BYTES, &tmap_y, full_leader + s * 8,
                                         kb * BK, t * BN + u * 256 + (int)pr * 128);
                }
            }
            // the loads issued have landed once the products that read them have completed
            const uint32_t n_issued = it;
            for (uint32_t s = 0; s < (uint32_t)L::STAGES && s < n_issued; ++s) {
                const uint32_t last = n_issued - 1 - ((n_issued - 1 + L::STAGES - s) % L::STAGES);
                mbar_wait(empty + s, (last / L::STAGES) & 1, kPolls);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && pr == 0) {  // ---- MMA issuer (even CTA)
            const uint32_t idesc = idesc_bf16(256, 256, false, false);
            uint32_t it = 0, tc = 0;
            for (int id = pair_id; id < a.n_tiles && !failed; id += pair_stride, ++tc) {
                const uint32_t acc = tc % NACC, use = tc / NACC;
                if (use > 0 && !mbar_wait(acc_empty + acc, (use - 1) & 1, kPolls)) {  // both epilogues read it
                    failed = 1;
                    *abort_flag = 1;
                    break;
                }
                fence_after_sync();
                const uint32_t d = tb + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % L::STAGES;
                    if (!mbar_wait(full + s, (it / L::STAGES) & 1, kPolls)) {
                        failed = 1;
                        *abort_flag = 1;
                        break;
                    }
                    fence_after_sync();
                    const uint32_t sa = s * L::STAGE, sbb = sa + L::A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
#pragma unroll
                        for (int u = 0; u < NSUB; ++u)  // sub-tile u: rows u * 256.. in TMEM columns u * 256..
                            mma_pair_ss(d + u * 256, sdesc_at(sb16, sa + k * 32, 16, 1024),
                                        sdesc_at(sb16, sbb + u * L::B_BYTES + k * 32, 16, 1024), idesc,
                                        (kb > kb0 || k) ? 1u : 0u);
                    mma_pair_commit(empty + s, pair_mask);  // both CTAs' stage s is free once these complete
                }
                if (failed) break;
                mma_pair_commit(acc_full + acc, pair_mask);
            }
            mma_pair_commit(drain, pair_mask);  // nothing issued may still run when TMEM is freed
        }
        if (lane == 0) mbar_wait(drain, 0, kPolls);
        __syncwarp();
    } else {  // ---- epilogue, warps 2-5 of both CTAs: TMEM lane quarter warp % 4
        const int q = warp & 3, m = q * 32 + lane;
        const uint32_t lane_base = tb + ((uint32_t)(q * 32) << 16);
        uint32_t tc = 0;
        for (int id = pair_id; id < a.n_tiles; id += pair_stride, ++tc) {
            int f, t;
            if (SPLIT == 1)
                pair_tile_coords(id, a.n_ft, a.n_tt, f, t);
            else
                f = id, t = 0;
            const uint32_t acc = tc % NACC, use = tc / NACC;
            const bool ok = !failed && !*abort_flag && mbar_wait(acc_full + acc, use & 1, kPolls);
            if (!ok) failed = 1;
            fence_after_sync();
            if (SPLIT == 1) {
                const int feat = f * 256 + (int)pr * 128 + m;
                const int t0 = t * BN;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t r0[16], r1[16];
                    if (ok) {
                        tmem_ld16(lane_base + acc * BN + c0, r0);
                        tmem_ld16(lane_base + acc * BN + c0 + 16, r1);
                        tmem_wait_ld();
                    }
                    const int nrow = min(32, a.M - (t0 + c0));
                    if (a.out_bf16) {
                        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(a.out) + (size_t)(t0 + c0) * a.N + feat;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nrow)
                                o[(size_t)j * a.N] = __float2bfloat16_rn(
                                    ok ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) : __int_as_float(0x7fc00000));
                    } else {
                        float *o = reinterpret_cast<float *>(a.out) + (size_t)(t0 + c0) * a.N + feat;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nrow)
                                o[(size_t)j * a.N] =
                                    ok ? __uint_as_float(j < 16 ? r0[j] : r1[j - 16]) : __int_as_float(0x7fc00000);
                    }
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0 && ok) {
                    if (pr == 0)
                        mbar_arrive(acc_empty + acc);
                    else
                        mbar_arrive_cluster(acc_empty_leader + acc * 8);
                }
            }
        }
    }
    if constexpr (SPLIT == 2) {
        // every product of the cluster is done (each epilogue warp saw its acc_full): the
        // upper pair's partial sums go into the lower pair's idle stage buffers
        __syncwarp();
        cluster_sync();
        constexpr int kPartPitch = BN + 4;
        static_assert(128 * kPartPitch * 4 <= L::STAGES * L::STAGE, "the partial sums fit in the stage buffers");
        const int q = warp & 3, m = q * 32 + lane;
        const uint32_t lane_base = tb + ((uint32_t)(q * 32) << 16);
        if (warp >= 2 && rank >= 2) {
            const uint32_t remote = map_to_rank(sb, rank - 2) + (uint32_t)(m * kPartPitch * 4);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(lane_base + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                    st_cluster_v4(remote + (uint32_t)((c0 + j) * 4), r[j], r[j + 1], r[j + 2], r[j + 3]);
            }
        }
        // a CTA of the upper pair that gave up marks the lower CTA it feeds, whose outputs
        // then hold NaN
        const int any_fail = __syncthreads_or(failed || *abort_flag);
        if (rank >= 2 && threadIdx.x == 0 && any_fail) {
            const uint32_t remote_flag = map_to_rank(smem_u32((const void *)abort_flag), rank - 2);
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote_flag), "r"(1) : "memory");
        }
        __syncwarp();
        cluster_sync();  // the partial sums (and any abort mark) are in place
        if (warp >= 2 && rank < 2) {
            const int f = pair_id;
            const int feat = f * 256 + (int)pr * 128 + m;
            const float *part = reinterpret_cast<const float *>(sm) + m * kPartPitch;
            // a timeout anywhere in the cluster shows in the flags of the CTAs that gave up;
            // this CTA's own flag and waits cover its half
            const bool bad = failed || *abort_flag;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(lane_base + c0, r);
                tmem_wait_ld();
                const int nrow = min(16, a.M - c0);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (j >= nrow) continue;
                    const float v = bad ? __int_as_float(0x7fc00000) : __uint_as_float(r[j]) + part[c0 + j];
                    if (a.out_bf16)
                        reinterpret_cast<__nv_bfloat16 *>(a.out)[(size_t)(c0 + j) * a.N + feat] = __float2bfloat16_rn(v);
                    else
                        reinterpret_cast<float *>(a.out)[(size_t)(c0 + j) * a.N + feat] = v;
                }
            }
        }
    }
    fence_before_sync();
    if (__syncthreads_or(failed) && threadIdx.x == 0) atomicAdd(&g_oproj_timeouts, 1);
    __syncwarp();
    cluster_sync();  // both CTAs of each pair are done with TMEM before it is freed
    fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tb, TMEM_COLS);
}

}  // namespace

int take_oproj_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_oproj_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_oproj_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("o_proj: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

bool o_proj_supported(int K, int N) { return K % BK == 0 && N % BM == 0; }

kda_status launch_o_proj(const void *y, const void *w, void *out, int out_bf16, int64_t M, int K, int N,
                         cudaStream_t st) {
    if (!o_proj_supported(K, N)) {
        set_error("o_proj: in_features must be a multiple of %d and out_features of %d", BK, BM);
        return KDA_ERR_UNSUPPORTED;
    }
    if (M == 0) return KDA_OK;
    chunk::EncodeTiledFn enc = reinterpret_cast<chunk::EncodeTiledFn>(tensor_map_encoder());
    if (!enc) {
        set_error("o_proj: cuTensorMapEncodeTiled is not available from the driver");
        return KDA_ERR_CUDA;
    }
    const int sms = sm_count();
    const int n_ft = N / BM;
    const int n_tt256 = (int)((M + 255) / 256);
    const int BN = (int64_t)n_ft * n_tt256 >= sms ? 256 : 128;
    const int n_tt = (int)((M + BN - 1) / BN);
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap tw, ty;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BM};
        const CUresult r = enc(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_error("o_proj: cuTensorMapEncodeTiled failed for w_o (%d)", (int)r);
            return KDA_ERR_CUDA;
        }
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)BN};
        const CUresult r = enc(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(y), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_error("o_proj: cuTensorMapEncodeTiled failed for y (%d)", (int)r);
            return KDA_ERR_CUDA;
        }
    }
    static DeviceOnce configured;
    const int dev = current_device();
    if (N % 256 == 0) {
        // the pair form: 256-feature tiles on CTA pairs; a decode batch splits K over two pairs
        static DeviceOnce configured_pair;
        if (!configured_pair.done(dev)) {
            cudaError_t e = cudaFuncSetAttribute(oproj_pair_kernel<1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 PairCfg<1>::SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(oproj_pair_kernel<1, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<2>::SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(oproj_pair_kernel<2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg<1>::SMEM);
            if (e != cudaSuccess) {
                set_error("o_proj: cannot reserve shared memory: %s", cudaGetErrorString(e));
                return KDA_ERR_CUDA;
            }
            configured_pair.set(dev);
        }
        CUtensorMap ty128;
        {
            const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
            const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
            const cuuint32_t box[2] = {(cuuint32_t)BK, 128u};
            const CUresult r = enc(&ty128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(y), dims, strides,
                                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) {
                set_error("o_proj: cuTensorMapEncodeTiled failed for y (%d)", (int)r);
                return KDA_ERR_CUDA;
            }
        }
        const int n_ft2 = N / 256;
        const bool split = M <= 256 && (K / BK) % 2 == 0 && 4 * n_ft2 <= sms;
        // 512-row tiles where there are more than 256 rows and every pair still gets a tile
        const bool wide = !split && M > 256 && (int64_t)n_ft2 * ((M + 511) / 512) >= sms / 2;
        const int tile_rows = wide ? 512 : 256;
        GemmArgs ga;
        memset(&ga, 0, sizeof(ga));
        ga.out = out;
        ga.out_bf16 = out_bf16;
        ga.M = (int)M;
        ga.N = N;
        ga.K = K;
        ga.n_ft = n_ft2;
        ga.n_tt = split ? 1 : (int)((M + tile_rows - 1) / tile_rows);
        ga.n_tiles = ga.n_ft * ga.n_tt;
        const int pairs = ga.n_tiles < sms / 2 ? ga.n_tiles : sms / 2;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(split ? 4 * n_ft2 : 2 * pairs, 1, 1);
        cfg.blockDim = dim3(kWarps * 32, 1, 1);
        cfg.dynamicSmemBytes = wide ? PairCfg<2>::SMEM : PairCfg<1>::SMEM;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = split ? 4 : 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = split  ? cudaLaunchKernelEx(&cfg, oproj_pair_kernel<2, 1>, tw, ty128, ga)
                              : wide ? cudaLaunchKernelEx(&cfg, oproj_pair_kernel<1, 2>, tw, ty128, ga)
                                     : cudaLaunchKernelEx(&cfg, oproj_pair_kernel<1, 1>, tw, ty128, ga);
        note_launch();
        if (e != cudaSuccess) {
            set_error("oproj_pair_kernel: %s", cudaGetErrorString(e));
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        return check_launch("oproj_pair_kernel");
    }
    if (!configured.done(dev)) {
        cudaError_t e = cudaFuncSetAttribute(oproj_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<256>::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(oproj_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::SMEM);
        if (e != cudaSuccess) {
            set_error("o_proj: cannot reserve shared memory: %s", cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
        configured.set(dev);
    }
    const bool splitk = M <= 256 && (K / BK) % 2 == 0 && 2 * n_ft <= sms;
    if (splitk) {
        static DeviceOnce configured_sk;
        if (!configured_sk.done(dev)) {
            const cudaError_t e = cudaFuncSetAttribute(oproj_splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       Cfg<256>::SMEM);
            if (e != cudaSuccess) {
                set_error("o_proj: cannot reserve shared memory: %s", cudaGetErrorString(e));
                return KDA_ERR_CUDA;
            }
            configured_sk.set(dev);
        }
        CUtensorMap ty256;
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)BK, 256u};
        const CUresult r = enc(&ty256, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(y), dims, strides, box,
                               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_error("o_proj: cuTensorMapEncodeTiled failed for y (%d)", (int)r);
            return KDA_ERR_CUDA;
        }
        GemmArgs ga;
        memset(&ga, 0, sizeof(ga));
        ga.out = out;
        ga.out_bf16 = out_bf16;
        ga.M = (int)M;
        ga.N = N;
        ga.K = K;
        ga.n_ft = n_ft;
        ga.n_tt = 1;
        ga.n_tiles = n_ft;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(2 * n_ft, 1, 1);
        cfg.blockDim = dim3(kWarps * 32, 1, 1);
        cfg.dynamicSmemBytes = Cfg<256>::SMEM;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, oproj_splitk_kernel, tw, ty256, ga);
        note_launch();
        if (e != cudaSuccess) {
            set_error("oproj_splitk_kernel: %s", cudaGetErrorString(e));
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        return check_launch("oproj_splitk_kernel");
    }
    GemmArgs ga;
    memset(&ga, 0, sizeof(ga));
    ga.out = out;
    ga.out_bf16 = out_bf16;
    ga.M = (int)M;
    ga.N = N;
    ga.K = K;
    ga.n_ft = n_ft;
    ga.n_tt = n_tt;
    ga.n_tiles = n_ft * n_tt;
    const int grid = ga.n_tiles < sms ? ga.n_tiles : sms;
    if (BN == 256)
        oproj_kernel<256><<<grid, kWarps * 32, Cfg<256>::SMEM, st>>>(tw, ty, ga);
    else
        oproj_kernel<128><<<grid, kWarps * 32, Cfg<128>::SMEM, st>>>(tw, ty, ga);
    note_launch();
    return check_launch("oproj_kernel");
}

}  // namespace kda
