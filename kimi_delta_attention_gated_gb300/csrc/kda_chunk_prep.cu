// kda_chunk_prep.cu -- the state-independent half of the split chunked prefill.
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (a prompt runs a
// chunked kernel that carries the state from one 64-token chunk to the next), sections
// 03/04 (per-key-channel decay applied before each delta-rule update, q and k
// L2-normalised in the kernel, q scaled by 1/sqrt(key_dim)).
//
// Everything of a chunk that does not depend on the state entering it (kda_chunk_common.cuh
// has the algebra): the L2 norms, the in-chunk cumulative decay, the decay-folded grams
//   A = strict_lower(diag(beta) Kd Km^T),  P = lower(Qd Km^T)
// on the tensor cores (tcgen05, split-bf16 operands hi*hi + hi*lo + lo*hi, fp32
// accumulation in TMEM), and the UT transform T = (I + A)^-1 (blocked, fp32 on CUDA
// cores).  T diag(beta) and P leave as split-bf16 operand images (kBlobBytes per chunk,
// the byte image of the chain kernel's shared-memory tiles) in the caller's workspace;
// the per-head chain kernel (kda_chunk_chain.cu) copies them straight into its tiles.
// Chunks whose decay range exceeds kRangeMax compute A and P exactly on CUDA cores with
// pairwise exponentials (Km would overflow there).
//
// Every item (chunk, head) is independent, so the kernel runs over all of them at once
// instead of one head per SM: persistent CTAs of 8 warps, two per SM (106 KB of shared
// memory and 128 TMEM columns each), walk the items with the grid as stride.  Warp w holds
// the tokens 8w..8w+7 of a chunk, lane l the key channels 4l..4l+3.  The next item's q,
// k and beta are loaded while the gram runs and its g arrives by TMA during the solve;
// while one CTA waits on its gram or solves, the other on the SM prepares its next chunk.
//
// The arithmetic of the norms, the cumulative decay (totals per group of 4 tokens, then
// their exclusive prefix), the operand tiles, the gram pass and the solve is the fused
// kernel's (kda_chunk_tc.cu), operation for operation, so the two forms give the same bits.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include "kda_chunk_common.cuh"
#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace chunk;

constexpr int kPT = 256;  // 8 warps

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t P_KQH = 0;      // [-Kd ; Qd] hi, 128 rows x 128 (32 KB)
constexpr uint32_t P_KQL = 32768;  // [-Kd ; Qd] lo
constexpr uint32_t P_KM = 65536;   // [Km hi ; Km lo] (32 KB); the chunk's g tile lands here first
// once the gram has read the [-Kd ; Qd] tiles their 64 KB hold the solve's buffers:
constexpr uint32_t P_A = 0;                     // A fp32 [64][AP]; after the solve, the T diag(beta) image (16 KB)
constexpr uint32_t P_T = P_A + 64 * AP * 4;     // T fp32 [64][AP]
constexpr uint32_t P_PIMG = P_T + 64 * AP * 4;  // P image, hi then lo (16 KB)
constexpr uint32_t P_SMALL = 98304;
// small buffers (floats)
constexpr uint32_t PF_BETA = 0;            // beta [64]
constexpr uint32_t PF_RQ = 64;             // q scale per token (norm * scale) [64]
constexpr uint32_t PF_RK = 128;            // k norm per token [64]
constexpr uint32_t PF_TOT = 192;           // decay totals of the 16 groups of 4 tokens [16][128]
constexpr uint32_t PF_END = PF_TOT + 2048;
constexpr uint32_t P_BARS = P_SMALL + PF_END * 4;  // 3 mbarriers, tmem slot, the next item's index
constexpr uint32_t PREP_SMEM = P_BARS + 48 + 1024;
// fallback (decay range too wide): exact G in the Km tile, P in fp32 where T goes
constexpr uint32_t P_FB_G = P_KM;

static_assert(P_PIMG + 16384 <= P_KM, "the solve's buffers fit in the dead [-Kd ; Qd] tiles");
static_assert(PREP_SMEM <= 113 * 1024, "two CTAs per SM");

// Set by a CTA whose bounded wait gave up; the workspace blobs of that item and of every
// later item of the CTA then hold NaN, which the chain kernel carries into o, y, the state.
__device__ int g_chunk_prep_timeouts = 0;

struct PrepArgs {
    SeqParams p;
    uint8_t *ws;      // workspace: n_slots x H blobs of kBlobBytes
    int64_t n_slots;  // blob_slots(rows, N)
    // concurrent form (null: split form): a blob's flag is set once its stores are complete;
    // an item is skipped while its (sequence, head)'s fused CTA has begun (progress) within
    // `lead` chunks of it, since that CTA decides for itself before the blob could be ready
    uint32_t *flags;
    const uint32_t *progress;
    int lead;
};

// Sequence n and chunk c of slot `slot`; false for a slot no chunk uses.  Slot starts
// are non-decreasing in n, so the sequence is the last one starting at or before it.
__device__ __forceinline__ bool slot_item(const SeqParams &p, int64_t slot, int &n, int &c, int &bos, int &len) {
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        int b, l;
        seq_range(p, mid, b, l);
        if (blob_slot(b, mid, 0) <= slot)
            lo = mid;
        else
            hi = mid - 1;
    }
    n = lo;
    seq_range(p, n, bos, len);
    const int64_t cc = slot - blob_slot(bos, n, 0);
    c = (int)cc;
    return cc >= 0 && cc * C < len;
}

struct Item {
    int64_t idx;  // slot * H + h, or >= n_items when done
    int n, c, h, bos, cn;
};

// The first item at or after idx (stepping by `step`) that a chunk uses.
__device__ __forceinline__ Item next_item(const SeqParams &p, int64_t idx, int64_t step, int64_t n_items) {
    Item it;
    for (; idx < n_items; idx += step) {
        int n, c, bos, len;
        if (slot_item(p, idx / p.H, n, c, bos, len)) {
            it.idx = idx;
            it.n = n;
            it.c = c;
            it.h = (int)(idx % p.H);
            it.bos = bos;
            it.cn = min(C, len - c * C);
            return it;
        }
    }
    it.idx = n_items;
    it.n = it.c = it.h = it.bos = it.cn = 0;
    return it;
}

// The index of the next item to run, at or after idx: next_item's choice, then, in the
// concurrent form, past every item whose fused CTA is already close to it (thread 0 only:
// the progress words change under it, so the CTA takes this one thread's choice).
__device__ __forceinline__ int64_t choose_item(const PrepArgs &a, int64_t idx, int64_t step, int64_t n_items) {
    for (;;) {
        const Item it = next_item(a.p, idx, step, n_items);
        if (it.idx >= n_items || !a.progress) return it.idx;
        const uint32_t begun = ld_relaxed_gpu(a.progress + (size_t)it.n * a.p.H + it.h);
        if ((int64_t)begun + a.lead <= it.c) return it.idx;
        idx = it.idx + step;
    }
}

// One item's q and k for this thread's 8 tokens x 4 key channels, and beta (or its logit's
// raw bits) of token 8 warp + lane for lanes 0-7.  Rows past the chunk's end read its last
// row and are zeroed when the chunk is prepared.
template <bool GL>
__device__ __forceinline__ void load_item(const SeqParams &p, const Item &it, uint2 (&q)[8], uint2 (&k)[8],
                                          float &beta, int warp, int lane) {
    if (it.cn <= 0) return;
    const int t0 = it.bos + it.c * C, l4 = lane * 4;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int i = min(warp * 8 + r, it.cn - 1);
        const size_t hk = ((size_t)(t0 + i) * p.H + it.h) * DK + l4;
        q[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) + hk));
        k[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.k) + hk));
    }
    const size_t bi = (size_t)(t0 + min(warp * 8 + (lane & 7), it.cn - 1)) * p.H + it.h;
    if (!GL) {
        beta = __ldg(p.beta + bi);
    } else {
        uint32_t raw;
        if (p.beta_logits_bf16)
            asm("ld.global.nc.u16 %0, [%1];" : "=r"(raw) : "l"(reinterpret_cast<const uint16_t *>(p.beta_logits) + bi));
        else
            asm("ld.global.nc.u32 %0, [%1];" : "=r"(raw) : "l"(reinterpret_cast<const uint32_t *>(p.beta_logits) + bi));
        beta = __uint_as_float(raw);
    }
}

// One 16 x 16 x 16 product of the triangular solve by one warp, each lane a 2 x 4 strip:
// dst = (acc ? dst : 0) + sign * X Y, blocks addressed by their top-left element.  Every
// output element is summed over k in order with the same packed operations as the fused
// kernel's 64-thread form, so the two give the same bits.
__device__ __forceinline__ void blk16w(float *dst, const float *X, const float *Y, float sign, bool acc, int lane) {
    const int r = (lane >> 2) * 2, c4 = (lane & 3) * 4;
    float x[2][16];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(X + (r + rr) * AP + k);
            x[rr][k] = v.x; x[rr][k + 1] = v.y; x[rr][k + 2] = v.z; x[rr][k + 3] = v.w;
        }
    float2 s01[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, s23[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float4 y = *reinterpret_cast<const float4 *>(Y + k * AP + c4);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const float2 xk = make_float2(x[rr][k], x[rr][k]);
            s01[rr] = __ffma2_rn(xk, make_float2(y.x, y.y), s01[rr]);
            s23[rr] = __ffma2_rn(xk, make_float2(y.z, y.w), s23[rr]);
        }
    }
    const float2 sg = make_float2(sign, sign);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float *d = dst + (r + rr) * AP + c4;
        const float4 o = acc ? *reinterpret_cast<const float4 *>(d) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float2 o01 = __ffma2_rn(sg, s01[rr], make_float2(o.x, o.y));
        const float2 o23 = __ffma2_rn(sg, s23[rr], make_float2(o.z, o.w));
        *reinterpret_cast<float4 *>(d) = make_float4(o01.x, o01.y, o23.x, o23.y);
    }
}

template <bool GL>
__global__ void __launch_bounds__(kPT, 2)
    chunk_prep_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ PrepArgs a) {
    const SeqParams &p = a.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm), sb16 = sb >> 4;
    float *fs = reinterpret_cast<float *>(sm + P_SMALL);
    float *Asm = reinterpret_cast<float *>(sm + P_A);
    float *Tsm = reinterpret_cast<float *>(sm + P_T);
    uint64_t *gram_bar = reinterpret_cast<uint64_t *>(sm + P_BARS);  // gram product of an item
    uint64_t *g_bar = gram_bar + 1;                                   // g tile of an item
    uint64_t *drain_bar = gram_bar + 2;                               // drain after a failure
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + P_BARS + 24);
    volatile int64_t *next_idx = reinterpret_cast<volatile int64_t *>(sm + P_BARS + 32);  // thread 0's choice

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, l4 = lane * 4;
    const int H = p.H;
    const int64_t n_items = a.n_slots * H, step = gridDim.x;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    if (tid == 0) {
        mbar_init(gram_bar, 1);
        mbar_init(g_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        *next_idx = choose_item(a, blockIdx.x, step, n_items);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    Item cur = next_item(p, *next_idx, step, n_items);
    uint2 q[8], k[8];
    float beta_r = 0.f;
    load_item<GL>(p, cur, q, k, beta_r, warp, lane);

    const uint32_t g_bytes = (GL && p.g_logits_bf16) ? C * DK * 2 : C * DK * 4;
    auto issue_g = [&](const Item &it) {
        mbar_arrive_expect_tx(g_bar, g_bytes);
        tma_load_3d(sb + P_KM, &tmap_g, g_bar, 0, it.h, it.bos + it.c * C);
    };
    uint32_t g_issued = 0, g_seen = 0;  // thread 0: g tiles issued, and seen complete
    bool stores_pending = false;         // thread 0: blob stores not yet known to have read the staging
    int64_t flag_pending = -1;           // thread 0: the flag of the blob those stores write
    // thread 0: once the pending stores have completed, the blob's flag (concurrent form)
    auto publish = [&]() {
        if (flag_pending >= 0) {
            fence_proxy_async_global();
            st_release_gpu(a.flags + flag_pending, 1u);
            flag_pending = -1;
        }
    };
    if (tid == 0 && cur.idx < n_items) {
        issue_g(cur);
        ++g_issued;
    }

    int failed = 0;
    uint32_t n_done = 0;  // items finished by this CTA: the phase of g_bar and gram_bar
    while (cur.idx < n_items) {
        const int cn = cur.cn, h = cur.h;
        const uint32_t par = n_done & 1;
        uint8_t *blob = a.ws + ((size_t)blob_slot(cur.bos, cur.n, cur.c) * H + h) * kBlobBytes;

        // ---- norms, beta and the decay totals of each group of 4 tokens, from the g tile
        if (!mbar_wait(g_bar, par, kPolls))
            failed = 1;
        else if (tid == 0)
            ++g_seen;
        float4 g[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = warp * 8 + r;
            if (i >= cn) {
                q[r] = make_uint2(0u, 0u);
                k[r] = make_uint2(0u, 0u);
            }
            if (GL && p.g_logits_bf16) {
                const uint2 u = *reinterpret_cast<const uint2 *>(sm + P_KM + (i * DK + l4) * 2);
                g[r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), 0.f, 0.f);
            } else {
                g[r] = *reinterpret_cast<const float4 *>(sm + P_KM + (i * DK + l4) * 4);
            }
            if (!GL && i >= cn) g[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (GL) {  // g from its logits; tokens past the chunk's end keep g = 0
            const float a_h = __expf(__ldg(p.A_log + h));
            const float4 db = p.dt_bias ? __ldg(reinterpret_cast<const float4 *>(p.dt_bias + (size_t)h * DK + l4))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float z[4];
                if (p.g_logits_bf16) {
                    const uint32_t ux = __float_as_uint(g[r].x), uy = __float_as_uint(g[r].y);
                    z[0] = bf16lo(ux); z[1] = bf16hi(ux); z[2] = bf16lo(uy); z[3] = bf16hi(uy);
                } else {
                    z[0] = g[r].x; z[1] = g[r].y; z[2] = g[r].z; z[3] = g[r].w;
                }
                const bool live = warp * 8 + r < cn;
                g[r] = make_float4(live ? gate_of_logit(z[0] + db.x, a_h, p.g_lower) : 0.f,
                                   live ? gate_of_logit(z[1] + db.y, a_h, p.g_lower) : 0.f,
                                   live ? gate_of_logit(z[2] + db.z, a_h, p.g_lower) : 0.f,
                                   live ? gate_of_logit(z[3] + db.w, a_h, p.g_lower) : 0.f);
            }
            if (lane < 8) {
                const uint32_t raw = __float_as_uint(beta_r);
                beta_r = warp * 8 + lane < cn ? beta_of_logit(__uint_as_float(p.beta_logits_bf16 ? raw << 16 : raw))
                                              : 0.f;
            }
        }
        if (!GL && warp * 8 + lane >= cn) beta_r = 0.f;
        {
            // sums of squares of q and k for the 8 tokens, reduced over the warp by a
            // reduce-scatter: lanes 2v and 2v + 1 end with sum v (q of tokens 0-7, then k)
            float a16[16];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float2 v0 = make_float2(bf16lo(q[r].x), bf16lo(k[r].x));
                const float2 v1 = make_float2(bf16hi(q[r].x), bf16hi(k[r].x));
                const float2 v2 = make_float2(bf16lo(q[r].y), bf16lo(k[r].y));
                const float2 v3 = make_float2(bf16hi(q[r].y), bf16hi(k[r].y));
                const float2 ss = __ffma2_rn(v0, v0, __ffma2_rn(v1, v1, __ffma2_rn(v2, v2, __fmul2_rn(v3, v3))));
                a16[r] = ss.x;
                a16[8 + r] = ss.y;
            }
            const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
            float b8[8], b4[4], b2[2];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                b8[j] = (u16 ? a16[j + 8] : a16[j]) + __shfl_xor_sync(0xffffffffu, u16 ? a16[j] : a16[j + 8], 16);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                b4[j] = (u8 ? b8[j + 4] : b8[j]) + __shfl_xor_sync(0xffffffffu, u8 ? b8[j] : b8[j + 4], 8);
#pragma unroll
            for (int j = 0; j < 2; ++j)
                b2[j] = (u4 ? b4[j + 2] : b4[j]) + __shfl_xor_sync(0xffffffffu, u4 ? b4[j] : b4[j + 2], 4);
            float d = (u2 ? b2[1] : b2[0]) + __shfl_xor_sync(0xffffffffu, u2 ? b2[0] : b2[1], 2);
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            if ((lane & 1) == 0) {
                const int v = lane >> 1;
                const float sc = p.l2norm ? rsqrtf(d + 1e-6f) : 1.f;
                if (v < 8)
                    fs[PF_RQ + warp * 8 + v] = sc * p.scale;
                else
                    fs[PF_RK + warp * 8 + v - 8] = sc;
            }
        }
        if (lane < 8) fs[PF_BETA + warp * 8 + lane] = beta_r;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // totals of tokens 8w..8w+3 and 8w+4..8w+7
            float2 t01 = make_float2(g[4 * half].x, g[4 * half].y), t23 = make_float2(g[4 * half].z, g[4 * half].w);
#pragma unroll
            for (int r = 1; r < 4; ++r) {
                t01 = __fadd2_rn(t01, make_float2(g[4 * half + r].x, g[4 * half + r].y));
                t23 = __fadd2_rn(t23, make_float2(g[4 * half + r].z, g[4 * half + r].w));
            }
            *reinterpret_cast<float4 *>(fs + PF_TOT + (2 * warp + half) * 128 + l4) = make_float4(t01.x, t01.y, t23.x, t23.y);
        }
        // the previous item's blob stores must have read the staging before the tiles below
        // overwrite it; in the concurrent form they must also be complete, and the blob's
        // flag is set
        if (tid == 0 && stores_pending) {
            if (a.flags) {
                bulk_wait_all();
                publish();
            } else {
                bulk_wait_read_all();
            }
            stores_pending = false;
        }
        __syncthreads();
        // ---- operand tiles: [-Kd ; Qd] and Km, hi and lo.  Each thread forms the exclusive
        // prefix of the 16 group totals for its channels and the chunk total itself, summing
        // the totals in order (the fused kernel's order, so the same bits) with no barrier
        int oor = 0;
        {
            float o4[2][4], gam[4] = {0.f, 0.f, 0.f, 0.f};
            auto add_total = [&](int w) {
                const float4 t = *reinterpret_cast<const float4 *>(fs + PF_TOT + w * 128 + l4);
                gam[0] += t.x;
                gam[1] += t.y;
                gam[2] += t.z;
                gam[3] += t.w;
            };
#pragma unroll 1
            for (int w = 0; w < 2 * warp; ++w) add_total(w);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[half][e] = gam[e];
                add_total(2 * warp + half);
            }
#pragma unroll 1
            for (int w = 2 * warp + 2; w < 16; ++w) add_total(w);
            oor = (-gam[0] > kRangeMax) | (-gam[1] > kRangeMax) | (-gam[2] > kRangeMax) | (-gam[3] > kRangeMax);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float2 o2[2] = {make_float2(o4[half][0], o4[half][1]), make_float2(o4[half][2], o4[half][3])};
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int r = 4 * half + rr, i = warp * 8 + r;
                    const float rk = fs[PF_RK + i], rq = fs[PF_RQ + i];
                    const float2 gr2[2] = {make_float2(g[r].x, g[r].y), make_float2(g[r].z, g[r].w)};
                    const float2 kv2[2] = {make_float2(bf16lo(k[r].x), bf16hi(k[r].x)),
                                           make_float2(bf16lo(k[r].y), bf16hi(k[r].y))};
                    const float2 qv2[2] = {make_float2(bf16lo(q[r].x), bf16hi(q[r].x)),
                                           make_float2(bf16lo(q[r].y), bf16hi(q[r].y))};
                    const float2 rk2 = make_float2(rk, rk), nrk2 = make_float2(-rk, -rk), rq2 = make_float2(rq, rq);
                    float2 km[2], kd[2], qd[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        o2[e] = __fadd2_rn(o2[e], gr2[e]);  // inclusive cumulative decay G of token i
                        const float2 em = make_float2(__expf(-o2[e].x), __expf(-o2[e].y));
                        km[e] = __fmul2_rn(__fmul2_rn(kv2[e], rk2), em);
                        const float2 eG = make_float2(__expf(o2[e].x), __expf(o2[e].y));
                        kd[e] = __fmul2_rn(__fmul2_rn(kv2[e], nrk2), eG);  // -k^ exp(G)
                        qd[e] = __fmul2_rn(__fmul2_rn(qv2[e], rq2), eG);
                    }
                    const uint32_t off = sw128_off(i, l4, 128);
                    uint32_t h0, lo0, h1, lo1;
                    split2(kd[0].x, kd[0].y, h0, lo0);
                    split2(kd[1].x, kd[1].y, h1, lo1);
                    st_shared_v2(sb + P_KQH + off, h0, h1);
                    st_shared_v2(sb + P_KQL + off, lo0, lo1);
                    split2(qd[0].x, qd[0].y, h0, lo0);
                    split2(qd[1].x, qd[1].y, h1, lo1);
                    st_shared_v2(sb + P_KQH + off + 8192, h0, h1);
                    st_shared_v2(sb + P_KQL + off + 8192, lo0, lo1);
                    split2(km[0].x, km[0].y, h0, lo0);
                    split2(km[1].x, km[1].y, h1, lo1);
                    st_shared_v2(sb + P_KM + off, h0, h1);
                    st_shared_v2(sb + P_KM + off + 8192, lo0, lo1);
                }
            }
        }
        fence_async_smem();
        fence_before_sync();
        if (tid == 0) *next_idx = choose_item(a, cur.idx + step, step, n_items);
        const int fallback = __syncthreads_or(oor);

        // ---- gram [-Kd;Qd] [Km_hi;Km_lo]^T (+ lo x hi) on the tensor cores
        if (tid == 0) {
            fence_after_sync();
            if (!fallback) {
                const uint32_t id128 = idesc_bf16(128, 128, false, false);
                const uint32_t id64 = idesc_bf16(128, 64, false, false);
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // [-Kd;Qd]_hi x [Km_hi;Km_lo]^T
                    const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_ss(tb, sdesc_at(sb16, P_KQH + koff, 16, 1024), sdesc_at(sb16, P_KM + koff, 16, 1024), id128,
                           s ? 1u : 0u);
                }
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // [-Kd;Qd]_lo x Km_hi^T into the first half
                    const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_ss(tb, sdesc_at(sb16, P_KQL + koff, 16, 1024), sdesc_at(sb16, P_KM + koff, 16, 1024), id64, 1u);
                }
            }
            mma_commit(gram_bar);  // an empty commit on fallback chunks
        }
        __syncwarp();
        // the next item's q, k and beta while the gram runs
        const Item nxt = next_item(p, *next_idx, step, n_items);
        load_item<GL>(p, nxt, q, k, beta_r, warp, lane);
        if (!mbar_wait(gram_bar, par, kPolls)) failed = 1;
        fence_after_sync();

        if (!fallback) {
            if (tid == 0 && nxt.idx < n_items && !failed) {  // the gram has read Km
                issue_g(nxt);
                ++g_issued;
            }
            // gram pass: row m of the accumulator (lane m), columns j0..j0+31 of both halves
            const int m = (warp & 3) * 32 + lane, j0 = (warp >> 2) * 32;
            uint32_t r1[32], r2[32];
            {
                uint32_t t[16];
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    tmem_ld16(tb + lane_off + j0 + hb * 16, t);
#pragma unroll
                    for (int e = 0; e < 16; ++e) r1[hb * 16 + e] = t[e];
                    tmem_ld16(tb + lane_off + 64 + j0 + hb * 16, t);
#pragma unroll
                    for (int e = 0; e < 16; ++e) r2[hb * 16 + e] = t[e];
                }
                tmem_wait_ld();
            }
            if (m < 64) {
                const int i = m;
                const float b = -fs[PF_BETA + i];  // gram rows hold -Kd Km^T
                float4 *dst = reinterpret_cast<float4 *>(Asm + i * AP + j0);
                const float2 b2 = make_float2(b, b);
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const float2 v = __fmul2_rn(
                            b2, __fadd2_rn(make_float2(__uint_as_float(r1[c + e]), __uint_as_float(r1[c + e + 1])),
                                           make_float2(__uint_as_float(r2[c + e]), __uint_as_float(r2[c + e + 1]))));
                        x[e] = (j0 + c + e < i) ? v.x : 0.f;
                        x[e + 1] = (j0 + c + e + 1 < i) ? v.y : 0.f;
                    }
                    dst[c / 4] = make_float4(x[0], x[1], x[2], x[3]);
                }
            } else {
                const int i = m - 64;
                float x[32];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float2 v = __fadd2_rn(make_float2(__uint_as_float(r1[c]), __uint_as_float(r1[c + 1])),
                                                make_float2(__uint_as_float(r2[c]), __uint_as_float(r2[c + 1])));
                    x[c] = (j0 + c <= i) ? v.x : 0.f;
                    x[c + 1] = (j0 + c + 1 <= i) ? v.y : 0.f;
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) st_tile8(sb + P_PIMG, sb + P_PIMG + 8192, 64, i, j0 + c8 * 8, x + c8 * 8);
            }
        } else {
            // exact grams with pairwise exponentials (the decay range is too wide for Km)
            float *Gs = reinterpret_cast<float *>(sm + P_FB_G);
            float *Pf = Tsm;  // P in fp32, converted to the image below
            const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(p.q);
            const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(p.k);
            const int t0 = cur.bos + cur.c * C;
            if (tid < DK) {  // G for every token and channel, from the inputs again
                float acc = 0.f;
                for (int i = 0; i < C; ++i) {
                    if (i < cn) acc += load_g(p, ((size_t)(t0 + i) * H + h) * DK + tid, h, tid);
                    Gs[i * 128 + tid] = acc;
                }
            }
            __syncthreads();
            for (int i = warp; i < C; i += kPT / 32) {
                const size_t ri = ((size_t)(t0 + i) * H + h) * DK;
                float qi[4], ki[4], gi[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int ch = lane + 32 * c;
                    qi[c] = i < cn ? __bfloat162float(qg[ri + ch]) : 0.f;
                    ki[c] = i < cn ? __bfloat162float(kg[ri + ch]) : 0.f;
                    gi[c] = Gs[i * 128 + ch];
                }
                for (int j = 0; j <= i; ++j) {
                    const size_t rj = ((size_t)(t0 + j) * H + h) * DK;
                    float av = 0.f, bv = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int ch = lane + 32 * c;
                        const float kj = (j < cn ? __bfloat162float(kg[rj + ch]) : 0.f) * __expf(gi[c] - Gs[j * 128 + ch]);
                        av = fmaf(ki[c], kj, av);
                        bv = fmaf(qi[c], kj, bv);
                    }
                    av = warp_sum(av) * fs[PF_RK + i] * fs[PF_RK + j];
                    bv = warp_sum(bv) * fs[PF_RQ + i] * fs[PF_RK + j];
                    if (lane == 0) {
                        Asm[i * AP + j] = (j < i) ? fs[PF_BETA + i] * av : 0.f;
                        Pf[i * AP + j] = bv;
                    }
                }
                if (lane == 0)
                    for (int j = i + 1; j < C; ++j) {
                        Asm[i * AP + j] = 0.f;
                        Pf[i * AP + j] = 0.f;
                    }
            }
            __syncthreads();
            for (int b = tid; b < 512; b += kPT) {  // P image, 8 columns per step
                const int i = b >> 3, j0 = (b & 7) * 8;
                float x[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) x[c] = Pf[i * AP + j0 + c];
                st_tile8(sb + P_PIMG, sb + P_PIMG + 8192, 64, i, j0, x);
            }
            __syncthreads();  // G scratch read: the Km tile takes the next g tile
            if (tid == 0 && nxt.idx < n_items && !failed) {
                issue_g(nxt);
                ++g_issued;
            }
        }
        __syncthreads();

        // ---- T = (I + A)^-1: 16 x 16 diagonal inverses (warps 6-7), then the off-diagonal
        // blocks from Y_IK = T_II A_IK (kept in A's unused upper blocks) in three phases of
        // independent K = 16 products, one product per warp:
        //   T_IJ = -sum_{K=J}^{I-1} Y_IK T_KJ   (block row I of (I + A) T = I)
        if (tid >= kPT - 64) {
            const int t = tid - (kPT - 64), b = t >> 4, c = t & 15, o = 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float av[16];
#pragma unroll
                for (int j4 = 0; j4 < i; j4 += 4) {  // row i of the block, 16 B at a time
                    const float4 v = *reinterpret_cast<const float4 *>(Asm + (o + i) * AP + o + j4);
                    av[j4] = v.x; av[j4 + 1] = v.y; av[j4 + 2] = v.z; av[j4 + 3] = v.w;
                }
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) acc = fmaf(av[j], x[j], acc);
                x[i] = (i < c) ? 0.f : (i == c ? 1.f : -acc);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tsm[(o + i) * AP + o + c] = x[i];
        }
        __syncthreads();
        {
            auto Ab = [&](int i, int j) { return Asm + 16 * i * AP + 16 * j; };
            auto Tb = [&](int i, int j) { return Tsm + 16 * i * AP + 16 * j; };
            auto Yb = [&](int i, int j) { return Asm + 16 * j * AP + 16 * i; };  // upper block (j, i) of A
            // (I, J) of the six blocks below the diagonal: (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
            const int w = warp;
            const int I6 = w < 3 ? w + 1 : (w == 3 ? 2 : 3), J6 = w < 3 ? w : (w == 4 ? 1 : 0);
            if (w < 6) blk16w(Yb(I6, J6), Tb(I6, I6), Ab(I6, J6), 1.f, false, lane);  // every Y_IJ
            __syncthreads();
            if (w < 6) blk16w(Tb(I6, J6), Yb(I6, J6), Tb(J6, J6), -1.f, false, lane);
            __syncthreads();
            if (w < 3) {  // (I, J, K) = (2,0,1) (3,1,2) (3,0,1)
                const int I = w == 0 ? 2 : 3, J = w == 1 ? 1 : 0, K = w == 1 ? 2 : 1;
                blk16w(Tb(I, J), Yb(I, K), Tb(K, J), -1.f, true, lane);
            }
            __syncthreads();
            if (w == 0) blk16w(Tb(3, 0), Yb(3, 2), Tb(2, 0), -1.f, true, lane);  // T30 -= Y32 T20
            __syncthreads();
        }
        // ---- T diag(beta) image (hi, then lo) over the dead A buffer: every block of 8
        // columns, zero above the diagonal
        for (int b = tid; b < 512; b += kPT) {
            const int i = b >> 3, j0 = (b & 7) * 8;
            float x[8];
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
                const float2 v = __fmul2_rn(make_float2(Tsm[i * AP + j0 + c], Tsm[i * AP + j0 + c + 1]),
                                            make_float2(fs[PF_BETA + j0 + c], fs[PF_BETA + j0 + c + 1]));
                x[c] = (j0 + c <= i) ? v.x : 0.f;
                x[c + 1] = (j0 + c + 1 <= i) ? v.y : 0.f;
            }
            st_tile8(sb + P_A, sb + P_A + 8192, 64, i, j0, x);
        }
        fence_async_smem();
        if (__syncthreads_or(failed)) break;
        if (tid == 0) {  // the blob: T diag(beta) hi/lo, then P hi/lo
            bulk_store(blob, sb + P_A, 16384);
            bulk_store(blob + 16384, sb + P_PIMG, 16384);
            bulk_commit();
            stores_pending = true;
            flag_pending = (int64_t)blob_slot(cur.bos, cur.n, cur.c) * H + h;
        }
        cur = nxt;
        ++n_done;
    }

    if (tid == 0 && stores_pending) {  // (issued after the CTA's last failure check passed)
        bulk_wait_all();
        if (a.flags) publish();
    }
    if (__syncthreads_or(failed)) {
        // drain what is in flight, then poison the blobs of this item and of every later item
        // of this CTA: NaN there reaches o, y and the state through the chain kernel
        if (tid == 0) {
            atomicAdd(&g_chunk_prep_timeouts, 1);
            mma_commit(drain_bar);
            if (g_issued > g_seen) mbar_wait(g_bar, g_seen & 1, kPolls);  // at most one tile in flight
        }
        __syncthreads();
        mbar_wait(drain_bar, 0, kPolls);
        for (Item it = cur; it.idx < n_items; it = next_item(p, it.idx + step, step, n_items)) {
            uint4 *b = reinterpret_cast<uint4 *>(a.ws + ((size_t)blob_slot(it.bos, it.n, it.c) * H + it.h) * kBlobBytes);
            for (int e = tid; e < (int)(kBlobBytes / 16); e += kPT) b[e] = make_uint4(~0u, ~0u, ~0u, ~0u);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 128);
}

}  // namespace

int take_chunk_prep_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_chunk_prep_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_chunk_prep_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("chunk_prep: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

size_t chunk_workspace_bytes(int64_t rows, int N, int H) { return WorkspaceLayout(rows, N, H).bytes; }

kda_status configure_chunk_prep() {
    static DeviceOnce configured;
    const int dev = current_device();
    if (configured.done(dev)) return KDA_OK;
    for (void *fn : {(void *)chunk_prep_kernel<false>, (void *)chunk_prep_kernel<true>}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, PREP_SMEM);
        if (e != cudaSuccess) {
            set_error("chunk_prep: cannot reserve %u bytes of shared memory: %s", PREP_SMEM, cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
    }
    configured.set(dev);
    return KDA_OK;
}

kda_status launch_chunk_prep(const SeqParams &p, void *ws, cudaStream_t st, const PrepConcurrent *cc) {
    const int64_t rows = p.cu_seqlens ? (int64_t)p.T : (int64_t)p.N * p.T;
    const int64_t n_slots = blob_slots(rows, p.N);
    const int64_t n_items = n_slots * p.H;
    if (rows <= 0 || n_items == 0) return KDA_OK;
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) {
        set_error("chunk_prep: cuTensorMapEncodeTiled is not available from the driver");
        return KDA_ERR_CUDA;
    }
    CUtensorMap tmap_g;
    const bool gb = p.g_logits && p.g_logits_bf16;
    const cuuint64_t es = gb ? 2 : 4;
    const void *gsrc = p.g_logits ? p.g_logits : (const void *)p.g;
    const cuuint64_t gdims[3] = {(cuuint64_t)DK, (cuuint64_t)p.H, (cuuint64_t)rows};
    const cuuint64_t gstrides[2] = {(cuuint64_t)DK * es, (cuuint64_t)p.H * DK * es};
    const cuuint32_t gbox[3] = {(cuuint32_t)DK, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult cres = enc(&tmap_g, gb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                              const_cast<void *>(gsrc), gdims, gstrides, gbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cres != CUDA_SUCCESS) {
        set_error("chunk_prep: cuTensorMapEncodeTiled failed for g (%d)", (int)cres);
        return KDA_ERR_CUDA;
    }
    const kda_status cs = configure_chunk_prep();
    if (cs != KDA_OK) return cs;
    PrepArgs a;
    memset(&a, 0, sizeof(a));
    a.p = p;
    a.ws = static_cast<uint8_t *>(ws);
    a.n_slots = n_slots;
    if (cc) {
        const WorkspaceLayout L(rows, p.N, p.H);
        a.flags = reinterpret_cast<uint32_t *>(a.ws + L.flags);
        a.progress = reinterpret_cast<const uint32_t *>(a.ws + L.progress);
        a.lead = cc->lead;
    }
    const int64_t cap = cc ? (int64_t)cc->grid : 2 * (int64_t)sm_count();
    const int grid = (int)(n_items < cap ? n_items : cap);
    if (p.g_logits)
        chunk_prep_kernel<true><<<grid, kPT, PREP_SMEM, st>>>(tmap_g, a);
    else
        chunk_prep_kernel<false><<<grid, kPT, PREP_SMEM, st>>>(tmap_g, a);
    note_launch();
    return check_launch("chunk_prep_kernel");
}

}  // namespace kda
