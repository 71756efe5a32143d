// kda_chunk_chain.cu -- the state-dependent half of the split chunked prefill: one CTA per
// (sequence, head) carries the state through the prompt's chunks on the tensor cores.
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (a prompt runs a
// chunked kernel that carries the state from one 64-token chunk to the next and never
// holds it per token), sections 03/04 (per-key-channel decay applied before each
// delta-rule update, q and k L2-normalised in the kernel, q scaled by 1/sqrt(key_dim));
// Kimi-K3 atlas "gate-project (decode, P = 1000)" for the fused sigmoid-gated RMSNorm.
//
// The pre-pass (kda_chunk_prep.cu) has already formed, for every chunk, T diag(beta) and P
// (kda_chunk_common.cuh has the algebra) and left them as operand images in the workspace.
// What stays on the serial chain from one chunk to the next is
//   [R | O]^T = [V^T I | 0] + S^T [-Kd ; Qd]^T,   D^T = R^T (T diag beta)^T,
//   [O | S]^T += D^T [P^T | Kg]  (S^T decayed by exp(gamma) first)
// with S^T in TMEM (fp32 accumulator and a split-bf16 copy as the A operand), the value
// dimension as the MMA M dimension, and every operand split into bf16 hi + lo (three
// products hi*hi + hi*lo + lo*hi; V enters through an exact bf16 identity).  The TMEM
// columns and the three MMA groups are the fused kernel's (kda_chunk_tc.cu); the gram,
// the triangular solve and their operand tiles are gone from the chain, and so is the
// exact fallback: Kd, Qd and Kg take non-positive exponents only (a channel whose decay
// range exceeds kRangeMax forms Kg from exp(gamma - G) directly).
//
// Per chunk, beside the tensor core (all 16 warps; thread 0 issues the MMAs and copies):
//   R/O product   the chunk's Kg^T rows are stored, the next chunk's q, k, beta loaded
//   R pass        R^T -> hi/lo in place; the next chunk's V tile is requested
//   D product     the next chunk's norms, beta and decay totals (its g tile arrived by TMA)
//   D pass        D^T -> hi/lo in place, S^T decayed; the next T diag(beta) image requested
//   O/S product   the next chunk's decay prefix and its [-Kd ; Qd] tiles and Kg
//   O/S pass      O out (+ gated norm), S^T -> hi/lo; the next P image requested
// Every wait is bounded; a CTA whose wait gives up writes NaN into its final state, o and y.
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

constexpr int kThreads = 512;  // 16 warps = 4 warpgroups

// TMEM columns (the fused kernel's, with the gram's columns holding D)
constexpr uint32_t T_R = 0, T_O = 64, T_S = 128, T_SH = 256, T_SL = 320, T_D = 384;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_V = 0;          // V tile, two TMA boxes of 64 tokens x 64 values (16 KB)
constexpr uint32_t S_KQH = 16384;    // [-Kd ; Qd] hi, 128 rows x 128 (32 KB)
constexpr uint32_t S_KQL = 49152;    // [-Kd ; Qd] lo
constexpr uint32_t S_GT = 81920;     // the next chunk's g (or logits) tile, 64 tokens x 128 (32 KB)
constexpr uint32_t S_PKGH = 114688;  // [P ; Kg^T] hi, 192 rows (i, then c) x 64 (j) (24 KB), K-major B
constexpr uint32_t S_PKGL = 139264;  // [P ; Kg^T] lo
constexpr uint32_t S_TBH = 163840;   // T diag(beta) hi, 64 x 64 (8 KB); lo follows at S_TBH + 8 KB
constexpr uint32_t S_ID = 180224;    // bf16 identity 64 x 64 (8 KB)
constexpr uint32_t S_GATE = 188416;  // fused norm: the chunk's bf16 gate tile, 64 tokens x 128 (16 KB)
constexpr uint32_t S_SCAN = 204800;  // decay totals [16][128], their exclusive prefix [16][128], total [128]
constexpr uint32_t S_SMALL = S_SCAN + 33 * 128 * 4;
// small buffers (floats)
constexpr uint32_t F_BETA = 0;    // beta [64]
constexpr uint32_t F_RQ = 64;     // q scale per token (norm * scale) [64]
constexpr uint32_t F_RK = 128;    // k norm per token [64]
constexpr uint32_t F_GEXP = 192;  // exp(gamma) [128]
constexpr uint32_t F_RED = 320;   // norm partials [4 wg][4 quarters][16]
constexpr uint32_t F_AH = 576;    // gates from logits: exp(A_log) of the head [1 of 4]
constexpr uint32_t F_DB = 580;    // gates from logits: dt_bias of the head's channels [128]
constexpr uint32_t F_END = 708;
constexpr uint32_t S_BARS = S_SMALL + F_END * 4;     // 10 mbarriers + tmem slot
constexpr uint32_t SMEM_BYTES = S_BARS + 96 + 1024;  // + alignment slack

static_assert(S_SMALL % 16 == 0 && S_BARS % 8 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Set by a CTA whose bounded wait on the tensor core or a copy gave up; that CTA also
// writes NaN into its final state, o and y so the failure cannot pass unnoticed.
__device__ int g_chunk_chain_timeouts = 0;

struct ChainParams {
    SeqParams p;
    const uint8_t *ws;  // the pre-pass's blobs
    int order_n;        // > 0: blockIdx -> sequence through order[]
    int order[64];
};

// One chunk's q and k for this thread's 4 tokens x 4 key channels and beta (or its
// logit's raw bits) of token 4 warp + lane for lanes 0-3.  Nothing here waits for the
// data: rows past the chunk's end read its last row and are zeroed when the chunk is
// prepared.
struct ChunkRegs {
    float4 g[4];  // g, or its raw logits (fp32, or bf16 bits in .x/.y) until the chunk is prepared
    uint2 q[4], k[4];
    float beta;
};

template <bool GL>
__device__ __forceinline__ void load_chunk(const SeqParams &p, ChunkRegs &cr, int bos, int t0, int cn, int h,
                                           int warp, int l4) {
    if (cn <= 0) return;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = min(warp * 4 + r, cn - 1);
        const size_t hk = ((size_t)(bos + t0 + i) * p.H + h) * DK + l4;
        cr.q[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) + hk));
        cr.k[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.k) + hk));
    }
    const size_t bi = (size_t)(bos + t0 + min(warp * 4 + ((l4 >> 2) & 3), cn - 1)) * p.H + h;
    if (!GL) {
        cr.beta = __ldg(p.beta + bi);
    } else {
        uint32_t raw;
        if (p.beta_logits_bf16)
            asm("ld.global.nc.u16 %0, [%1];" : "=r"(raw) : "l"(reinterpret_cast<const uint16_t *>(p.beta_logits) + bi));
        else
            asm("ld.global.nc.u32 %0, [%1];" : "=r"(raw) : "l"(reinterpret_cast<const uint32_t *>(p.beta_logits) + bi));
        cr.beta = __uint_as_float(raw);
    }
}

// barrier over warps 1-15 (warp 0 is issuing tensor-core work)
__device__ __forceinline__ void tbar() { asm volatile("bar.sync 1, 480;" ::: "memory"); }

// GL: g and beta come from their logits.  NORM: the output goes through the fused
// sigmoid-gated RMSNorm.  Both are compile-time choices.
template <bool GL, bool NORM>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_chain_kernel(const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_g,
                       const __grid_constant__ CUtensorMap tmap_gate, const __grid_constant__ ChainParams cp) {
    const SeqParams &p = cp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb16 = sb >> 4;
    float *fs = reinterpret_cast<float *>(sm + S_SMALL);
    // one barrier per tensor-core group or copy, each completing exactly once per chunk
    uint64_t *bar_r = reinterpret_cast<uint64_t *>(sm + S_BARS);  // R and O
    uint64_t *bar_d = bar_r + 1;                                    // D
    uint64_t *bar_s = bar_r + 2;                                    // O and S updates
    uint64_t *v_bar = bar_r + 3;                                    // V tile
    uint64_t *g_bar = bar_r + 4;                                    // g tile
    uint64_t *tb_bar = bar_r + 5;                                   // T diag(beta) image
    uint64_t *p_bar = bar_r + 6;                                    // P image
    uint64_t *gate_bar = bar_r + 7;                                 // fused norm: gate tile
    uint64_t *pre_bar = bar_r + 8;                                  // decay prefix written (128 arrivals)
    uint64_t *drain_bar = bar_r + 9;                                // drain after a failure
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_BARS + 80);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, wq = warp & 3;
    const int m = wq * 32 + lane;  // TMEM lane this thread reads/writes
    const int l4 = lane * 4;       // this thread's 4 key channels in the preparation
    const int H = p.H;
    int n = blockIdx.x / H;
    const int h = blockIdx.x % H;
    if (cp.order_n > 0) n = cp.order[n];
    const int unit = n * H + h;
    int bos, len;
    seq_range(p, n, bos, len);
    const int nchunks = (len + C - 1) / C;
    auto blob = [&](int chunk) { return cp.ws + ((size_t)blob_slot(bos, n, chunk) * H + h) * kBlobBytes; };

    // first chunk's inputs are in flight while the CTA sets up
    ChunkRegs cr;
    load_chunk<GL>(p, cr, bos, 0, min(C, len), h, warp, l4);

    if (tid == 0) {
        for (int b = 0; b < 10; ++b) mbar_init(bar_r + b, b == 8 ? 128 : 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    {  // bf16 identity tile (K-major, rows i, columns j)
        const int i = tid >> 3, j0 = (tid & 7) * 8;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (i >= j0 && i < j0 + 8) w[(i - j0) >> 1] = (i & 1) ? 0x3F800000u : 0x00003F80u;
        st_shared_v4(sb + S_ID + sw128_off(i, j0, 64), w[0], w[1], w[2], w[3]);
    }
    if (GL) {  // the head's gate constants, read by every chunk's conversion
        if (tid < DK) fs[F_DB + tid] = p.dt_bias ? __ldg(p.dt_bias + (size_t)h * DK + tid) : 0.f;
        if (tid == DK) fs[F_AH] = __expf(__ldg(p.A_log + h));
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;

    // copies (thread 0); each *_pending is the chunk whose copy is in flight, or -1
    int v_pending = -1, g_pending = -1, tb_pending = -1, p_pending = -1, q_pending = -1;
    auto issue_v = [&](int chunk) {
        mbar_arrive_expect_tx(v_bar, 16384);
        tma_load_3d(sb + S_V, &tmap_v, v_bar, 0, h, bos + chunk * C);
        tma_load_3d(sb + S_V + 8192, &tmap_v, v_bar, 64, h, bos + chunk * C);
        v_pending = chunk;
    };
    const uint32_t g_bytes = (GL && p.g_logits_bf16) ? C * DK * 2 : C * DK * 4;
    auto issue_g = [&](int chunk) {
        mbar_arrive_expect_tx(g_bar, g_bytes);
        tma_load_3d(sb + S_GT, &tmap_g, g_bar, 0, h, bos + chunk * C);
        g_pending = chunk;
    };
    auto issue_tb = [&](int chunk) {  // T diag(beta) hi and lo: 16 contiguous KB
        mbar_arrive_expect_tx(tb_bar, 16384);
        bulk_load(sb + S_TBH, blob(chunk), 16384, tb_bar);
        tb_pending = chunk;
    };
    auto issue_p = [&](int chunk) {  // P hi and lo into rows 0-63 of the [P ; Kg^T] tiles
        mbar_arrive_expect_tx(p_bar, 16384);
        bulk_load(sb + S_PKGH, blob(chunk) + 16384, 8192, p_bar);
        bulk_load(sb + S_PKGL, blob(chunk) + 24576, 8192, p_bar);
        p_pending = chunk;
    };
    int failed = 0;  // a bounded wait gave up
    if (tid == 0 && nchunks > 0) {
        issue_v(0);
        issue_g(0);
        issue_tb(0);
        issue_p(0);
    }

    {  // initial state -> S^T accumulator and its hi/lo copy; O^T = 0
        const int c0 = wg * 32;
        float s[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = p.s0 ? p.s0[((size_t)unit * DK + c0 + c) * DV + m] : 0.f;
        uint32_t r[16], hi[16], lo[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int c = 0; c < 16; ++c) r[c] = __float_as_uint(s[half * 16 + c]);
            tmem_st16(tb + lane_off + T_S + c0 + half * 16, r);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            split2(s[2 * c], s[2 * c + 1], hi[c], lo[c]);
            r[c] = 0u;
        }
        tmem_st16(tb + lane_off + T_SH + c0 / 2, hi);
        tmem_st16(tb + lane_off + T_SL + c0 / 2, lo);
        tmem_st16(tb + lane_off + T_O + wg * 16, r);
        tmem_wait_st();
    }

    auto wait_bar = [&](uint64_t *bar, int parity) {
        const bool ok = mbar_wait(bar, (uint32_t)parity, kPolls);
        fence_after_sync();
        return ok;
    };

    float *scan = reinterpret_cast<float *>(sm + S_SCAN);
    float *pre = scan + 16 * 128;

    // ---- preparation of a chunk, first half: per-token norm scales and beta into the
    // small buffers, each warp's decay totals per key channel into the scan buffer.  The 8
    // sums of squares of a warp's 4 tokens are reduced with a reduce-scatter (9 shuffles);
    // lanes 4v..4v+3 end with sum v (q of tokens 0-3, then k).
    auto prep_norms = [&](ChunkRegs &c, int cnn, int chunk) {
        if (!mbar_wait(g_bar, (uint32_t)(chunk & 1), kPolls))
            failed = 1;
        else if (tid == 0)
            g_pending = -1;
#pragma unroll
        for (int r = 0; r < 4; ++r)  // tokens past the chunk's end: q = k = 0 (loaded as a copy)
            if (warp * 4 + r >= cnn) {
                c.q[r] = make_uint2(0u, 0u);
                c.k[r] = make_uint2(0u, 0u);
            }
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // tokens past the chunk's end read as g = 0
            const int i = warp * 4 + r;
            if (GL && p.g_logits_bf16) {
                const uint2 u = *reinterpret_cast<const uint2 *>(sm + S_GT + (i * DK + l4) * 2);
                c.g[r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), 0.f, 0.f);
            } else {
                c.g[r] = *reinterpret_cast<const float4 *>(sm + S_GT + (i * DK + l4) * 4);
            }
            if (!GL && i >= cnn) c.g[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (GL) {  // g from its logits; tokens past the chunk's end keep g = 0
            const float a_h = fs[F_AH];
            const float4 db = *reinterpret_cast<const float4 *>(fs + F_DB + l4);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float z[4];
                if (p.g_logits_bf16) {
                    const uint32_t ux = __float_as_uint(c.g[r].x), uy = __float_as_uint(c.g[r].y);
                    z[0] = bf16lo(ux); z[1] = bf16hi(ux); z[2] = bf16lo(uy); z[3] = bf16hi(uy);
                } else {
                    z[0] = c.g[r].x; z[1] = c.g[r].y; z[2] = c.g[r].z; z[3] = c.g[r].w;
                }
                const bool live = warp * 4 + r < cnn;
                c.g[r] = make_float4(live ? gate_of_logit(z[0] + db.x, a_h, p.g_lower) : 0.f,
                                     live ? gate_of_logit(z[1] + db.y, a_h, p.g_lower) : 0.f,
                                     live ? gate_of_logit(z[2] + db.z, a_h, p.g_lower) : 0.f,
                                     live ? gate_of_logit(z[3] + db.w, a_h, p.g_lower) : 0.f);
            }
            if (lane < 4) {
                const uint32_t raw = __float_as_uint(c.beta);
                c.beta = warp * 4 + lane < cnn ? beta_of_logit(__uint_as_float(p.beta_logits_bf16 ? raw << 16 : raw))
                                               : 0.f;
            }
        }
        if (!GL && warp * 4 + lane >= cnn) c.beta = 0.f;
        float a[8];
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // (q, k) sums of squares as packed pairs
            const float2 v0 = make_float2(bf16lo(c.q[r].x), bf16lo(c.k[r].x));
            const float2 v1 = make_float2(bf16hi(c.q[r].x), bf16hi(c.k[r].x));
            const float2 v2 = make_float2(bf16lo(c.q[r].y), bf16lo(c.k[r].y));
            const float2 v3 = make_float2(bf16hi(c.q[r].y), bf16hi(c.k[r].y));
            const float2 ss = __ffma2_rn(v0, v0, __ffma2_rn(v1, v1, __ffma2_rn(v2, v2, __fmul2_rn(v3, v3))));
            a[r] = ss.x;
            a[4 + r] = ss.y;
        }
        const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
        float b[4], d2[2];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b[j] = (u16 ? a[j + 4] : a[j]) + __shfl_xor_sync(0xffffffffu, u16 ? a[j] : a[j + 4], 16);
#pragma unroll
        for (int j = 0; j < 2; ++j)
            d2[j] = (u8 ? b[j + 2] : b[j]) + __shfl_xor_sync(0xffffffffu, u8 ? b[j] : b[j + 2], 8);
        float d = (u4 ? d2[1] : d2[0]) + __shfl_xor_sync(0xffffffffu, u4 ? d2[0] : d2[1], 4);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if ((lane & 3) == 0) {
            const int v = lane >> 2;
            const float sc = p.l2norm ? rsqrtf(d + 1e-6f) : 1.f;
            if (v < 4)
                fs[F_RQ + warp * 4 + v] = sc * p.scale;
            else
                fs[F_RK + warp * 4 + v - 4] = sc;
        }
        if (lane < 4) fs[F_BETA + warp * 4 + lane] = c.beta;
        float2 t01 = make_float2(c.g[0].x, c.g[0].y), t23 = make_float2(c.g[0].z, c.g[0].w);
#pragma unroll
        for (int r = 1; r < 4; ++r) {
            t01 = __fadd2_rn(t01, make_float2(c.g[r].x, c.g[r].y));
            t23 = __fadd2_rn(t23, make_float2(c.g[r].z, c.g[r].w));
        }
        *reinterpret_cast<float4 *>(scan + warp * 128 + l4) = make_float4(t01.x, t01.y, t23.x, t23.y);
    };

    // ---- exclusive prefix of the warps' decay totals per key channel, and the chunk total
    // (row 16), by warps 1-4; then a barrier of warps 1-15 (warp 0 is issuing and reads the
    // prefix after the mbarrier the 128 writers arrive on)
    auto scan_prefix = [&]() {
        if (warp >= 1 && warp <= 4) {
            const int c = tid - 32;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float t = scan[w * 128 + c];
                pre[w * 128 + c] = acc;
                acc += t;
            }
            pre[16 * 128 + c] = acc;
            mbar_arrive(pre_bar);
        }
        tbar();
    };

    // ---- preparation, second half: cumulative decay, exp(gamma) and the [-Kd ; Qd] tiles
    // of the chunk; Kg is returned in registers because its tile may still be in use.
    // With use_pre the prefix comes from scan_prefix, otherwise (first chunk) each thread
    // sums the warps' totals itself, in the same order.
    auto prep_tiles = [&](const ChunkRegs &c, float (&kgv)[4][4], bool use_pre) {
        float o4[4] = {0.f, 0.f, 0.f, 0.f}, gam[4] = {0.f, 0.f, 0.f, 0.f};
        if (use_pre) {
            const float4 t = *reinterpret_cast<const float4 *>(pre + warp * 128 + l4);
            const float4 u = *reinterpret_cast<const float4 *>(pre + 16 * 128 + l4);
            o4[0] = t.x; o4[1] = t.y; o4[2] = t.z; o4[3] = t.w;
            gam[0] = u.x; gam[1] = u.y; gam[2] = u.z; gam[3] = u.w;
        } else {
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float4 t = *reinterpret_cast<const float4 *>(scan + w * 128 + l4);
                const float tt[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (w < warp) o4[e] += tt[e];
                    gam[e] += tt[e];
                }
            }
        }
        float egam[4];
        bool wide[4];  // the channel's decay range is too wide for exp(-G) exp(gamma)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            egam[e] = __expf(gam[e]);
            wide[e] = -gam[e] > kRangeMax;
        }
        if (warp == 1) *reinterpret_cast<float4 *>(fs + F_GEXP + l4) = make_float4(egam[0], egam[1], egam[2], egam[3]);
        const float4 rq4 = *reinterpret_cast<const float4 *>(fs + F_RQ + warp * 4);
        const float4 rk4 = *reinterpret_cast<const float4 *>(fs + F_RK + warp * 4);
        const float rq[4] = {rq4.x, rq4.y, rq4.z, rq4.w}, rk[4] = {rk4.x, rk4.y, rk4.z, rk4.w};
        float2 o2[2] = {make_float2(o4[0], o4[1]), make_float2(o4[2], o4[3])};
        const float2 eg2[2] = {make_float2(egam[0], egam[1]), make_float2(egam[2], egam[3])};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = warp * 4 + r;
            const float2 gr2[2] = {make_float2(c.g[r].x, c.g[r].y), make_float2(c.g[r].z, c.g[r].w)};
            const float2 kv2[2] = {make_float2(bf16lo(c.k[r].x), bf16hi(c.k[r].x)),
                                   make_float2(bf16lo(c.k[r].y), bf16hi(c.k[r].y))};
            const float2 qv2[2] = {make_float2(bf16lo(c.q[r].x), bf16hi(c.q[r].x)),
                                   make_float2(bf16lo(c.q[r].y), bf16hi(c.q[r].y))};
            const float2 rk2 = make_float2(rk[r], rk[r]), nrk2 = make_float2(-rk[r], -rk[r]);
            const float2 rq2 = make_float2(rq[r], rq[r]);
            float2 kd[2], qd[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                o2[e] = __fadd2_rn(o2[e], gr2[e]);  // inclusive cumulative decay G of token i
                const float2 em = make_float2(__expf(-o2[e].x), __expf(-o2[e].y));
                const float2 km = __fmul2_rn(__fmul2_rn(kv2[e], rk2), em);
                const float2 kg = __fmul2_rn(km, eg2[e]);
                kgv[r][2 * e] = wide[2 * e] ? kv2[e].x * rk[r] * __expf(gam[2 * e] - o2[e].x) : kg.x;
                kgv[r][2 * e + 1] = wide[2 * e + 1] ? kv2[e].y * rk[r] * __expf(gam[2 * e + 1] - o2[e].y) : kg.y;
                const float2 eG = make_float2(__expf(o2[e].x), __expf(o2[e].y));
                kd[e] = __fmul2_rn(__fmul2_rn(kv2[e], nrk2), eG);  // -k^ exp(G)
                qd[e] = __fmul2_rn(__fmul2_rn(qv2[e], rq2), eG);
            }
            const uint32_t off = sw128_off(i, l4, 128);  // rows i and 64 + i share the swizzle phase
            uint32_t h0, lo0, h1, lo1;
            split2(kd[0].x, kd[0].y, h0, lo0);
            split2(kd[1].x, kd[1].y, h1, lo1);
            st_shared_v2(sb + S_KQH + off, h0, h1);
            st_shared_v2(sb + S_KQL + off, lo0, lo1);
            split2(qd[0].x, qd[0].y, h0, lo0);
            split2(qd[1].x, qd[1].y, h1, lo1);
            st_shared_v2(sb + S_KQH + off + 8192, h0, h1);
            st_shared_v2(sb + S_KQL + off + 8192, lo0, lo1);
        }
    };

    // ---- first chunk's preparation (later chunks are prepared inside the previous
    // chunk's tensor-core waits)
    float kgv[4][4];  // the chunk's Kg, stored when its [P ; Kg^T] tile is free
    if (nchunks > 0) {
        prep_norms(cr, min(C, len), 0);
        __syncthreads();
        if (tid == 0 && nchunks > 1 && !failed) issue_g(1);  // every thread has read g(0)
        prep_tiles(cr, kgv, false);
    }

    for (int ch = 0; ch < nchunks; ++ch) {
        const int par = ch & 1;
        const int t0 = ch * C;
        const int cn = min(C, len - t0);
        const int cn_next = min(C, len - t0 - C);
        fence_async_smem();
        fence_before_sync();  // the previous state pass (or the initial state) wrote TMEM
        // ---- operand tiles of this chunk and S(n-1) are ready
        if (__syncthreads_or(failed)) break;

        // ================= R^T = V^T I + S^T (-Kd)^T, O^T = S^T Qd^T
        if (tid == 0) {
            fence_after_sync();
            if (mbar_wait(v_bar, (uint32_t)par, kPolls))
                v_pending = -1;
            else
                failed = 1;
            const uint32_t id_mn = idesc_bf16(128, 64, true, false);
#pragma unroll 1
            for (int s = 0; s < 4; ++s)
                mma_ss(tb + T_R, sdesc_at(sb16, S_V + s * 2048, 8192, 1024), sdesc_at(sb16, S_ID + s * 32, 16, 1024), id_mn,
                       s ? 1u : 0u);
            const uint32_t id128 = idesc_bf16(128, 128, false, false);
#pragma unroll
            for (int cb = 0; cb < 3; ++cb)
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {
                    const uint32_t a = tb + (combo_a(cb) ? T_SL : T_SH) + s * 8;
                    const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_ts(tb + T_R, a, sdesc_at(sb16, (combo_b(cb) ? S_KQL : S_KQH) + koff, 16, 1024), id128, 1u);
                }
            mma_commit(bar_r);
            // fused norm, bf16 gate: this chunk's gate tile, read by the O pass (the previous
            // O pass has finished with the buffer)
            if (NORM && p.gate_bf16) {
                mbar_arrive_expect_tx(gate_bar, C * DV * 2);
                tma_load_3d(sb + S_GATE, &tmap_gate, gate_bar, 0, h, bos + t0);
                q_pending = ch;
            }
        }
        __syncwarp();
        // this chunk's Kg^T rows (the previous O/S product has read the old ones)
        st_kgt(sb + S_PKGH, sb + S_PKGL, l4, warp * 4, kgv);
        fence_async_smem();
        if (ch + 1 < nchunks) load_chunk<GL>(p, cr, bos, t0 + C, cn_next, h, warp, l4);

        // ================= R pass: R^T (lane v, column j) -> hi/lo operand in TMEM
        if (!wait_bar(bar_r, par)) failed = 1;
        if (tid == 0 && ch + 1 < nchunks && !failed) issue_v(ch + 1);  // the V tile has been read
        {
            uint32_t r[16], hi[8], lo[8];
            tmem_ld16(tb + lane_off + T_R + wg * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) split2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]), hi[c], lo[c]);
            tmem_st8(tb + lane_off + T_R + wg * 16, hi);  // in place: tokens 16 wg.. as hi, then lo
            tmem_st8(tb + lane_off + T_R + wg * 16 + 8, lo);
            tmem_wait_st();
        }
        fence_before_sync();
        // ---- R^T hi/lo are ready
        if (__syncthreads_or(failed)) break;

        // ================= D^T = R^T (T diag beta)^T
        if (tid == 0) {
            fence_after_sync();
            if (mbar_wait(tb_bar, (uint32_t)par, kPolls))
                tb_pending = -1;
            else
                failed = 1;
            // R^T_hi [T diag(beta)_hi ; _lo]^T (N = 128: the two tiles are contiguous) into
            // [D_a | D_b], then R^T_lo (T diag beta)_hi^T onto D_a
            const uint32_t id128 = idesc_bf16(128, 128, false, false), id64 = idesc_bf16(128, 64, false, false);
#pragma unroll 1
            for (int s = 0; s < 4; ++s)
                mma_ts(tb + T_D, tb + T_R + s * 16, sdesc_at(sb16, S_TBH + s * 32, 16, 1024), id128, s ? 1u : 0u);
#pragma unroll 1
            for (int s = 0; s < 4; ++s)
                mma_ts(tb + T_D, tb + T_R + s * 16 + 8, sdesc_at(sb16, S_TBH + s * 32, 16, 1024), id64, 1u);
            mma_commit(bar_d);
        }
        __syncwarp();
        // while D runs: the next chunk's norms, beta and decay totals
        if (ch + 1 < nchunks) prep_norms(cr, cn_next, ch + 1);

        // ================= D pass (hi/lo into TMEM) and S decay by exp(gamma)
        if (!wait_bar(bar_d, par)) failed = 1;
        if (tid == 0 && ch + 1 < nchunks && !failed) issue_tb(ch + 1);  // the T diag(beta) tile has been read
        {
            uint32_t r[16], s1[16], s2[16], hi[8], lo[8];
            const int c0 = wg * 32;
            {
                uint32_t rb[16];
                tmem_ld16(tb + lane_off + T_D + wg * 16, r);
                tmem_ld16(tb + lane_off + T_D + 64 + wg * 16, rb);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; c += 2) {  // D = D_a + D_b
                    const float2 v = __fadd2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])),
                                                make_float2(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])));
                    r[c] = __float_as_uint(v.x);
                    r[c + 1] = __float_as_uint(v.y);
                }
            }
            tmem_ld16(tb + lane_off + T_S + c0, s1);
            tmem_ld16(tb + lane_off + T_S + c0 + 16, s2);
#pragma unroll
            for (int c = 0; c < 8; ++c) split2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]), hi[c], lo[c]);
            tmem_st8(tb + lane_off + T_D + wg * 16, hi);  // in place: tokens 16 wg.. as hi, then lo
            tmem_st8(tb + lane_off + T_D + wg * 16 + 8, lo);
            tmem_wait_ld();
            const float4 *ge = reinterpret_cast<const float4 *>(fs + F_GEXP + c0);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const float4 a = ge[c4], b = ge[4 + c4];
                const float2 x0 = __fmul2_rn(make_float2(__uint_as_float(s1[4 * c4]), __uint_as_float(s1[4 * c4 + 1])),
                                             make_float2(a.x, a.y));
                const float2 x1 = __fmul2_rn(make_float2(__uint_as_float(s1[4 * c4 + 2]), __uint_as_float(s1[4 * c4 + 3])),
                                             make_float2(a.z, a.w));
                const float2 y0 = __fmul2_rn(make_float2(__uint_as_float(s2[4 * c4]), __uint_as_float(s2[4 * c4 + 1])),
                                             make_float2(b.x, b.y));
                const float2 y1 = __fmul2_rn(make_float2(__uint_as_float(s2[4 * c4 + 2]), __uint_as_float(s2[4 * c4 + 3])),
                                             make_float2(b.z, b.w));
                s1[4 * c4 + 0] = __float_as_uint(x0.x); s1[4 * c4 + 1] = __float_as_uint(x0.y);
                s1[4 * c4 + 2] = __float_as_uint(x1.x); s1[4 * c4 + 3] = __float_as_uint(x1.y);
                s2[4 * c4 + 0] = __float_as_uint(y0.x); s2[4 * c4 + 1] = __float_as_uint(y0.y);
                s2[4 * c4 + 2] = __float_as_uint(y1.x); s2[4 * c4 + 3] = __float_as_uint(y1.y);
            }
            tmem_st16(tb + lane_off + T_S + c0, s1);
            tmem_st16(tb + lane_off + T_S + c0 + 16, s2);
            tmem_wait_st();
            fence_before_sync();
        }
        // ---- D^T hi/lo ready, S^T decayed; every thread has read the next chunk's g tile
        if (__syncthreads_or(failed)) break;

        // ================= [O|S]^T += D^T [P^T | Kg]
        if (tid == 0) {
            fence_after_sync();
            if (mbar_wait(p_bar, (uint32_t)par, kPolls))
                p_pending = -1;
            else
                failed = 1;
            const uint32_t id192 = idesc_bf16(128, 192, false, false);
#pragma unroll
            for (int cb = 0; cb < 3; ++cb)
#pragma unroll 1
                for (int s = 0; s < 4; ++s)
                    mma_ts(tb + T_O, tb + T_D + s * 16 + (combo_a(cb) ? 8 : 0),
                           sdesc_at(sb16, (combo_b(cb) ? S_PKGL : S_PKGH) + s * 32, 16, 1024), id192, 1u);
            mma_commit(bar_s);
            if (ch + 2 < nchunks && !failed) issue_g(ch + 2);
        }
        __syncwarp();
        // while O and S update: the next chunk's operand tiles (its Kg waits for this MMA)
        if (ch + 1 < nchunks) {
            if (warp > 0)
                scan_prefix();
            else if (!mbar_wait(pre_bar, (uint32_t)(ch & 1), kPolls))  // warp 0, after its O/S issue
                failed = 1;
            prep_tiles(cr, kgv, true);
        }
        // ================= O pass (+ gated norm) and state pass
        if (!wait_bar(bar_s, par)) failed = 1;
        if (tid == 0 && ch + 1 < nchunks && !failed) issue_p(ch + 1);  // the P rows have been read
        {
            uint32_t r[16];
            const int c0 = wg * 32;
            {  // S^T columns c0.. as packed hi/lo pairs, 16 columns at a time
                uint32_t s1[16], hi[8], lo[8];
                tmem_ld16(tb + lane_off + T_O + wg * 16, r);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    tmem_ld16(tb + lane_off + T_S + c0 + half * 16, s1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        split2(__uint_as_float(s1[2 * c]), __uint_as_float(s1[2 * c + 1]), hi[c], lo[c]);
                    tmem_st8(tb + lane_off + T_SH + wg * 16 + half * 8, hi);
                    tmem_st8(tb + lane_off + T_SL + wg * 16 + half * 8, lo);
                }
                const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                tmem_st16(tb + lane_off + T_O + wg * 16, zero);  // O^T starts from zero next chunk
            }
            const int v = m;
            const int i0 = wg * 16;
            const size_t base = ((size_t)(bos + t0 + i0) * H + h) * DV + v, stride = (size_t)H * DV;
            if (NORM) {
                // sum of squares of each of the 16 rows over this warp's 32 value channels,
                // by a reduce-scatter (16 shuffles): lane pair (2c, 2c + 1) ends with row c
                float *red = fs + F_RED;
                float x2[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float x = __uint_as_float(r[c]);
                    x2[c] = x * x;
                }
                const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
                float a8[8], a4[4], a2[2];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    a8[j] = (u16 ? x2[j + 8] : x2[j]) + __shfl_xor_sync(0xffffffffu, u16 ? x2[j] : x2[j + 8], 16);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    a4[j] = (u8 ? a8[j + 4] : a8[j]) + __shfl_xor_sync(0xffffffffu, u8 ? a8[j] : a8[j + 4], 8);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    a2[j] = (u4 ? a4[j + 2] : a4[j]) + __shfl_xor_sync(0xffffffffu, u4 ? a4[j] : a4[j + 2], 4);
                float e = (u2 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, u2 ? a2[0] : a2[1], 2);
                e += __shfl_xor_sync(0xffffffffu, e, 1);
                if (!(lane & 1)) red[(wg * 4 + wq) * 16 + ((lane >> 1) & 15)] = e;
                const float w = __ldg(p.norm_w + v);
                // sigmoid of the gates before the barrier, with the correctly rounded
                // reciprocal (the value 1 / x has).  A bf16 gate comes from its tile in
                // shared memory; an fp32 one from global memory
                float sg[16];
                if (p.gate_bf16) {
                    if (!mbar_wait(gate_bar, (uint32_t)(ch & 1), kPolls))
                        failed = 1;
                    else if (tid == 0)
                        q_pending = -1;
                    const uint16_t *gs = reinterpret_cast<const uint16_t *>(sm + S_GATE) + i0 * DV + v;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        sg[c] = __frcp_rn(1.0f + __expf(-__uint_as_float((uint32_t)gs[c * DV] << 16)));
                } else {
                    const float *gp = reinterpret_cast<const float *>(p.gate) + ((size_t)(bos + t0) * H + h) * DV + v;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        sg[c] = __frcp_rn(1.0f + __expf(-__ldg(gp + (size_t)min(i0 + c, cn - 1) * H * DV)));
                }
                __syncthreads();
                // lane l forms 1 / rms of row l % 16 once; the others take it by shuffle
                const int cl = lane & 15;
                const float ssl = red[(wg * 4 + 0) * 16 + cl] + red[(wg * 4 + 1) * 16 + cl] +
                                  red[(wg * 4 + 2) * 16 + cl] + red[(wg * 4 + 3) * 16 + cl];
                const float invl = rsqrtf(ssl * (1.f / DV) + p.eps);
                const int rows = min(16, cn - i0);
                if (p.o_bf16) {
                    __nv_bfloat16 *yb = reinterpret_cast<__nv_bfloat16 *>(p.y) + base;
                    __nv_bfloat16 *ob = p.o ? reinterpret_cast<__nv_bfloat16 *>(p.o) + base : nullptr;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float inv = __shfl_sync(0xffffffffu, invl, c);
                        const float x = __uint_as_float(r[c]);
                        if (c < rows) {
                            yb[c * stride] = __float2bfloat16_rn(x * inv * w * sg[c]);
                            if (ob) ob[c * stride] = __float2bfloat16_rn(x);
                        }
                    }
                } else {
                    float *yf = reinterpret_cast<float *>(p.y) + base;
                    float *of = p.o ? reinterpret_cast<float *>(p.o) + base : nullptr;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float inv = __shfl_sync(0xffffffffu, invl, c);
                        const float x = __uint_as_float(r[c]);
                        if (c < rows) {
                            yf[c * stride] = x * inv * w * sg[c];
                            if (of) of[c * stride] = x;
                        }
                    }
                }
            } else if (p.o) {
                // rows i0.. of this head: one base pointer, a constant row stride
                if (!p.o_bf16 && i0 + 16 <= cn) {
                    float *ob = reinterpret_cast<float *>(p.o) + base;
#pragma unroll
                    for (int c = 0; c < 16; ++c) ob[c * stride] = __uint_as_float(r[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (i0 + c < cn) st_out(p.o, base + c * stride, __uint_as_float(r[c]), p.o_bf16);
                }
            }
            tmem_wait_st();
        }
        // the next chunk's first barrier (or the final one) orders these writes before their use
    }
    failed = __syncthreads_or(failed);

    if (failed) {
        if (tid == 0) {
            atomicAdd(&g_chunk_chain_timeouts, 1);
            mma_commit(drain_bar);  // arrives once the tensor-core work already issued has drained
            if (v_pending >= 0) mbar_wait(v_bar, (uint32_t)(v_pending & 1), kPolls);
            if (g_pending >= 0) mbar_wait(g_bar, (uint32_t)(g_pending & 1), kPolls);
            if (tb_pending >= 0) mbar_wait(tb_bar, (uint32_t)(tb_pending & 1), kPolls);
            if (p_pending >= 0) mbar_wait(p_bar, (uint32_t)(p_pending & 1), kPolls);
            if (q_pending >= 0) mbar_wait(gate_bar, (uint32_t)(q_pending & 1), kPolls);
        }
        __syncthreads();
        mbar_wait(drain_bar, 0, kPolls);
        const float nan = __int_as_float(0x7fc00000);
        if (p.sT)
            for (int e = tid; e < DK * DV; e += kThreads) p.sT[(size_t)unit * DK * DV + e] = nan;
        for (int e = tid; e < len * DV; e += kThreads) {  // every row of this (sequence, head)
            const size_t idx = ((size_t)(bos + e / DV) * H + h) * DV + e % DV;
            if (p.o) st_out(p.o, idx, nan, p.o_bf16);
            if (NORM) st_out(p.y, idx, nan, p.o_bf16);
        }
    } else if (p.sT) {  // final state: S[c][v] from S^T (lane v, column c)
        uint32_t s1[16], s2[16];
        const int c0 = wg * 32;
        tmem_ld16(tb + lane_off + T_S + c0, s1);
        tmem_ld16(tb + lane_off + T_S + c0 + 16, s2);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            p.sT[((size_t)unit * DK + c0 + c) * DV + m] = __uint_as_float(s1[c]);
            p.sT[((size_t)unit * DK + c0 + 16 + c) * DV + m] = __uint_as_float(s2[c]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

int take_chunk_chain_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_chunk_chain_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_chunk_chain_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("chunk_chain: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

kda_status launch_chunk_chain(const SeqParams &p_in, const void *ws, cudaStream_t st) {
    const int units = p_in.N * p_in.H;
    if (units == 0) return KDA_OK;
    const long long rows = p_in.cu_seqlens ? (long long)p_in.T : (long long)p_in.N * p_in.T;
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!enc) {
        set_error("chunk_chain: cuTensorMapEncodeTiled is not available from the driver");
        return KDA_ERR_CUDA;
    }
    const cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap tmap;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)p_in.H, (cuuint64_t)rows};
        const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)p_in.H * DV * 2};
        const cuuint32_t box[3] = {64, 1, 64};
        const CUresult cres = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p_in.v), dims, strides,
                                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cres != CUDA_SUCCESS) {
            set_error("chunk_chain: cuTensorMapEncodeTiled failed (%d)", (int)cres);
            return KDA_ERR_CUDA;
        }
    }
    CUtensorMap tmap_g;
    {
        const bool gb = p_in.g_logits && p_in.g_logits_bf16;
        const cuuint64_t es = gb ? 2 : 4;
        const void *gsrc = p_in.g_logits ? p_in.g_logits : (const void *)p_in.g;
        const cuuint64_t gdims[3] = {(cuuint64_t)DK, (cuuint64_t)p_in.H, (cuuint64_t)rows};
        const cuuint64_t gstrides[2] = {(cuuint64_t)DK * es, (cuuint64_t)p_in.H * DK * es};
        const cuuint32_t gbox[3] = {(cuuint32_t)DK, 1, (cuuint32_t)C};
        const CUresult cres =
            enc(&tmap_g, gb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                const_cast<void *>(gsrc), gdims, gstrides, gbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cres != CUDA_SUCCESS) {
            set_error("chunk_chain: cuTensorMapEncodeTiled failed for g (%d)", (int)cres);
            return KDA_ERR_CUDA;
        }
    }
    // fused norm with a bf16 gate: the gate tile of a chunk by one TMA copy; otherwise the
    // map is not read (V's map stands in)
    CUtensorMap tmap_gate = tmap;
    if (p_in.gate && p_in.gate_bf16) {
        const cuuint64_t qdims[3] = {(cuuint64_t)DV, (cuuint64_t)p_in.H, (cuuint64_t)rows};
        const cuuint64_t qstrides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)p_in.H * DV * 2};
        const cuuint32_t qbox[3] = {(cuuint32_t)DV, 1, (cuuint32_t)C};
        const CUresult cres = enc(&tmap_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p_in.gate), qdims,
                                  qstrides, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cres != CUDA_SUCCESS) {
            set_error("chunk_chain: cuTensorMapEncodeTiled failed for the gate (%d)", (int)cres);
            return KDA_ERR_CUDA;
        }
    }
    ChainParams cp;
    memset(&cp, 0, sizeof(cp));
    cp.p = p_in;
    cp.ws = static_cast<const uint8_t *>(ws);
    // longest sequences first when the host copy of cu_seqlens is known
    if (p_in.cu_seqlens && p_in.cu_host && p_in.N <= 64) {
        cp.order_n = p_in.N;
        for (int i = 0; i < p_in.N; ++i) cp.order[i] = i;
        for (int i = 1; i < p_in.N; ++i) {  // insertion sort by length, descending
            const int x = cp.order[i];
            const int lx = p_in.cu_host[x + 1] - p_in.cu_host[x];
            int j = i - 1;
            while (j >= 0 && p_in.cu_host[cp.order[j] + 1] - p_in.cu_host[cp.order[j]] < lx) {
                cp.order[j + 1] = cp.order[j];
                --j;
            }
            cp.order[j + 1] = x;
        }
    }
    static DeviceOnce configured;
    const int dev = current_device();
    if (!configured.done(dev)) {
        for (void *fn : {(void *)chunk_chain_kernel<false, false>, (void *)chunk_chain_kernel<true, false>,
                         (void *)chunk_chain_kernel<false, true>, (void *)chunk_chain_kernel<true, true>}) {
            const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            if (e != cudaSuccess) {
                set_error("chunk_chain: cannot reserve %u bytes of shared memory: %s", SMEM_BYTES, cudaGetErrorString(e));
                return KDA_ERR_CUDA;
            }
        }
        configured.set(dev);
    }
    auto kern = p_in.g_logits ? (p_in.gate ? chunk_chain_kernel<true, true> : chunk_chain_kernel<true, false>)
                              : (p_in.gate ? chunk_chain_kernel<false, true> : chunk_chain_kernel<false, false>);
    kern<<<units, kThreads, SMEM_BYTES, st>>>(tmap, tmap_g, tmap_gate, cp);
    note_launch();
    return check_launch("chunk_chain_kernel");
}

}  // namespace kda
