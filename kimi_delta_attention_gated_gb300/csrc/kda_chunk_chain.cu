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
// columns and the three MMA groups are the fused kernel's (kda_chunk_tc.cu).
//
// The CTA's 16 warps are two groups that meet only through mbarriers:
//   pass warps 0-7   the chain: after each MMA group they move its accumulator through
//                    registers (R^T and D^T into split-bf16 in place, S^T decayed and split,
//                    O out with the gated norm); thread 0 issues every MMA and copy.  Warp w
//                    serves TMEM lanes 32 (w % 4).. and half w / 4 of the columns.  Their
//                    barriers are named barrier 1 with an OR-vote, so a failed wait takes
//                    every pass warp out of the loop together.
//   prep warps 8-15  the next chunk's operands, one chunk ahead of the chain: q, k and
//                    norms (tokens 8w..8w+7 of warp 8 + w, key channels 4 lane..), the
//                    in-chunk cumulative decay, exp(gamma), the [-Kd ; Qd] tiles (once the
//                    chain's R/O product has read the previous ones) and the Kg^T rows (once
//                    its O/S product has read those); named barrier 2.
// So the tile preparation no longer lengthens the chain: it runs beside it instead of in
// fixed windows between its barriers, and the warp that issues the MMAs prepares nothing.
// Kd, Qd and Kg take non-positive exponents only (a channel whose decay range exceeds
// kRangeMax forms Kg from exp(gamma - G) directly), so the chain needs no exact fallback.
// The arithmetic of the norms, the cumulative decay and the tiles is the fused kernel's,
// so the split form gives the fused form's bits wherever no channel takes that branch.
// Every wait is bounded; a CTA whose wait gives up writes NaN into its final state, o, y.
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

constexpr int kThreads = 512;  // 16 warps: pass warps 0-7, prep warps 8-15
constexpr int kGroup = 256;    // threads per group

// TMEM columns.  The R/O product writes [R_hh | O_hh | R_hl | O_hl] over [0, 256): the hi
// part of S^T against the hi and lo [-Kd ; Qd] rows stacked along N (one N = 256 product
// per K step), then the lo part against the hi rows onto [R | O] at [0, 128).  The R pass
// folds R_hl into R (split into hi/lo in place at [0, 64)) and O_hh into O at [192, 256),
// which lies just before S^T so that the O/S product writes [O | S] as one N = 192 block;
// the D accumulator takes the columns [64, 192) the R pass has freed.
constexpr uint32_t T_R = 0, T_D = 64, T_O = 192, T_S = 256, T_SH = 384, T_SL = 448;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_V = 0;          // V tile, two TMA boxes of 64 tokens x 64 values (16 KB)
constexpr uint32_t S_KQ = 16384;     // [-Kd ; Qd], 128 rows x 128 (64 KB): per 64 key channels, the hi rows
                                     // then the lo rows (16 KB each), i.e. one 256-row operand per K block
constexpr uint32_t S_GT = 81920;     // g (or logits) tile of the chunk being prepared, 64 tokens x 128 (32 KB)
constexpr uint32_t S_PKGH = 114688;  // [P ; Kg^T] hi, 192 rows (i, then c) x 64 (j) (24 KB), K-major B
constexpr uint32_t S_PKGL = 139264;  // [P ; Kg^T] lo
constexpr uint32_t S_TBH = 163840;   // T diag(beta) hi, 64 x 64 (8 KB); lo follows at S_TBH + 8 KB
constexpr uint32_t S_ID = 180224;    // bf16 identity 64 x 64 (8 KB)
constexpr uint32_t S_GATE = 188416;  // fused norm: the chunk's bf16 gate tile, 64 tokens x 128 (16 KB)
constexpr uint32_t S_SCAN = 204800;  // decay totals of the 16 groups of 4 tokens [2 parities][16][128]
constexpr uint32_t S_SMALL = S_SCAN + 2 * 16 * 128 * 4;
// small buffers (floats)
constexpr uint32_t F_RQ = 0;      // q scale per token (norm * scale) [64]
constexpr uint32_t F_RK = 64;     // k norm per token [64]
constexpr uint32_t F_GEXP = 128;  // exp(gamma) of the chunk, double-buffered by its parity [2][128]
constexpr uint32_t F_RED = 384;   // norm partials [2 halves][4 quarters][32 tokens]
constexpr uint32_t F_AH = 640;    // gates from logits: exp(A_log) of the head [1 of 4]
constexpr uint32_t F_DB = 644;    // gates from logits: dt_bias of the head's channels [128]
constexpr uint32_t F_END = 772;
constexpr uint32_t S_BARS = S_SMALL + F_END * 4;     // 11 mbarriers + tmem slot + failure flag
constexpr uint32_t SMEM_BYTES = S_BARS + 112 + 1024;  // + alignment slack

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

// Named barrier `id` over `n` threads that also ORs `pred` across them (the vote makes a
// failure leave the loop in every participating warp at once).
template <int id, int n>
__device__ __forceinline__ int group_sync_or(int pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred), "n"(id), "n"(n)
        : "memory");
    return (int)out;
}

// The 16 sums (q of tokens 0-7, then k) of a prep warp reduced over its lanes by a
// reduce-scatter: lanes 2v and 2v + 1 end with sum v.  Each sum goes through the same
// pairing tree as in the fused kernel's 8-sum form, so the norms are the same bits.
__device__ __forceinline__ float reduce_scatter16(const float (&a)[16], int lane) {
    const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
    float b8[8], b4[4], b2[2];
#pragma unroll
    for (int j = 0; j < 8; ++j) b8[j] = (u16 ? a[j + 8] : a[j]) + __shfl_xor_sync(0xffffffffu, u16 ? a[j] : a[j + 8], 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) b4[j] = (u8 ? b8[j + 4] : b8[j]) + __shfl_xor_sync(0xffffffffu, u8 ? b8[j] : b8[j + 4], 8);
#pragma unroll
    for (int j = 0; j < 2; ++j) b2[j] = (u4 ? b4[j + 2] : b4[j]) + __shfl_xor_sync(0xffffffffu, u4 ? b4[j] : b4[j + 2], 4);
    float d = (u2 ? b2[1] : b2[0]) + __shfl_xor_sync(0xffffffffu, u2 ? b2[0] : b2[1], 2);
    return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

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
    float *scan = reinterpret_cast<float *>(sm + S_SCAN);
    // one barrier per tensor-core group, copy or hand-over, each completing once per chunk
    uint64_t *bar_r = reinterpret_cast<uint64_t *>(sm + S_BARS);  // R and O products
    uint64_t *bar_d = bar_r + 1;                                    // D product
    uint64_t *bar_s = bar_r + 2;                                    // O and S updates
    uint64_t *v_bar = bar_r + 3;                                    // V tile
    uint64_t *g_bar = bar_r + 4;                                    // g tile
    uint64_t *tb_bar = bar_r + 5;                                   // T diag(beta) image
    uint64_t *p_bar = bar_r + 6;                                    // P image
    uint64_t *gate_bar = bar_r + 7;                                 // fused norm: gate tile
    uint64_t *tiles_bar = bar_r + 8;                                // [-Kd ; Qd] tiles written (8 prep warps)
    uint64_t *kg_bar = bar_r + 9;                                   // Kg^T rows written (8 prep warps)
    uint64_t *drain_bar = bar_r + 10;                               // drain after a failure
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_BARS + 88);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H;
    int n = blockIdx.x / H;
    const int h = blockIdx.x % H;
    if (cp.order_n > 0) n = cp.order[n];
    const int unit = n * H + h;
    int bos, len;
    seq_range(p, n, bos, len);
    const int nchunks = (len + C - 1) / C;
    auto blob = [&](int chunk) { return cp.ws + ((size_t)blob_slot(bos, n, chunk) * H + h) * kBlobBytes; };

    if (tid == 0) {
        for (int b = 0; b < 11; ++b) mbar_init(bar_r + b, (b == 8 || b == 9) ? 8 : 1);
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
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int failed = 0;
    // copies in flight (the issuing thread's view): chunk whose copy is pending, or -1
    int v_pending = -1, g_pending = -1, tb_pending = -1, p_pending = -1, q_pending = -1;

    if (warp < 8) {
        // ===================================================================== pass warps
        const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
        const int m = q4 * 32 + lane;             // TMEM lane = value channel
        auto issue_v = [&](int chunk) {
            mbar_arrive_expect_tx(v_bar, 16384);
            tma_load_3d(sb + S_V, &tmap_v, v_bar, 0, h, bos + chunk * C);
            tma_load_3d(sb + S_V + 8192, &tmap_v, v_bar, 64, h, bos + chunk * C);
            v_pending = chunk;
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
        if (tid == 0 && nchunks > 0) {
            issue_v(0);
            issue_tb(0);
            issue_p(0);
        }
        // The fp32 accumulator holds the state already decayed by the chunk about to be
        // processed (S^T exp(gamma), ready for the O/S product), while the hi/lo copy that the
        // R/O product reads holds it undecayed: each state pass writes both.  The first
        // chunk's exp(gamma) comes from the prep warps, published with its tiles.
        const bool have_first = nchunks > 0 && mbar_wait(tiles_bar, 0u, kPolls);
        if (nchunks > 0 && !have_first) failed = 1;
        {  // initial state -> S^T accumulator and its hi/lo copy (channels 64 hf..)
            const int c0 = hf * 64;
            const float *ge = fs + F_GEXP + c0;  // exp(gamma) of chunk 0 (parity 0)
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                float s[32];
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    s[c] = p.s0 ? p.s0[((size_t)unit * DK + c0 + qq * 32 + c) * DV + m] : 0.f;
                uint32_t r[16], hi[16], lo[16];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        r[c] = __float_as_uint(have_first ? s[half * 16 + c] * ge[qq * 32 + half * 16 + c] : s[half * 16 + c]);
                    tmem_st16(tb + lane_off + T_S + c0 + qq * 32 + half * 16, r);
                }
#pragma unroll
                for (int c = 0; c < 16; ++c) split2(s[2 * c], s[2 * c + 1], hi[c], lo[c]);
                tmem_st16(tb + lane_off + T_SH + (c0 + qq * 32) / 2, hi);
                tmem_st16(tb + lane_off + T_SL + (c0 + qq * 32) / 2, lo);
            }
            tmem_wait_st();
        }
        auto wait_bar = [&](uint64_t *bar, int parity) {
            const bool ok = mbar_wait(bar, (uint32_t)parity, kPolls);
            fence_after_sync();
            return ok;
        };
        // splits 16 fp32 columns (two blocks of 8 pairs) already in registers into [hi x 8 | lo x 8]
        auto split_store = [&](uint32_t col, const uint32_t (&r)[16]) {
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) split2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]), hi[c], lo[c]);
            tmem_st8(tb + lane_off + col, hi);
            tmem_st8(tb + lane_off + col + 8, lo);
        };

        for (int ch = 0; ch < nchunks; ++ch) {
            const int par = ch & 1;
            const int t0 = ch * C;
            const int cn = min(C, len - t0);
            fence_before_sync();  // the previous state pass (or the initial state) wrote TMEM
            if (group_sync_or<1, kGroup>(failed)) break;

            // ================= R^T = V^T I + S^T (-Kd)^T, O^T = S^T Qd^T
            if (tid == 0) {
                fence_after_sync();
                if (!mbar_wait(tiles_bar, (uint32_t)par, kPolls)) failed = 1;  // the prep warps' tiles
                if (mbar_wait(v_bar, (uint32_t)par, kPolls))
                    v_pending = -1;
                else
                    failed = 1;
                fence_after_sync();
                const uint32_t id256 = idesc_bf16(128, 256, false, false), id128 = idesc_bf16(128, 128, false, false);
                const uint32_t id_mn = idesc_bf16(128, 64, true, false);
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // S^T_hi [KQ_hi ; KQ_lo]^T -> [R_hh | O_hh | R_hl | O_hl]
                    const uint32_t koff = (s >> 2) * 32768 + (s & 3) * 32;
                    mma_ts(tb + T_R, tb + T_SH + s * 8, sdesc_at(sb16, S_KQ + koff, 16, 1024), id256, s ? 1u : 0u);
                }
#pragma unroll 1
                for (int s = 0; s < 4; ++s)  // + V^T (exact bf16 identity) onto R
                    mma_ss(tb + T_R, sdesc_at(sb16, S_V + s * 2048, 8192, 1024), sdesc_at(sb16, S_ID + s * 32, 16, 1024),
                           id_mn, 1u);
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // S^T_lo KQ_hi^T onto [R | O]
                    const uint32_t koff = (s >> 2) * 32768 + (s & 3) * 32;
                    mma_ts(tb + T_R, tb + T_SL + s * 8, sdesc_at(sb16, S_KQ + koff, 16, 1024), id128, 1u);
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

            // ================= R pass: R^T (lane v, tokens 32 hf..) -> hi/lo in place
            if (!wait_bar(bar_r, par)) failed = 1;
            if (tid == 0 && ch + 1 < nchunks && !failed) issue_v(ch + 1);  // the V tile has been read
#pragma unroll
            for (int b = 0; b < 2; ++b) {  // tokens 32 hf + 16 b ..: R = R_hh + R_hl, O = O_hh + O_hl
                const uint32_t col = hf * 32 + b * 16;
                uint32_t rh[16], rl[16], oh[16], ol[16];
                tmem_ld16(tb + lane_off + T_R + col, rh);
                tmem_ld16(tb + lane_off + T_R + 128 + col, rl);
                tmem_ld16(tb + lane_off + T_R + 64 + col, oh);
                tmem_ld16(tb + lane_off + T_R + 192 + col, ol);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float2 rv = __fadd2_rn(make_float2(__uint_as_float(rh[c]), __uint_as_float(rh[c + 1])),
                                                 make_float2(__uint_as_float(rl[c]), __uint_as_float(rl[c + 1])));
                    const float2 ov = __fadd2_rn(make_float2(__uint_as_float(oh[c]), __uint_as_float(oh[c + 1])),
                                                 make_float2(__uint_as_float(ol[c]), __uint_as_float(ol[c + 1])));
                    rh[c] = __float_as_uint(rv.x); rh[c + 1] = __float_as_uint(rv.y);
                    oh[c] = __float_as_uint(ov.x); oh[c + 1] = __float_as_uint(ov.y);
                }
                split_store(T_R + col, rh);
                tmem_st16(tb + lane_off + T_O + col, oh);
            }
            tmem_wait_st();
            fence_before_sync();
            if (group_sync_or<1, kGroup>(failed)) break;

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

            // ================= D pass: D = D_a + D_b -> hi/lo in place
            if (!wait_bar(bar_d, par)) failed = 1;
            if (tid == 0 && ch + 1 < nchunks && !failed) issue_tb(ch + 1);  // the T diag(beta) tile has been read
            {
                const uint32_t col = T_D + hf * 32;
                uint32_t a0[16], a1[16], b0[16], b1[16];
                tmem_ld16(tb + lane_off + col, a0);
                tmem_ld16(tb + lane_off + col + 16, a1);
                tmem_ld16(tb + lane_off + col + 64, b0);
                tmem_ld16(tb + lane_off + col + 80, b1);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float2 v0 = __fadd2_rn(make_float2(__uint_as_float(a0[c]), __uint_as_float(a0[c + 1])),
                                                 make_float2(__uint_as_float(b0[c]), __uint_as_float(b0[c + 1])));
                    const float2 v1 = __fadd2_rn(make_float2(__uint_as_float(a1[c]), __uint_as_float(a1[c + 1])),
                                                 make_float2(__uint_as_float(b1[c]), __uint_as_float(b1[c + 1])));
                    a0[c] = __float_as_uint(v0.x); a0[c + 1] = __float_as_uint(v0.y);
                    a1[c] = __float_as_uint(v1.x); a1[c + 1] = __float_as_uint(v1.y);
                }
                split_store(col, a0);
                split_store(col + 16, a1);
                tmem_wait_st();
            }
            fence_before_sync();
            if (group_sync_or<1, kGroup>(failed)) break;

            // ================= [O|S]^T += D^T [P^T | Kg]
            if (tid == 0) {
                fence_after_sync();
                if (mbar_wait(p_bar, (uint32_t)par, kPolls))
                    p_pending = -1;
                else
                    failed = 1;
                if (!mbar_wait(kg_bar, (uint32_t)par, kPolls)) failed = 1;  // the prep warps' Kg^T rows
                fence_after_sync();
                const uint32_t id192 = idesc_bf16(128, 192, false, false);
#pragma unroll
                for (int cb = 0; cb < 3; ++cb)
#pragma unroll 1
                    for (int s = 0; s < 4; ++s)
                        mma_ts(tb + T_O, tb + T_D + s * 16 + (combo_a(cb) ? 8 : 0),
                               sdesc_at(sb16, (combo_b(cb) ? S_PKGL : S_PKGH) + s * 32, 16, 1024), id192, 1u);
                mma_commit(bar_s);
            }
            __syncwarp();

            // ================= O pass (+ gated norm) and state pass
            if (!wait_bar(bar_s, par)) failed = 1;
            if (tid == 0 && ch + 1 < nchunks && !failed) issue_p(ch + 1);  // the P rows have been read
            // the next chunk's exp(gamma), published by the prep warps with its tiles
            const bool next = ch + 1 < nchunks;
            if (next && !mbar_wait(tiles_bar, (uint32_t)((ch + 1) & 1), kPolls)) failed = 1;
            {
                const float *ge = fs + F_GEXP + ((ch + 1) & 1) * 128 + hf * 64;
                uint32_t r[32];
                // S^T channels 64 hf..: the hi/lo copy of the state the next chunk starts from,
                // and the fp32 accumulator decayed by that chunk's exp(gamma)
#pragma unroll
                for (int qh = 0; qh < 2; ++qh) {
                    uint32_t s0[16], s1[16];
                    tmem_ld16(tb + lane_off + T_S + hf * 64 + qh * 32, s0);
                    tmem_ld16(tb + lane_off + T_S + hf * 64 + qh * 32 + 16, s1);
                    if (qh == 0) {
                        uint32_t o0[16], o1[16];  // (the next R/O product overwrites these columns)
                        tmem_ld16(tb + lane_off + T_O + hf * 32, o0);
                        tmem_ld16(tb + lane_off + T_O + hf * 32 + 16, o1);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            r[c] = o0[c];
                            r[16 + c] = o1[c];
                        }
                    } else {
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        uint32_t(&sv)[16] = b ? s1 : s0;
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            split2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1]), hi[c], lo[c]);
                        tmem_st8(tb + lane_off + T_SH + hf * 32 + qh * 16 + b * 8, hi);
                        tmem_st8(tb + lane_off + T_SL + hf * 32 + qh * 16 + b * 8, lo);
                        if (next) {
#pragma unroll
                            for (int c4 = 0; c4 < 4; ++c4) {
                                const float4 a = *reinterpret_cast<const float4 *>(ge + qh * 32 + b * 16 + c4 * 4);
                                const float2 x0 = __fmul2_rn(
                                    make_float2(__uint_as_float(sv[4 * c4]), __uint_as_float(sv[4 * c4 + 1])), make_float2(a.x, a.y));
                                const float2 x1 = __fmul2_rn(
                                    make_float2(__uint_as_float(sv[4 * c4 + 2]), __uint_as_float(sv[4 * c4 + 3])), make_float2(a.z, a.w));
                                sv[4 * c4 + 0] = __float_as_uint(x0.x); sv[4 * c4 + 1] = __float_as_uint(x0.y);
                                sv[4 * c4 + 2] = __float_as_uint(x1.x); sv[4 * c4 + 3] = __float_as_uint(x1.y);
                            }
                            tmem_st16(tb + lane_off + T_S + hf * 64 + qh * 32 + b * 16, sv);
                        }
                    }
                }
                const int v = m, i0 = hf * 32;
                const int rows = min(32, cn - i0);
                const size_t base = ((size_t)(bos + t0 + i0) * H + h) * DV + v, stride = (size_t)H * DV;
                if (NORM) {
                    // sum of squares of each of the 32 rows over this warp's 32 value channels, by a
                    // reduce-scatter: lane j ends with row j
                    float *red = fs + F_RED;
                    float x2[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float x = __uint_as_float(r[c]);
                        x2[c] = x * x;
                    }
                    float e;
                    {
                        const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
                        float a16[16], a8[8], a4[4], a2[2];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            a16[j] = (u16 ? x2[j + 16] : x2[j]) + __shfl_xor_sync(0xffffffffu, u16 ? x2[j] : x2[j + 16], 16);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            a8[j] = (u8 ? a16[j + 8] : a16[j]) + __shfl_xor_sync(0xffffffffu, u8 ? a16[j] : a16[j + 8], 8);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            a4[j] = (u4 ? a8[j + 4] : a8[j]) + __shfl_xor_sync(0xffffffffu, u4 ? a8[j] : a8[j + 4], 4);
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            a2[j] = (u2 ? a4[j + 2] : a4[j]) + __shfl_xor_sync(0xffffffffu, u2 ? a4[j] : a4[j + 2], 2);
                        e = (u1 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, u1 ? a2[0] : a2[1], 1);
                    }
                    red[(hf * 4 + q4) * 32 + lane] = e;
                    const float w = __ldg(p.norm_w + v);
                    // sigmoid of the gates before the barrier, with the fast reciprocal (2 ulp).
                    // A bf16 gate comes from its tile, an fp32 one from global memory
                    float sg[32];
                    if (p.gate_bf16) {
                        if (!mbar_wait(gate_bar, (uint32_t)par, kPolls))
                            failed = 1;
                        else if (tid == 0)
                            q_pending = -1;
                        const uint16_t *gs = reinterpret_cast<const uint16_t *>(sm + S_GATE) + i0 * DV + v;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            sg[c] = __fdividef(1.0f, 1.0f + __expf(-__uint_as_float((uint32_t)gs[c * DV] << 16)));
                    } else {
                        const float *gp = reinterpret_cast<const float *>(p.gate) + ((size_t)(bos + t0) * H + h) * DV + v;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            sg[c] = __fdividef(1.0f, 1.0f + __expf(-__ldg(gp + (size_t)min(i0 + c, cn - 1) * H * DV)));
                    }
                    group_sync_or<1, kGroup>(0);
                    // lane j forms 1 / rms of row j once; the others take it by shuffle
                    const float ssl = red[(hf * 4 + 0) * 32 + lane] + red[(hf * 4 + 1) * 32 + lane] +
                                      red[(hf * 4 + 2) * 32 + lane] + red[(hf * 4 + 3) * 32 + lane];
                    const float invl = rsqrtf(ssl * (1.f / DV) + p.eps);
                    if (p.o_bf16) {
                        __nv_bfloat16 *yb = reinterpret_cast<__nv_bfloat16 *>(p.y) + base;
                        __nv_bfloat16 *ob = p.o ? reinterpret_cast<__nv_bfloat16 *>(p.o) + base : nullptr;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
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
                        for (int c = 0; c < 32; ++c) {
                            const float inv = __shfl_sync(0xffffffffu, invl, c);
                            const float x = __uint_as_float(r[c]);
                            if (c < rows) {
                                yf[c * stride] = x * inv * w * sg[c];
                                if (of) of[c * stride] = x;
                            }
                        }
                    }
                } else if (p.o) {
                    if (!p.o_bf16 && rows == 32) {
                        float *ob = reinterpret_cast<float *>(p.o) + base;
#pragma unroll
                        for (int c = 0; c < 32; ++c) ob[c * stride] = __uint_as_float(r[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (c < rows) st_out(p.o, base + c * stride, __uint_as_float(r[c]), p.o_bf16);
                    }
                }
                tmem_wait_st();
            }
            // the next chunk's first pass-group barrier orders these writes before their use
        }
    } else {
        // ===================================================================== prep warps
        const int pw = warp - 8, l4 = lane * 4;
        const uint32_t g_bytes = (GL && p.g_logits_bf16) ? C * DK * 2 : C * DK * 4;
        auto issue_g = [&](int chunk) {
            mbar_arrive_expect_tx(g_bar, g_bytes);
            tma_load_3d(sb + S_GT, &tmap_g, g_bar, 0, h, bos + chunk * C);
            g_pending = chunk;
        };
        // q and k of one chunk for this thread's 8 tokens x 4 key channels, into registers
        uint2 qr[8], kr[8];
        auto load_qk = [&](int chunk) {
            const int cnn = min(C, len - chunk * C);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = min(pw * 8 + r, cnn - 1);
                const size_t hk = ((size_t)(bos + chunk * C + i) * H + h) * DK + l4;
                qr[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) + hk));
                kr[r] = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.k) + hk));
            }
        };
        if (tid == 256 && nchunks > 0) issue_g(0);
        if (nchunks > 0) load_qk(0);
        float kgv[8][4];  // the chunk's Kg, stored when its [P ; Kg^T] tile is free

        for (int ch = 0; ch < nchunks; ++ch) {
            const int par = ch & 1;
            const int cn = min(C, len - ch * C);
            // ---- norms and the decay totals of each group of 4 tokens, from the g tile
            if (!mbar_wait(g_bar, (uint32_t)par, kPolls))
                failed = 1;
            else if (tid == 256)
                g_pending = -1;
            float4 g[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int i = pw * 8 + r;
                if (i >= cn) {  // tokens past the chunk's end: q = k = 0 (loaded as a copy), g = 0
                    qr[r] = make_uint2(0u, 0u);
                    kr[r] = make_uint2(0u, 0u);
                }
                if (GL && p.g_logits_bf16) {
                    const uint2 u = *reinterpret_cast<const uint2 *>(sm + S_GT + (i * DK + l4) * 2);
                    g[r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), 0.f, 0.f);
                } else {
                    g[r] = *reinterpret_cast<const float4 *>(sm + S_GT + (i * DK + l4) * 4);
                }
                if (!GL && i >= cn) g[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (GL) {  // g from its logits; tokens past the chunk's end keep g = 0
                const float a_h = fs[F_AH];
                const float4 db = *reinterpret_cast<const float4 *>(fs + F_DB + l4);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    float z[4];
                    if (p.g_logits_bf16) {
                        const uint32_t ux = __float_as_uint(g[r].x), uy = __float_as_uint(g[r].y);
                        z[0] = bf16lo(ux); z[1] = bf16hi(ux); z[2] = bf16lo(uy); z[3] = bf16hi(uy);
                    } else {
                        z[0] = g[r].x; z[1] = g[r].y; z[2] = g[r].z; z[3] = g[r].w;
                    }
                    const bool live = pw * 8 + r < cn;
                    g[r] = make_float4(live ? gate_of_logit(z[0] + db.x, a_h, p.g_lower) : 0.f,
                                       live ? gate_of_logit(z[1] + db.y, a_h, p.g_lower) : 0.f,
                                       live ? gate_of_logit(z[2] + db.z, a_h, p.g_lower) : 0.f,
                                       live ? gate_of_logit(z[3] + db.w, a_h, p.g_lower) : 0.f);
                }
            }
            {
                float a16[16];
#pragma unroll
                for (int r = 0; r < 8; ++r) {  // (q, k) sums of squares as packed pairs
                    const float2 v0 = make_float2(bf16lo(qr[r].x), bf16lo(kr[r].x));
                    const float2 v1 = make_float2(bf16hi(qr[r].x), bf16hi(kr[r].x));
                    const float2 v2 = make_float2(bf16lo(qr[r].y), bf16lo(kr[r].y));
                    const float2 v3 = make_float2(bf16hi(qr[r].y), bf16hi(kr[r].y));
                    const float2 ss = __ffma2_rn(v0, v0, __ffma2_rn(v1, v1, __ffma2_rn(v2, v2, __fmul2_rn(v3, v3))));
                    a16[r] = ss.x;
                    a16[8 + r] = ss.y;
                }
                const float d = reduce_scatter16(a16, lane);
                if ((lane & 1) == 0) {
                    const int v = lane >> 1;
                    const float sc = p.l2norm ? rsqrtf(d + 1e-6f) : 1.f;
                    if (v < 8)
                        fs[F_RQ + pw * 8 + v] = sc * p.scale;
                    else
                        fs[F_RK + pw * 8 + v - 8] = sc;
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // totals of tokens 8pw..8pw+3 and 8pw+4..8pw+7
                float2 t01 = make_float2(g[4 * half].x, g[4 * half].y), t23 = make_float2(g[4 * half].z, g[4 * half].w);
#pragma unroll
                for (int r = 1; r < 4; ++r) {
                    t01 = __fadd2_rn(t01, make_float2(g[4 * half + r].x, g[4 * half + r].y));
                    t23 = __fadd2_rn(t23, make_float2(g[4 * half + r].z, g[4 * half + r].w));
                }
                *reinterpret_cast<float4 *>(scan + par * 2048 + (2 * pw + half) * 128 + l4) =
                    make_float4(t01.x, t01.y, t23.x, t23.y);
            }
            if (group_sync_or<2, kGroup>(failed)) break;
            // the g tile is consumed: the next chunk's arrives while this one is prepared
            if (tid == 256 && ch + 1 < nchunks) issue_g(ch + 1);
            // ---- exclusive prefix of the 16 group totals per channel (each thread sums them in
            // order itself), the chunk total and exp(gamma).  The totals are double-buffered by
            // the chunk's parity: a warp that runs ahead writes the next chunk's while a slower
            // one still reads these (it cannot get two chunks ahead: the barrier above)
            float o4[2][4], gam[4] = {0.f, 0.f, 0.f, 0.f};
            auto add_total = [&](int w) {
                const float4 t = *reinterpret_cast<const float4 *>(scan + par * 2048 + w * 128 + l4);
                gam[0] += t.x;
                gam[1] += t.y;
                gam[2] += t.z;
                gam[3] += t.w;
            };
#pragma unroll 1
            for (int w = 0; w < 2 * pw; ++w) add_total(w);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[half][e] = gam[e];
                add_total(2 * pw + half);
            }
#pragma unroll 1
            for (int w = 2 * pw + 2; w < 16; ++w) add_total(w);
            float egam[4];
            bool wide = false;  // a channel whose decay range is too wide for exp(-G) exp(gamma)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                egam[e] = __expf(gam[e]);
                wide |= -gam[e] > kRangeMax;
            }
            if (pw == 1) *reinterpret_cast<float4 *>(fs + F_GEXP + par * 128 + l4) = make_float4(egam[0], egam[1], egam[2], egam[3]);
            // ---- the [-Kd ; Qd] tiles, once the chain's previous R/O product has read them
            if (ch > 0 && !mbar_wait(bar_r, (uint32_t)((ch - 1) & 1), kPolls)) failed = 1;
            const float2 eg2[2] = {make_float2(egam[0], egam[1]), make_float2(egam[2], egam[3])};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float2 o2[2] = {make_float2(o4[half][0], o4[half][1]), make_float2(o4[half][2], o4[half][3])};
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int r = 4 * half + rr, i = pw * 8 + r;
                    const float rk = fs[F_RK + i], rq = fs[F_RQ + i];
                    const float2 gr2[2] = {make_float2(g[r].x, g[r].y), make_float2(g[r].z, g[r].w)};
                    const float2 kv2[2] = {make_float2(bf16lo(kr[r].x), bf16hi(kr[r].x)),
                                           make_float2(bf16lo(kr[r].y), bf16hi(kr[r].y))};
                    const float2 qv2[2] = {make_float2(bf16lo(qr[r].x), bf16hi(qr[r].x)),
                                           make_float2(bf16lo(qr[r].y), bf16hi(qr[r].y))};
                    const float2 rk2 = make_float2(rk, rk), nrk2 = make_float2(-rk, -rk), rq2 = make_float2(rq, rq);
                    float2 kd[2], qd[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        o2[e] = __fadd2_rn(o2[e], gr2[e]);  // inclusive cumulative decay G of token i
                        const float2 em = make_float2(__expf(-o2[e].x), __expf(-o2[e].y));
                        const float2 kg = __fmul2_rn(__fmul2_rn(__fmul2_rn(kv2[e], rk2), em), eg2[e]);
                        kgv[r][2 * e] = kg.x;
                        kgv[r][2 * e + 1] = kg.y;
                        const float2 eG = make_float2(__expf(o2[e].x), __expf(o2[e].y));
                        kd[e] = __fmul2_rn(__fmul2_rn(kv2[e], nrk2), eG);  // -k^ exp(G)
                        qd[e] = __fmul2_rn(__fmul2_rn(qv2[e], rq2), eG);
                    }
                    if (wide) {  // exp(-G) exp(gamma) would overflow: exp(gamma - G) directly
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (-gam[e] > kRangeMax) {
                                const float ke = (e & 1) ? kv2[e >> 1].y : kv2[e >> 1].x;
                                const float ge = (e & 1) ? o2[e >> 1].y : o2[e >> 1].x;
                                kgv[r][e] = ke * rk * __expf(gam[e] - ge);
                            }
                    }
                    // rows i and 64 + i share the swizzle phase; each 64-channel block holds the
                    // 128 hi rows, then the 128 lo rows
                    const uint32_t off = sw128_off(i, l4 & 63, 128) + (uint32_t)(l4 >> 6) * 32768u;
                    uint32_t h0, lo0, h1, lo1;
                    split2(kd[0].x, kd[0].y, h0, lo0);
                    split2(kd[1].x, kd[1].y, h1, lo1);
                    st_shared_v2(sb + S_KQ + off, h0, h1);
                    st_shared_v2(sb + S_KQ + off + 16384, lo0, lo1);
                    split2(qd[0].x, qd[0].y, h0, lo0);
                    split2(qd[1].x, qd[1].y, h1, lo1);
                    st_shared_v2(sb + S_KQ + off + 8192, h0, h1);
                    st_shared_v2(sb + S_KQ + off + 8192 + 16384, lo0, lo1);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(tiles_bar);
            // the next chunk's q and k, in flight while the Kg^T rows wait for their tile
            if (ch + 1 < nchunks) load_qk(ch + 1);
            // ---- the Kg^T rows, once the chain's previous O/S product has read the tile
            if (ch > 0 && !mbar_wait(bar_s, (uint32_t)((ch - 1) & 1), kPolls)) failed = 1;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float x[4][4];
#pragma unroll
                for (int t = 0; t < 4; ++t)
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[t][e] = kgv[4 * half + t][e];
                st_kgt(sb + S_PKGH, sb + S_PKGL, l4, pw * 8 + 4 * half, x);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(kg_bar);
        }
    }
    failed = __syncthreads_or(failed);

    if (failed) {
        if (tid == 0) {
            atomicAdd(&g_chunk_chain_timeouts, 1);
            mma_commit(drain_bar);  // arrives once the tensor-core work already issued has drained
            if (v_pending >= 0) mbar_wait(v_bar, (uint32_t)(v_pending & 1), kPolls);
            if (tb_pending >= 0) mbar_wait(tb_bar, (uint32_t)(tb_pending & 1), kPolls);
            if (p_pending >= 0) mbar_wait(p_bar, (uint32_t)(p_pending & 1), kPolls);
            if (q_pending >= 0) mbar_wait(gate_bar, (uint32_t)(q_pending & 1), kPolls);
        }
        if (tid == 256 && g_pending >= 0) mbar_wait(g_bar, (uint32_t)(g_pending & 1), kPolls);
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
        const int c0 = (warp >> 2) * 32, mm = (warp & 3) * 32 + lane;
        tmem_ld16(tb + lane_off + T_S + c0, s1);
        tmem_ld16(tb + lane_off + T_S + c0 + 16, s2);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            p.sT[((size_t)unit * DK + c0 + c) * DV + mm] = __uint_as_float(s1[c]);
            p.sT[((size_t)unit * DK + c0 + 16 + c) * DV + mm] = __uint_as_float(s2[c]);
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
