// kda_chunk_tc.cu -- chunked KDA prefill on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (a prompt runs a
// chunked kernel that carries the state from one 64-token chunk to the next and
// never holds it per token), sections 03/04 (per-key-channel decay applied before
// each delta-rule update, q and k L2-normalised in the kernel, q scaled by
// 1/sqrt(key_dim)); Kimi-K3 atlas "gate-project (decode, P = 1000)" for the fused
// sigmoid-gated RMSNorm epilogue.
//
// Chunk algebra (derived from the recurrence, exact in real arithmetic).  For one
// (sequence, head) and a chunk of C = 64 tokens entering with state S [K x V]:
//   G_i = sum_{s<=i} g_s (inclusive, per key channel), gamma = G_{C-1}
//   Kd = k^ exp(G), Qd = q^ exp(G), Kg = k^ exp(gamma - G), Km = k^ exp(-G)
//   A = strict_lower(diag(beta) Kd Km^T),  P = lower(Qd Km^T)          (grams)
//   T = (I + A)^-1,  W = T diag(beta) Kd,  U = T diag(beta) V          (WY/UT form)
//   D = U - W S,  O = Qd S + P D,  S' = Diag(exp gamma) S + Kg^T D
// Km carries exp(-G) >= 1: it stays finite while the chunk's decay range
// max_c(-gamma[c]) <= 80.  Chunks beyond that (g near the -5 lower bound on many
// tokens) compute A and P exactly on CUDA cores with pairwise exponentials instead.
//
// Precision: every contraction runs on the tensor cores with bf16 operands split
// into hi + lo parts (x = hi + lo, three MMAs hi*hi + hi*lo + lo*hi, fp32
// accumulation), about 16 significant bits per operand; U uses two MMAs because v
// is an exact bf16 input.  Plain bf16 operands miss the 5e-3 max-error bound by an
// order of magnitude, plain tf32 sits right at it.
//
// Mapping: one CTA of 16 warps per (sequence, head).  Everything is transposed so
// that the value dimension (128) is the MMA M dimension and TMEM lane:
//   TMEM columns   [0,128)  S^T fp32 accumulator (lane v, column c)
//                [128,192)  S^T hi, packed bf16 pairs (A operand of the state MMAs)
//                [192,256)  S^T lo
//                [256,320)  D^T accumulator (U^T then - S^T W^T)
//                [320,384)  O^T accumulator
//                [384,448)  gram accumulator [A ; P] (lanes 0-63 / 64-127), then
//                           D^T hi [384,416) and D^T lo [416,448)
//                [448,512)  W^T accumulator (lane c, column i)
//   per chunk:  gram     [Kd;Qd] Km^T           M=128 N=64  K=128
//               W^T    = Kd^T (T diag beta)^T   M=128 N=64  K=64
//               U^T    = V^T (T diag beta)^T    M=128 N=64  K=64   (V tile by TMA)
//               D^T   += S^T (-W^T)             M=128 N=64  K=128  (A from TMEM)
//               O^T    = S^T Qd^T               M=128 N=64  K=128  (A from TMEM)
//               O^T   += D^T P^T                M=128 N=64  K=64   (A from TMEM)
//               S^T    = S^T Diag(exp gamma) + D^T Kg   M=128 N=128 K=64
// The triangular inverse runs on CUDA cores (blocked, 16 x 16 diagonal blocks).
#include <cuda.h>
#include <math.h>
#include <string.h>

#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = 64;         // tokens per chunk
constexpr int DK = 128;       // key dim
constexpr int DV = 128;       // value dim
constexpr int kThreads = 512; // 16 warps = 4 warpgroups
constexpr float kRangeMax = 80.f;
constexpr uint32_t kPolls = 1u << 26;  // bound on every mbarrier wait

// TMEM columns
constexpr uint32_t T_S = 0, T_SH = 128, T_SL = 192, T_D = 256, T_O = 320, T_G = 384, T_DH = 384, T_DL = 416,
                   T_W = 448;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_V = 0;             // V tile, two TMA boxes of 64 tokens x 64 values (16 KB)
constexpr uint32_t S_KQH = 16384;       // [Kd ; Qd] hi, 128 rows x 128 (32 KB)
constexpr uint32_t S_KQL = 49152;       // [Kd ; Qd] lo
constexpr uint32_t S_KMH = 81920;       // Km hi (then Kg hi), 64 rows x 128 (16 KB)
constexpr uint32_t S_KML = 98304;       // Km lo (then Kg lo)
constexpr uint32_t S_TBH = 114688;      // T diag(beta) hi, 64 x 64 (8 KB)
constexpr uint32_t S_TBL = 122880;
constexpr uint32_t S_PH = 131072;       // P hi 64 x 64
constexpr uint32_t S_PL = 139264;
constexpr uint32_t S_WH = 147456;       // W, rows c x 64 i (16 KB)
constexpr uint32_t S_WL = 163840;
constexpr int AP = 68;                  // fp32 pitch of A and T
constexpr uint32_t S_A = 180224;        // A fp32 [64][AP] (17408 B)
constexpr uint32_t S_T = S_A + 64 * AP * 4;  // T fp32 [64][AP]
constexpr uint32_t S_SMALL = S_T + 64 * AP * 4;
// small buffers (floats)
constexpr uint32_t F_GEXP = 0;    // exp(gamma)   [128]
constexpr uint32_t F_GNEG = 128;  // exp(-gamma)  [128]
constexpr uint32_t F_GAM = 256;   // gamma        [128]
constexpr uint32_t F_BETA = 384;  // beta         [64]
constexpr uint32_t F_RQ = 448;    // q scale per token (norm * scale) [64]
constexpr uint32_t F_RK = 512;    // k norm per token [64]
constexpr uint32_t F_RED = 576;   // norm partials [4 wg][4 quarters][16]
constexpr uint32_t F_END = 832;
constexpr uint32_t S_BARS = S_SMALL + F_END * 4;   // 2 mbarriers + tmem slot + flags
constexpr uint32_t SMEM_BYTES = S_BARS + 64 + 1024;  // + alignment slack
// scan scratch aliases T (free during prep): [16 warps][128] floats
constexpr uint32_t S_SCAN = S_T;
// fallback scratch (only for chunks beyond the decay range): G fp32 [64][128] in the
// W tiles, raw q and k bf16 [64][128] in the T diag(beta) and Km hi tiles
constexpr uint32_t S_FB_G = S_WH, S_FB_Q = S_TBH, S_FB_K = S_KMH;

static_assert(S_A % 16 == 0 && S_SMALL % 16 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Set by a CTA whose bounded wait on the tensor core or the TMA gave up; that CTA
// also writes NaN into its final state so the failure cannot pass unnoticed.
__device__ int g_chunk_tc_timeouts = 0;

struct TcParams {
    SeqParams p;
    int order_n;            // > 0: blockIdx -> sequence through order[]
    int order[64];
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Writes 4 consecutive columns (col % 4 == 0) of one row of a SW128 tile as hi/lo.
__device__ __forceinline__ void st_tile4(uint32_t hi_base, uint32_t lo_base, uint32_t rows, uint32_t row,
                                         uint32_t col, float a, float b, float c, float d) {
    uint32_t h0, l0, h1, l1;
    split2(a, b, h0, l0);
    split2(c, d, h1, l1);
    const uint32_t off = sw128_off(row, col, rows);
    st_shared_v2(hi_base + off, h0, h1);
    st_shared_v2(lo_base + off, l0, l1);
}

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

__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ TcParams tp) {
    const SeqParams &p = tp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    float *fs = reinterpret_cast<float *>(sm + S_SMALL);
    float *Asm = reinterpret_cast<float *>(sm + S_A);
    float *Tsm = reinterpret_cast<float *>(sm + S_T);
    uint64_t *mma_bar = reinterpret_cast<uint64_t *>(sm + S_BARS);
    uint64_t *tma_bar = mma_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_BARS + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, wq = warp & 3;
    const int m = wq * 32 + lane;  // TMEM lane this thread reads/writes
    const int H = p.H;
    int n = blockIdx.x / H;
    const int h = blockIdx.x % H;
    if (tp.order_n > 0) n = tp.order[n];
    const int unit = n * H + h;
    int bos, len;
    seq_range(p, n, bos, len);

    if (tid == 0) {
        mbar_init(mma_bar, 1);
        mbar_init(tma_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    uint32_t mma_phase = 0, tma_phase = 0;
    bool failed = false;

    // ---- initial state -> S^T accumulator and its hi/lo operand copy
    {
        const int c0 = wg * 32;
        float s[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
            s[c] = p.s0 ? p.s0[((size_t)unit * DK + c0 + c) * DV + m] : 0.f;
        uint32_t r[16], hi[16], lo[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int c = 0; c < 16; ++c) r[c] = __float_as_uint(s[half * 16 + c]);
            tmem_st16(tb + lane_off + T_S + c0 + half * 16, r);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) split2(s[2 * c], s[2 * c + 1], hi[c], lo[c]);
        tmem_st16(tb + lane_off + T_SH + c0 / 2, hi);
        tmem_st16(tb + lane_off + T_SL + c0 / 2, lo);
        tmem_wait_st();
    }

    const int nchunks = (len + C - 1) / C;
    auto issue_v = [&](int chunk) {
        mbar_arrive_expect_tx(tma_bar, 16384);
        tma_load_3d(sb + S_V, &tmap_v, tma_bar, 0, h, bos + chunk * C);
        tma_load_3d(sb + S_V + 8192, &tmap_v, tma_bar, 64, h, bos + chunk * C);
    };
    if (tid == 0 && nchunks > 0) issue_v(0);

    // all threads wait on the MMA barrier; a timeout marks the CTA failed
    auto mma_wait = [&]() {
        const bool ok = mbar_wait(mma_bar, mma_phase, kPolls);
        mma_phase ^= 1;
        fence_after_sync();
        return ok;
    };

    for (int ch = 0; ch < nchunks && !failed; ++ch) {
        const int t0 = ch * C;
        const int cn = min(C, len - t0);
        // ================= prep: loads, norms, cumulative decay, operand tiles
        const int l4 = lane * 4;  // this thread's 4 key channels
        float g4[4][4], q4[4][4], k4[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = warp * 4 + r;
            const bool valid = i < cn;
            const size_t hk = ((size_t)(bos + t0 + i) * H + h) * DK + l4;
            float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);
            uint2 qv = make_uint2(0u, 0u), kv = make_uint2(0u, 0u);
            if (valid) {
                gv = __ldg(reinterpret_cast<const float4 *>(p.g + hk));
                qv = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) + hk));
                kv = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.k) + hk));
            }
            g4[r][0] = gv.x; g4[r][1] = gv.y; g4[r][2] = gv.z; g4[r][3] = gv.w;
            q4[r][0] = bf16lo(qv.x); q4[r][1] = bf16hi(qv.x); q4[r][2] = bf16lo(qv.y); q4[r][3] = bf16hi(qv.y);
            k4[r][0] = bf16lo(kv.x); k4[r][1] = bf16hi(kv.x); k4[r][2] = bf16lo(kv.y); k4[r][3] = bf16hi(kv.y);
        }
        float rq[4], rk[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float aq = 0.f, ak = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                aq = fmaf(q4[r][c], q4[r][c], aq);
                ak = fmaf(k4[r][c], k4[r][c], ak);
            }
            aq = warp_sum(aq);
            ak = warp_sum(ak);
            rq[r] = (p.l2norm ? rsqrtf(aq + 1e-6f) : 1.f) * p.scale;
            rk[r] = p.l2norm ? rsqrtf(ak + 1e-6f) : 1.f;
        }
        if (lane < 4) {
            const int i = warp * 4 + lane;
            fs[F_BETA + i] = (i < cn) ? p.beta[(size_t)(bos + t0 + i) * H + h] : 0.f;
            fs[F_RQ + i] = rq[lane];
            fs[F_RK + i] = rk[lane];
        }
        // local inclusive prefix over the thread's 4 tokens; warp totals to the scan buffer
#pragma unroll
        for (int r = 1; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) g4[r][c] += g4[r - 1][c];
        float *scan = reinterpret_cast<float *>(sm + S_SCAN);
        *reinterpret_cast<float4 *>(scan + warp * 128 + l4) = make_float4(g4[3][0], g4[3][1], g4[3][2], g4[3][3]);
        __syncthreads();
        if (tid < 128) {  // exclusive scan of the 16 warp totals, per channel
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float t = scan[w * 128 + tid];
                scan[w * 128 + tid] = acc;
                acc += t;
            }
            fs[F_GAM + tid] = acc;
            fs[F_GEXP + tid] = __expf(acc);
            fs[F_GNEG + tid] = __expf(-acc);
        }
        const int fallback = __syncthreads_or(tid < 128 && -fs[F_GAM + tid] > kRangeMax ? 1 : 0);
        // (the predicate above reads gamma written before the barrier by the same thread)
        float kg[4][4];
        {
            const float4 off = *reinterpret_cast<const float4 *>(scan + warp * 128 + l4);
            const float4 gam = *reinterpret_cast<const float4 *>(fs + F_GAM + l4);
            const float4 gneg = *reinterpret_cast<const float4 *>(fs + F_GNEG + l4);
            const float offs[4] = {off.x, off.y, off.z, off.w};
            const float gams[4] = {gam.x, gam.y, gam.z, gam.w};
            const float gnegs[4] = {gneg.x, gneg.y, gneg.z, gneg.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = warp * 4 + r;
                float kd[4], qd[4], km[4], G[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    G[c] = offs[c] + g4[r][c];
                    const float eG = __expf(G[c]);
                    const float kh = k4[r][c] * rk[r], qh = q4[r][c] * rq[r];
                    kd[c] = kh * eG;
                    qd[c] = qh * eG;
                    kg[r][c] = kh * __expf(gams[c] - G[c]);
                    km[c] = kg[r][c] * gnegs[c];
                }
                st_tile4(sb + S_KQH, sb + S_KQL, 128, i, l4, kd[0], kd[1], kd[2], kd[3]);
                st_tile4(sb + S_KQH, sb + S_KQL, 128, 64 + i, l4, qd[0], qd[1], qd[2], qd[3]);
                if (!fallback) {
                    st_tile4(sb + S_KMH, sb + S_KML, 64, i, l4, km[0], km[1], km[2], km[3]);
                } else {
                    float *Gs = reinterpret_cast<float *>(sm + S_FB_G);
                    *reinterpret_cast<float4 *>(Gs + i * 128 + l4) = make_float4(G[0], G[1], G[2], G[3]);
                    __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(sm + S_FB_Q);
                    __nv_bfloat16 *ks = reinterpret_cast<__nv_bfloat16 *>(sm + S_FB_K);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        qs[i * 128 + l4 + c] = __float2bfloat16_rn(q4[r][c]);  // exact: inputs are bf16
                        ks[i * 128 + l4 + c] = __float2bfloat16_rn(k4[r][c]);
                    }
                }
            }
        }
        fence_async_smem();
        __syncthreads();

        // ================= grams A (strict lower, beta-scaled) and P (lower)
        if (!fallback) {
            if (tid == 0) {
                fence_after_sync();
                const uint32_t idesc = idesc_bf16(128, 64, false, false);
                const uint32_t ah[2] = {sb + S_KQH, sb + S_KQL}, bh[2] = {sb + S_KMH, sb + S_KML};
                const int combos[3][2] = {{0, 0}, {0, 1}, {1, 0}};
                int first = 1;
                for (int cb = 0; cb < 3; ++cb)
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t koff = (s >> 2) * 0u + (s & 3) * 32u;
                        const uint64_t ad = sdesc(ah[combos[cb][0]] + (s >> 2) * 16384 + koff, 16, 1024);
                        const uint64_t bd = sdesc(bh[combos[cb][1]] + (s >> 2) * 8192 + koff, 16, 1024);
                        mma_ss(tb + T_G, ad, bd, idesc, first ? 0u : 1u);
                        first = 0;
                    }
                mma_commit(mma_bar);
            }
            __syncwarp();
            if (__syncthreads_or(!mma_wait())) { failed = true; break; }
            {
                uint32_t r[16];
                tmem_ld16(tb + lane_off + T_G + wg * 16, r);
                tmem_wait_ld();
                const int j0 = wg * 16;
                if (m < 64) {
                    const int i = m;
                    const float b = fs[F_BETA + i];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        Asm[i * AP + j0 + c] = (j0 + c < i) ? b * __uint_as_float(r[c]) : 0.f;
                } else {
                    const int i = m - 64;
                    float x[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) x[c] = (j0 + c <= i) ? __uint_as_float(r[c]) : 0.f;
                    st_tile8(sb + S_PH, sb + S_PL, 64, i, j0, x);
                    st_tile8(sb + S_PH, sb + S_PL, 64, i, j0 + 8, x + 8);
                }
            }
        } else {
            // exact grams with pairwise exponentials (decay range too wide for Km)
            const float *Gs = reinterpret_cast<const float *>(sm + S_FB_G);
            const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm + S_FB_Q);
            const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(sm + S_FB_K);
            float *Pf = Tsm;  // P in fp32, converted to the tile below
            for (int pr = warp; pr < C * C; pr += 16) {
                const int i = pr >> 6, j = pr & 63;
                float a = 0.f, b = 0.f;
                if (j <= i) {
                    for (int c = lane; c < DK; c += 32) {
                        const float e = __expf(Gs[i * 128 + c] - Gs[j * 128 + c]);
                        const float kj = __bfloat162float(ks[j * 128 + c]) * e;
                        a = fmaf(__bfloat162float(ks[i * 128 + c]), kj, a);
                        b = fmaf(__bfloat162float(qs[i * 128 + c]), kj, b);
                    }
                    a = warp_sum(a) * fs[F_RK + i] * fs[F_RK + j];
                    b = warp_sum(b) * fs[F_RQ + i] * fs[F_RK + j];
                }
                if (lane == 0) {
                    Asm[i * AP + j] = (j < i) ? fs[F_BETA + i] * a : 0.f;
                    Pf[i * AP + j] = (j <= i) ? b : 0.f;
                }
            }
            __syncthreads();
            {
                const int i = tid >> 3, j0 = (tid & 7) * 8;
                float x[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) x[c] = Pf[i * AP + j0 + c];
                st_tile8(sb + S_PH, sb + S_PL, 64, i, j0, x);
            }
            __syncthreads();
        }
        // Kg into the Km tiles (the gram that read Km has completed)
#pragma unroll
        for (int r = 0; r < 4; ++r)
            st_tile4(sb + S_KMH, sb + S_KML, 64, warp * 4 + r, lane * 4, kg[r][0], kg[r][1], kg[r][2], kg[r][3]);
        __syncthreads();

        // ================= T = (I + A)^-1, blocked with 16 x 16 diagonal blocks
        if (tid < 64) {
            const int b = tid >> 4, c = tid & 15, o = 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) acc = fmaf(Asm[(o + i) * AP + o + j], x[j], acc);
                x[i] = (i < c) ? 0.f : (i == c ? 1.f : -acc);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tsm[(o + i) * AP + o + c] = x[i];
        }
        __syncthreads();
        for (int d = 1; d < 4; ++d) {
            const int np = 4 - d;
            for (int it = tid; it < np * 256; it += kThreads) {  // X = sum_K A_IK T_KJ -> A's upper block (J, I)
                const int I = d + (it >> 8), J = I - d, e = it & 255, r = e >> 4, cc = e & 15;
                float acc = 0.f;
                for (int Kb = J; Kb < I; ++Kb)
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        acc = fmaf(Asm[(16 * I + r) * AP + 16 * Kb + t], Tsm[(16 * Kb + t) * AP + 16 * J + cc], acc);
                Asm[(16 * J + r) * AP + 16 * I + cc] = acc;
            }
            __syncthreads();
            for (int it = tid; it < np * 256; it += kThreads) {  // T_IJ = -T_II X
                const int I = d + (it >> 8), J = I - d, e = it & 255, r = e >> 4, cc = e & 15;
                float acc = 0.f;
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    acc = fmaf(Tsm[(16 * I + r) * AP + 16 * I + t], Asm[(16 * J + t) * AP + 16 * I + cc], acc);
                Tsm[(16 * I + r) * AP + 16 * J + cc] = -acc;
            }
            __syncthreads();
        }
        {  // T diag(beta) -> hi/lo tile (rows i, K = j)
            const int i = tid >> 3, j0 = (tid & 7) * 8;
            float x[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = (j0 + c <= i) ? Tsm[i * AP + j0 + c] * fs[F_BETA + j0 + c] : 0.f;
            st_tile8(sb + S_TBH, sb + S_TBL, 64, i, j0, x);
        }
        fence_async_smem();
        __syncthreads();

        // ================= W^T = Kd^T (T diag beta)^T ; U^T = V^T (T diag beta)^T
        if (tid == 0) {
            const bool v_ok = mbar_wait(tma_bar, tma_phase, kPolls);
            if (!v_ok) failed = true;
            fence_after_sync();
            const uint32_t idesc_w = idesc_bf16(128, 64, true, false);
            const uint32_t kq[2] = {sb + S_KQH, sb + S_KQL}, tbt[2] = {sb + S_TBH, sb + S_TBL};
            const int combos[3][2] = {{0, 0}, {0, 1}, {1, 0}};
            int first = 1;
            for (int cb = 0; cb < 3; ++cb)
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ad = sdesc(kq[combos[cb][0]] + s * 2048, 16384, 1024);
                    const uint64_t bd = sdesc(tbt[combos[cb][1]] + s * 32, 16, 1024);
                    mma_ss(tb + T_W, ad, bd, idesc_w, first ? 0u : 1u);
                    first = 0;
                }
            first = 1;
            for (int cb = 0; cb < 2; ++cb)
                for (int s = 0; s < 4; ++s) {
                    const uint64_t ad = sdesc(sb + S_V + s * 2048, 8192, 1024);
                    const uint64_t bd = sdesc(tbt[cb] + s * 32, 16, 1024);
                    mma_ss(tb + T_D, ad, bd, idesc_w, first ? 0u : 1u);
                    first = 0;
                }
            mma_commit(mma_bar);
        }
        tma_phase ^= 1;
        __syncwarp();
        if (__syncthreads_or(!mma_wait() || failed)) { failed = true; break; }
        if (tid == 0 && ch + 1 < nchunks) issue_v(ch + 1);  // V tile is free again

        // ================= W pass: W^T (lane c, column i) -> W tile (rows c, 64 i)
        {
            uint32_t r[16];
            tmem_ld16(tb + lane_off + T_W + wg * 16, r);
            tmem_wait_ld();
            float x[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) x[c] = __uint_as_float(r[c]);
            st_tile8(sb + S_WH, sb + S_WL, 128, m, wg * 16, x);
            st_tile8(sb + S_WH, sb + S_WL, 128, m, wg * 16 + 8, x + 8);
        }
        fence_async_smem();
        fence_before_sync();
        __syncthreads();

        // ================= D^T += S^T (-W^T) ; O^T = S^T Qd^T
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idesc_d = idesc_bf16(128, 64, false, true, false, true);  // B = W, MN-major, negated
            const uint32_t idesc_o = idesc_bf16(128, 64, false, false);
            const uint32_t sa[2] = {tb + T_SH, tb + T_SL};
            const uint32_t wt[2] = {sb + S_WH, sb + S_WL}, kq[2] = {sb + S_KQH, sb + S_KQL};
            const int combos[3][2] = {{0, 0}, {0, 1}, {1, 0}};
            for (int cb = 0; cb < 3; ++cb)
                for (int s = 0; s < 8; ++s) {
                    const uint64_t bd = sdesc(wt[combos[cb][1]] + s * 2048, 8192, 1024);
                    mma_ts(tb + T_D, sa[combos[cb][0]] + s * 8, bd, idesc_d, 1u);
                }
            int first = 1;
            for (int cb = 0; cb < 3; ++cb)
                for (int s = 0; s < 8; ++s) {
                    const uint64_t bd = sdesc(kq[combos[cb][1]] + 8192 + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024);
                    mma_ts(tb + T_O, sa[combos[cb][0]] + s * 8, bd, idesc_o, first ? 0u : 1u);
                    first = 0;
                }
            mma_commit(mma_bar);
        }
        __syncwarp();
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }

        // ================= D pass (hi/lo into TMEM) and S decay by exp(gamma)
        {
            uint32_t r[16], hi[8], lo[8];
            tmem_ld16(tb + lane_off + T_D + wg * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) split2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]), hi[c], lo[c]);
            tmem_st8(tb + lane_off + T_DH + wg * 8, hi);
            tmem_st8(tb + lane_off + T_DL + wg * 8, lo);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c0 = wg * 32 + half * 16;
                tmem_ld16(tb + lane_off + T_S + c0, r);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * fs[F_GEXP + c0 + c]);
                tmem_st16(tb + lane_off + T_S + c0, r);
            }
            tmem_wait_st();
        }
        fence_before_sync();
        __syncthreads();

        // ================= O^T += D^T P^T ; S^T += D^T Kg
        if (tid == 0) {
            fence_after_sync();
            const uint32_t idesc_p = idesc_bf16(128, 64, false, false);
            const uint32_t idesc_s = idesc_bf16(128, 128, false, true);
            const uint32_t da[2] = {tb + T_DH, tb + T_DL};
            const uint32_t pt[2] = {sb + S_PH, sb + S_PL}, kgt[2] = {sb + S_KMH, sb + S_KML};
            const int combos[3][2] = {{0, 0}, {0, 1}, {1, 0}};
            for (int cb = 0; cb < 3; ++cb)
                for (int s = 0; s < 4; ++s) {
                    mma_ts(tb + T_O, da[combos[cb][0]] + s * 8, sdesc(pt[combos[cb][1]] + s * 32, 16, 1024), idesc_p, 1u);
                    mma_ts(tb + T_S, da[combos[cb][0]] + s * 8, sdesc(kgt[combos[cb][1]] + s * 2048, 8192, 1024),
                           idesc_s, 1u);
                }
            mma_commit(mma_bar);
        }
        __syncwarp();
        if (__syncthreads_or(!mma_wait())) { failed = true; break; }

        // ================= O pass (+ gated norm) and state pass
        {
            uint32_t r[16];
            tmem_ld16(tb + lane_off + T_O + wg * 16, r);
            tmem_wait_ld();
            const int v = m;
            const int i0 = wg * 16;
            if (p.gate) {
                float* red = fs + F_RED;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float x = __uint_as_float(r[c]);
                    const float s2 = warp_sum(x * x);
                    if (lane == 0) red[(wg * 4 + wq) * 16 + c] = s2;
                }
                __syncthreads();
                const float w = p.norm_w[v];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int i = i0 + c;
                    if (i < cn) {
                        const float ss = red[(wg * 4 + 0) * 16 + c] + red[(wg * 4 + 1) * 16 + c] +
                                         red[(wg * 4 + 2) * 16 + c] + red[(wg * 4 + 3) * 16 + c];
                        const float inv = rsqrtf(ss * (1.f / DV) + p.eps);
                        const size_t idx = ((size_t)(bos + t0 + i) * H + h) * DV + v;
                        const float x = __uint_as_float(r[c]);
                        const float gt = ld_in(p.gate, idx, p.gate_bf16);
                        st_out(p.y, idx, x * inv * w * sigmoidf_(gt), p.o_bf16);
                        if (p.o) st_out(p.o, idx, x, p.o_bf16);
                    }
                }
            } else if (p.o) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int i = i0 + c;
                    if (i < cn) st_out(p.o, ((size_t)(bos + t0 + i) * H + h) * DV + v, __uint_as_float(r[c]), p.o_bf16);
                }
            }
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld16(tb + lane_off + T_S + wg * 32 + half * 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    split2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]), hi[half * 8 + c], lo[half * 8 + c]);
            }
            tmem_st16(tb + lane_off + T_SH + wg * 16, hi);
            tmem_st16(tb + lane_off + T_SL + wg * 16, lo);
            tmem_wait_st();
        }
        fence_before_sync();
        __syncthreads();
    }

    if (failed) {
        if (tid == 0) {
            atomicAdd(&g_chunk_tc_timeouts, 1);
            mma_commit(mma_bar);  // arrives once the tensor-core work already issued has drained
        }
        mbar_wait(mma_bar, mma_phase, kPolls);
        if (p.sT)
            for (int e = tid; e < DK * DV; e += kThreads) p.sT[(size_t)unit * DK * DV + e] = __int_as_float(0x7fc00000);
    } else if (p.sT) {  // final state: S[c][v] from S^T (lane v, column c)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t r[16];
            const int c0 = wg * 32 + half * 16;
            tmem_ld16(tb + lane_off + T_S + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) p.sT[((size_t)unit * DK + c0 + c) * DV + m] = __uint_as_float(r[c]);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace

bool chunk_tc_supported(int K, int V, int chunk) { return K == DK && V == DV && chunk == C; }

kda_status launch_chunk_tc(const SeqParams &p_in, int K, int V, int chunk, cudaStream_t st) {
    if (!chunk_tc_supported(K, V, chunk)) {
        set_error("chunk_tc: needs K = V = 128 and chunk = 64");
        return KDA_ERR_UNSUPPORTED;
    }
    const int units = p_in.N * p_in.H;
    if (units == 0) return KDA_OK;
    const long long rows = p_in.cu_seqlens ? (long long)p_in.T : (long long)p_in.N * p_in.T;
    if (rows <= 0) {
        set_error("chunk_tc: no tokens (use the fp32 path for empty prompts)");
        return KDA_ERR_UNSUPPORTED;
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        set_error("chunk_tc: cuTensorMapEncodeTiled is not available from the driver");
        return KDA_ERR_CUDA;
    }
    CUtensorMap tmap;
    const cuuint64_t dims[3] = {(cuuint64_t)DV, (cuuint64_t)p_in.H, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)DV * 2, (cuuint64_t)p_in.H * DV * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult cr = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p_in.v), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        set_error("chunk_tc: cuTensorMapEncodeTiled failed (%d)", (int)cr);
        return KDA_ERR_CUDA;
    }
    TcParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.p = p_in;
    // longest sequences first when the host copy of cu_seqlens is known
    if (p_in.cu_seqlens && p_in.cu_host && p_in.N <= 64) {
        tp.order_n = p_in.N;
        for (int i = 0; i < p_in.N; ++i) tp.order[i] = i;
        for (int i = 1; i < p_in.N; ++i) {  // insertion sort by length, descending
            const int x = tp.order[i];
            const int lx = p_in.cu_host[x + 1] - p_in.cu_host[x];
            int j = i - 1;
            while (j >= 0 && p_in.cu_host[tp.order[j] + 1] - p_in.cu_host[tp.order[j]] < lx) {
                tp.order[j + 1] = tp.order[j];
                --j;
            }
            tp.order[j + 1] = x;
        }
    }
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) {
            set_error("chunk_tc: cannot reserve %u bytes of shared memory: %s", SMEM_BYTES, cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
        configured = true;
    }
    chunk_tc_kernel<<<units, kThreads, SMEM_BYTES, st>>>(tmap, tp);
    note_launch();
    return check_launch("chunk_tc_kernel");
}

}  // namespace kda
