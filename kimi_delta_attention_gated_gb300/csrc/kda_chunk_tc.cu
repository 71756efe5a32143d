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
//   Kd = k^ exp(G), Qd = q^ exp(G), Km = k^ exp(-G), Kg = k^ exp(gamma - G)
//   A = strict_lower(diag(beta) Kd Km^T),  P = lower(Qd Km^T)          (grams)
//   T = (I + A)^-1                                                    (UT transform)
//   R = V - Kd S,  D = T diag(beta) R   (= U - W S of the WY form, reassociated)
//   O = Qd S + P D,  S' = Diag(exp gamma) S + Kg^T D
// Km carries exp(-G) >= 1 and stays finite while the chunk's decay range
// max_c(-gamma[c]) <= 80.  Chunks beyond it (g near the -5 lower bound on many
// tokens) compute A and P exactly on CUDA cores with pairwise exponentials.
//
// Precision: every contraction runs on the tensor cores with bf16 operands split
// into hi + lo parts (x = hi + lo, three products hi*hi + hi*lo + lo*hi, fp32
// accumulation), about 16 significant bits per operand.  V enters R through an MMA
// with a bf16 identity (exact).  Plain bf16 operands miss the 5e-3 max-error bound
// by an order of magnitude; plain tf32 sits right at it.
//
// Mapping: one CTA of 16 warps per (sequence, head); thread 0 issues the TMA and
// every tcgen05.mma.  A dependent M=128 MMA costs about 100 cycles whatever its N up
// to 128, so the products are stacked along N (fewer, wider instructions), and the
// R/O product is issued while warps 1-15 run the triangular solve (thread 0's warp
// stalls on the MMA queue meanwhile).  Everything is transposed so that the value
// dimension (128) is the MMA M dimension and the TMEM lane:
//   TMEM columns   [0,64)   R^T accumulator, then R^T hi/lo in place: for tokens
//                           16b..16b+15, hi in [16b, 16b+8) and lo in [16b+8, 16b+16)
//                 [64,128)  O^T accumulator
//                [128,256)  S^T fp32 accumulator (lane v, column c)
//                [256,320)  S^T hi, packed bf16 pairs (A operand of the state MMAs)
//                [320,384)  S^T lo
//                [384,512)  gram accumulator: [hi*hi + lo*hi | hi*lo]; then the D^T
//                           accumulator [hi*(hi;lo) + lo*hi | ...], summed into D^T hi/lo
//                           in place in [384,448) with the layout of R^T
//   per chunk (B operands in shared memory are K-major unless noted):
//     gram   [-Kd;Qd] [Km_hi;Km_lo]^T  M=128 N=128 K=128, + [-Kd;Qd]_lo Km_hi^T N=64
//     R^T  = V^T I (N=64), then [R|O]^T += S^T [-Kd;Qd]^T   N=128 K=128 (S^T in TMEM)
//       ... meanwhile on CUDA cores: gram pass, T = (I + A)^-1, T diag(beta) tile
//     D^T  = R^T (T diag beta)^T   N=128 (hi against both halves) + N=64, K=64 (R^T in TMEM)
//     [O|S]^T += D^T [P^T | Kg]  (S^T pre-scaled by exp(gamma))  N=192 K=64
// The next chunk's q and k are loaded into registers and its g (or logits) arrives by
// TMA while the current one runs; its CUDA-core preparation (norms, cumulative decay,
// operand tiles) is done while this chunk's D and [O|S] products run on the tensor
// cores.  Warp 0, which issues every product and stalls behind the tensor core's queue
// meanwhile, prepares its own tokens' norms during the solve instead (g and beta given).
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

constexpr int kThreads = 512;    // 16 warps = 4 warpgroups

// TMEM columns
constexpr uint32_t T_R = 0, T_O = 64, T_S = 128, T_SH = 256, T_SL = 320, T_G = 384;

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t S_V = 0;             // V tile, two TMA boxes of 64 tokens x 64 values (16 KB)
constexpr uint32_t S_KQH = 16384;       // [-Kd ; Qd] hi, 128 rows x 128 (32 KB)
constexpr uint32_t S_KQL = 49152;       // [-Kd ; Qd] lo
constexpr uint32_t S_KM = 81920;        // [Km hi ; Km lo], 128 rows x 128 (32 KB)
constexpr uint32_t S_PKGH = 114688;     // [P ; Kg^T] hi, 192 rows (i, then c) x 64 (j) (24 KB), K-major B
constexpr uint32_t S_PKGL = 139264;     // [P ; Kg^T] lo
constexpr uint32_t S_TBH = 163840;      // T diag(beta) hi, 64 x 64 (8 KB)
constexpr uint32_t S_TBL = 172032;
constexpr uint32_t S_ID = 180224;       // bf16 identity 64 x 64 (8 KB)
constexpr uint32_t S_A = 188416;        // A fp32 [64][AP] (17408 B)
constexpr uint32_t S_T = S_A + 64 * AP * 4;  // T fp32 [64][AP]
constexpr uint32_t S_SMALL = S_T + 64 * AP * 4;
// small buffers (floats)
constexpr uint32_t F_BETA = 0;    // beta [64]
constexpr uint32_t F_RQ = 64;     // q scale per token (norm * scale) [64]
constexpr uint32_t F_RK = 128;    // k norm per token [64]
constexpr uint32_t F_GEXP = 192;  // exp(gamma) [128]
constexpr uint32_t F_RED = 320;   // norm partials [4 wg][4 quarters][16]
constexpr uint32_t F_BETA0 = 576; // beta of tokens 0-3 (warp 0 prepares them while the solve reads F_BETA)
constexpr uint32_t F_SCAN0 = 580; // decay totals of tokens 0-3 [128]
constexpr uint32_t F_AH = 708;    // gates from logits: exp(A_log) of the head [1 of 4]
constexpr uint32_t F_DB = 712;    // gates from logits: dt_bias of the head's channels [128]
constexpr uint32_t F_BLOB = 840;  // concurrent form: this chunk's blob is ready (thread 0 -> all)
constexpr uint32_t F_END = 844;
constexpr uint32_t S_BARS = S_SMALL + F_END * 4;     // 8 mbarriers, tmem slot, gate and blob mbarriers
constexpr uint32_t SMEM_BYTES = S_BARS + 96 + 1024;  // + alignment slack
// scan scratch aliases T (free during prep): [16 warps][128] floats of decay totals, then
// their exclusive prefixes [16][128] and the chunk total [128]
constexpr uint32_t S_SCAN = S_T;
// fallback scratch: G fp32 [64][128] in the Km tile (Km is not used then)
constexpr uint32_t S_FB_G = S_KM;

static_assert(S_A % 1024 == 0 && S_SMALL % 16 == 0, "alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Set by a CTA whose bounded wait on the tensor core or the TMA gave up; that CTA
// also writes NaN into its final state, o and y so the failure cannot pass unnoticed.
// The waits on copies from global memory (the V, g and gate tiles, a pre-pass blob) take
// the caller's bound (SeqParams::polls, kda_set_wait_limit); the waits on the tensor core
// and those that let copies land before the CTA exits keep kPolls.
__device__ int g_chunk_tc_timeouts = 0;
// Chunks whose T diag(beta) and P came from the concurrent pre-pass (a diagnostic).
__device__ unsigned long long g_chunk_tc_blob_chunks = 0;

struct TcParams {
    SeqParams p;
    int order_n;            // > 0: blockIdx -> sequence through order[]
    int order[64];
    // concurrent form (null: none): the pre-pass's blobs, their ready flags, and this
    // kernel's progress words (chunks begun per (sequence, head)), in one workspace
    const uint8_t *ws;
    const uint32_t *flags;
    uint32_t *progress;
};


// barrier over warps 1-15 (the triangular solve, while warp 0 issues MMAs)
__device__ __forceinline__ void tbar() { asm volatile("bar.sync 1, 480;" ::: "memory"); }

// barrier over the 4 warps of warpgroup wg (named barriers 2-5, one per warpgroup)
__device__ __forceinline__ void wg_bar(int wg) {
    switch (wg) {
        case 0: asm volatile("bar.sync 2, 128;" ::: "memory"); break;
        case 1: asm volatile("bar.sync 3, 128;" ::: "memory"); break;
        case 2: asm volatile("bar.sync 4, 128;" ::: "memory"); break;
        default: asm volatile("bar.sync 5, 128;" ::: "memory"); break;
    }
}





// One 16 x 16 x 16 product of the triangular solve, 64 threads, each a 1 x 4 strip:
// dst = (acc ? dst : 0) + sign * X Y, blocks addressed by their top-left element.
// The whole row of X (4 x 16 B) and the strip of Y (16 x 16 B) are loaded up front.
__device__ __forceinline__ void blk16(float *dst, const float *X, const float *Y, float sign, bool acc, int t) {
    const int r = t >> 2, c4 = (t & 3) * 4;
    float x[16];
#pragma unroll
    for (int k = 0; k < 16; k += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(X + r * AP + k);
        x[k] = v.x; x[k + 1] = v.y; x[k + 2] = v.z; x[k + 3] = v.w;
    }
    const float4 o = acc ? *reinterpret_cast<const float4 *>(dst + r * AP + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);  // packed f32x2 accumulators
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float4 y = *reinterpret_cast<const float4 *>(Y + k * AP + c4);
        const float2 xk = make_float2(x[k], x[k]);
        s01 = __ffma2_rn(xk, make_float2(y.x, y.y), s01);
        s23 = __ffma2_rn(xk, make_float2(y.z, y.w), s23);
    }
    const float2 sg = make_float2(sign, sign);
    const float2 o01 = __ffma2_rn(sg, s01, make_float2(o.x, o.y));
    const float2 o23 = __ffma2_rn(sg, s23, make_float2(o.z, o.w));
    *reinterpret_cast<float4 *>(dst + r * AP + c4) = make_float4(o01.x, o01.y, o23.x, o23.y);
}

// Off-diagonal 16 x 16 blocks of T = (I + A)^-1 from the diagonal inverses T_II.  Block
// row I of (I + A) T = I gives, for I > J,
//   T_IJ = -sum_{K=J}^{I-1} Y_IK T_KJ,   Y_IK = T_II A_IK,
// so after one phase that forms every Y (kept in A's unused upper block (K, I)) the
// blocks follow in three more phases of independent K = 16 products; the partial sums
// of T_20, T_31 and T_30 accumulate in place.
__device__ __forceinline__ void tri_offdiag(float *Asm, float *Tsm, int ctid) {
    auto A = [&](int i, int j) { return Asm + 16 * i * AP + 16 * j; };
    auto T = [&](int i, int j) { return Tsm + 16 * i * AP + 16 * j; };
    auto Y = [&](int i, int j) { return Asm + 16 * j * AP + 16 * i; };  // upper block (j, i) of A
    const int p = ctid >> 6, t = ctid & 63;
    // (I, J) of the six blocks below the diagonal: (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
    const int I6 = p < 3 ? p + 1 : (p == 3 ? 2 : 3), J6 = p < 3 ? p : (p == 4 ? 1 : 0);
    if (p < 6) blk16(Y(I6, J6), T(I6, I6), A(I6, J6), 1.f, false, t);  // every Y_IJ
    tbar();
    // T10, T21, T32 = -Y T_JJ; the first terms -Y20 T00, -Y31 T11, -Y30 T00 of T20, T31, T30
    if (p < 6) blk16(T(I6, J6), Y(I6, J6), T(J6, J6), -1.f, false, t);
    tbar();
    if (p < 3) {  // T20 -= Y21 T10, T31 -= Y32 T21, T30 -= Y31 T10: (I, J, K) = (2,0,1) (3,1,2) (3,0,1)
        const int I = p == 0 ? 2 : 3, J = p == 1 ? 1 : 0, K = p == 1 ? 2 : 1;
        blk16(T(I, J), Y(I, K), T(K, J), -1.f, true, t);
    }
    tbar();
    if (p == 0) blk16(T(3, 0), Y(3, 2), T(2, 0), -1.f, true, t);  // T30 -= Y32 T20
    tbar();
}

// One chunk's q and k for this thread's 4 tokens x 4 key channels (loaded into
// registers ahead of use), and g, read from its TMA-staged tile when the chunk is prepared.
struct ChunkRegs {
    float4 g[4];  // g, or its raw logits (fp32, or bf16 bits in .x/.y) until the chunk is prepared
    uint2 q[4], k[4];
    float beta;   // token warp * 4 + lane, lanes 0-3 (or its logit until prepared)
};

// The next chunk's q, k (and beta, or the raw bits of its logit) into registers.  Nothing
// here waits for the data: rows past the chunk's end read its last row instead and are
// zeroed when the chunk is prepared, and a logit is converted there too.
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
    // beta of token warp * 4 + lane (lanes 0-3; the others hold a copy)
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

// GL: g and beta come from their logits.  NORM: the output goes through the fused
// sigmoid-gated RMSNorm.  Both are compile-time choices, so the plain path carries no
// trace of either.
template <bool GL, bool NORM>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_g,
                    const __grid_constant__ CUtensorMap tmap_gate, const __grid_constant__ TcParams tp) {
    const SeqParams &p = tp.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb16 = sb >> 4;
    float *fs = reinterpret_cast<float *>(sm + S_SMALL);
    float *Asm = reinterpret_cast<float *>(sm + S_A);
    float *Tsm = reinterpret_cast<float *>(sm + S_T);
    // one barrier per tensor-core group, each completing exactly once per chunk
    uint64_t *bar_g = reinterpret_cast<uint64_t *>(sm + S_BARS);  // gram
    uint64_t *bar_r = bar_g + 1;                                    // R and O
    uint64_t *bar_d = bar_g + 2;                                    // D
    uint64_t *bar_s = bar_g + 3;                                    // O and S updates
    uint64_t *tma_bar = bar_g + 4;                                  // V tile
    uint64_t *drain_bar = bar_g + 5;                                // drain after a failure
    uint64_t *gt_bar = bar_g + 6;                                   // g tile
    uint64_t *pre_bar = bar_g + 7;                                  // decay prefix written (128 arrivals)
    uint64_t *gate_bar = reinterpret_cast<uint64_t *>(sm + S_BARS + 72);  // fused norm: gate tile
    uint64_t *blob_bar = reinterpret_cast<uint64_t *>(sm + S_BARS + 80);  // concurrent form: a chunk's blob
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + S_BARS + 64);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wg = warp >> 2, wq = warp & 3;
    const int m = wq * 32 + lane;  // TMEM lane this thread reads/writes
    const int l4 = lane * 4;       // this thread's 4 key channels in the prep phase
    const int H = p.H;
    int n = blockIdx.x / H;
    const int h = blockIdx.x % H;
    if (tp.order_n > 0) n = tp.order[n];
    const int unit = n * H + h;
    int bos, len;
    seq_range(p, n, bos, len);
    const int nchunks = (len + C - 1) / C;

    // first chunk's inputs are in flight while the CTA sets up
    ChunkRegs cr;
    load_chunk<GL>(p, cr, bos, 0, min(C, len), h, warp, l4);

    if (tid == 0) {
        for (int b = 0; b < 7; ++b) mbar_init(bar_g + b, 1);
        mbar_init(pre_bar, 128);
        if (NORM) mbar_init(gate_bar, 1);
        mbar_init(blob_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // bf16 identity tile (K-major, rows i, columns j)
    {
        const int i = tid >> 3, j0 = (tid & 7) * 8;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (i >= j0 && i < j0 + 8) w[(i - j0) >> 1] = (i & 1) ? 0x3F800000u : 0x00003F80u;
        st_shared_v4(sb + S_ID + sw128_off(i, j0, 64), w[0], w[1], w[2], w[3]);
        // T diag(beta) tiles (hi and lo, 8 KB each): zero; each chunk rewrites only the
        // blocks on or below the diagonal
        st_shared_v4(sb + S_TBH + tid * 32, 0u, 0u, 0u, 0u);
        st_shared_v4(sb + S_TBH + tid * 32 + 16, 0u, 0u, 0u, 0u);
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


    auto issue_v = [&](int chunk) {
        mbar_arrive_expect_tx(tma_bar, 16384);
        tma_load_3d(sb + S_V, &tmap_v, tma_bar, 0, h, bos + chunk * C);
        tma_load_3d(sb + S_V + 8192, &tmap_v, tma_bar, 64, h, bos + chunk * C);
    };
    int v_pending = -1;  // chunk whose V tile is in flight (thread 0 only)
    int q_pending = -1;  // chunk whose gate tile is in flight (thread 0 only)
    // g (or its logits) of one chunk, 64 tokens x 128 channels, into the Km tile, which is
    // free from the end of a gram pass until the next operand tiles are written
    const uint32_t g_bytes = (GL && p.g_logits_bf16) ? C * DK * 2 : C * DK * 4;
    auto issue_g = [&](int chunk) {
        mbar_arrive_expect_tx(gt_bar, g_bytes);
        tma_load_3d(sb + S_KM, &tmap_g, gt_bar, 0, h, bos + chunk * C);
    };
    int g_pending = -1;  // chunk whose g tile is in flight (thread 0 only)
    int b_pending = -1;  // blob copy in flight (thread 0 only): the phase of blob_bar it completes
    uint32_t n_blobs = 0;  // blob copies issued (thread 0 only)
    int failed = 0;      // a bounded wait gave up
    if (tid == 0 && nchunks > 0) {
        issue_v(0);
        v_pending = 0;
        issue_g(0);
        g_pending = 0;
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

    auto wait_group = [&](uint64_t *bar, int parity) {
        const bool ok = mbar_wait(bar, (uint32_t)parity, kPolls);
        fence_after_sync();
        return ok;
    };

    float *scan = reinterpret_cast<float *>(sm + S_SCAN);

    // ---- preparation of a chunk, first half: per-token norm scales and beta into the
    // small buffers, each warp's decay totals per key channel into the scan buffer.
    // The 8 sums of squares of a warp's 4 tokens are reduced with a reduce-scatter
    // (9 shuffles); lanes 4v..4v+3 end with sum v (q of tokens 0-3, then k).
    auto prep_norms = [&](ChunkRegs &c, int cnn, int chunk) {
        if (!mbar_wait(gt_bar, (uint32_t)(chunk & 1), p.polls))
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
                const uint2 u = *reinterpret_cast<const uint2 *>(sm + S_KM + (i * DK + l4) * 2);
                c.g[r] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), 0.f, 0.f);
            } else {
                c.g[r] = *reinterpret_cast<const float4 *>(sm + S_KM + (i * DK + l4) * 4);
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
        }
        if (GL && lane < 4) {
            const uint32_t raw = __float_as_uint(c.beta);
            c.beta = warp * 4 + lane < cnn ? beta_of_logit(__uint_as_float(p.beta_logits_bf16 ? raw << 16 : raw)) : 0.f;
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
        if (lane < 4) fs[(!GL && warp == 0 ? F_BETA0 : F_BETA + warp * 4) + lane] = c.beta;
        float2 t01 = make_float2(c.g[0].x, c.g[0].y), t23 = make_float2(c.g[0].z, c.g[0].w);
#pragma unroll
        for (int r = 1; r < 4; ++r) {
            t01 = __fadd2_rn(t01, make_float2(c.g[r].x, c.g[r].y));
            t23 = __fadd2_rn(t23, make_float2(c.g[r].z, c.g[r].w));
        }
        const float4 t = make_float4(t01.x, t01.y, t23.x, t23.y);
        *reinterpret_cast<float4 *>(!GL && warp == 0 ? fs + F_SCAN0 + l4 : scan + warp * 128 + l4) = t;
    };
    // With g and beta given (!GL), warp 0 (which issues the tensor-core work) prepares its
    // tokens' norms while the solve runs, into side buffers; beta joins the others once
    // the current chunk's solve has read F_BETA.  With logits, the transforms take longer
    // than the solve leaves, and warp 0 prepares its tokens with the others.
    auto beta0_publish = [&]() {
        if (!GL && warp == 0 && lane < 4) fs[F_BETA + lane] = fs[F_BETA0 + lane];
    };

    // ---- preparation, second half (after a barrier): cumulative decay, exp(gamma),
    // the [-Kd ; Qd] and Km operand tiles; Kg is returned in registers because its
    // tile may still be in use.  Returns 1 if the chunk's decay range is too wide.
    // ---- exclusive prefix of the warps' decay totals per key channel, and the chunk
    // total (row 16), by warps 1-4; then a barrier of warps 1-15 (warp 0 is issuing)
    float *pre = scan + 16 * 128;
    auto scan_prefix = [&]() {
        if (warp >= 1 && warp <= 4) {
            const int c = tid - 32;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float t = (!GL && w == 0) ? fs[F_SCAN0 + c] : scan[w * 128 + c];
                pre[w * 128 + c] = acc;
                acc += t;
            }
            pre[16 * 128 + c] = acc;
            mbar_arrive(pre_bar);  // for warp 0, which is not in the barrier below
        }
        tbar();
    };

    // [-Kd ; Qd] rows of token i (hi and lo tiles) from its cumulative decay G on this
    // lane's four key channels; rows i and 64 + i share the swizzle phase, 8 KB apart
    auto put_kq = [&](int i, const float2 (&G)[2], uint2 q, uint2 k, float rq, float rk) {
        const float2 qv2[2] = {make_float2(bf16lo(q.x), bf16hi(q.x)), make_float2(bf16lo(q.y), bf16hi(q.y))};
        const float2 kv2[2] = {make_float2(bf16lo(k.x), bf16hi(k.x)), make_float2(bf16lo(k.y), bf16hi(k.y))};
        const float2 nrk2 = make_float2(-rk, -rk), rq2 = make_float2(rq, rq);
        float2 kd[2], qd[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 eG = make_float2(__expf(G[e].x), __expf(G[e].y));
            kd[e] = __fmul2_rn(__fmul2_rn(kv2[e], nrk2), eG);  // -k^ exp(G)
            qd[e] = __fmul2_rn(__fmul2_rn(qv2[e], rq2), eG);
        }
        const uint32_t off = sw128_off(i, l4, 128);
        uint32_t h0, l0, h1, l1;
        split2(kd[0].x, kd[0].y, h0, l0);
        split2(kd[1].x, kd[1].y, h1, l1);
        st_shared_v2(sb + S_KQH + off, h0, h1);
        st_shared_v2(sb + S_KQL + off, l0, l1);
        split2(qd[0].x, qd[0].y, h0, l0);
        split2(qd[1].x, qd[1].y, h1, l1);
        st_shared_v2(sb + S_KQH + off + 8192, h0, h1);
        st_shared_v2(sb + S_KQL + off + 8192, l0, l1);
    };
    auto prep_tiles = [&](const ChunkRegs &c, float (&kgv)[4][4], bool use_pre) -> int {
        float o4[4] = {0.f, 0.f, 0.f, 0.f}, gam[4] = {0.f, 0.f, 0.f, 0.f};
        if (use_pre) {  // offset of this warp's tokens and the chunk total, per channel
            const float4 t = *reinterpret_cast<const float4 *>(pre + warp * 128 + l4);
            const float4 u = *reinterpret_cast<const float4 *>(pre + 16 * 128 + l4);
            o4[0] = t.x; o4[1] = t.y; o4[2] = t.z; o4[3] = t.w;
            gam[0] = u.x; gam[1] = u.y; gam[2] = u.z; gam[3] = u.w;
        } else {
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const float4 t = *reinterpret_cast<const float4 *>(!GL && w == 0 ? fs + F_SCAN0 + l4 : scan + w * 128 + l4);
                const float tt[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (w < warp) o4[e] += tt[e];
                    gam[e] += tt[e];
                }
            }
        }
        float egam[4];
        int oor = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            egam[e] = __expf(gam[e]);
            oor |= (-gam[e] > kRangeMax);
        }
        if (warp == 1) *reinterpret_cast<float4 *>(fs + F_GEXP + l4) = make_float4(egam[0], egam[1], egam[2], egam[3]);
        const float4 rq4 = *reinterpret_cast<const float4 *>(fs + F_RQ + warp * 4);
        const float4 rk4 = *reinterpret_cast<const float4 *>(fs + F_RK + warp * 4);
        const float rq[4] = {rq4.x, rq4.y, rq4.z, rq4.w}, rk[4] = {rk4.x, rk4.y, rk4.z, rk4.w};
        // channel pairs (0,1) and (2,3) in packed f32x2 arithmetic, each product in the
        // same order as its scalar form
        float2 o2[2] = {make_float2(o4[0], o4[1]), make_float2(o4[2], o4[3])};
        const float2 eg2[2] = {make_float2(egam[0], egam[1]), make_float2(egam[2], egam[3])};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = warp * 4 + r;
            const float2 gr2[2] = {make_float2(c.g[r].x, c.g[r].y), make_float2(c.g[r].z, c.g[r].w)};
            const float2 kv2[2] = {make_float2(bf16lo(c.k[r].x), bf16hi(c.k[r].x)),
                                   make_float2(bf16lo(c.k[r].y), bf16hi(c.k[r].y))};
            const float2 rk2 = make_float2(rk[r], rk[r]);
            float2 km[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                o2[e] = __fadd2_rn(o2[e], gr2[e]);  // inclusive cumulative decay G of token i
                const float2 em = make_float2(__expf(-o2[e].x), __expf(-o2[e].y));
                km[e] = __fmul2_rn(__fmul2_rn(kv2[e], rk2), em);
                const float2 kg = __fmul2_rn(km[e], eg2[e]);
                kgv[r][2 * e] = kg.x;
                kgv[r][2 * e + 1] = kg.y;
            }
            put_kq(i, o2, c.q[r], c.k[r], rq[r], rk[r]);
            const uint32_t off = sw128_off(i, l4, 128);
            uint32_t h0, l0, h1, l1;
            split2(km[0].x, km[0].y, h0, l0);
            split2(km[1].x, km[1].y, h1, l1);
            st_shared_v2(sb + S_KM + off, h0, h1);
            st_shared_v2(sb + S_KM + off + 8192, l0, l1);
        }
        return oor;
    };

    auto st_kg = [&](const float (&kgv)[4][4]) { st_kgt(sb + S_PKGH, sb + S_PKGL, l4, warp * 4, kgv); };

    // ---- first chunk's preparation (later chunks are prepared inside the previous
    // chunk's tensor-core waits)
    int oor_next = 0;
    float kgv[4][4];  // the next chunk's Kg, stored while that chunk's gram runs
    const float norm_wv = NORM ? __ldg(p.norm_w + m) : 0.f;  // the norm weight of this thread's value channel
    if (nchunks > 0) {
        prep_norms(cr, min(C, len), 0);
        beta0_publish();
        __syncthreads();
        oor_next = prep_tiles(cr, kgv, false);
    }

    for (int ch = 0; ch < nchunks; ++ch) {
        const int par = ch & 1;
        const int t0 = ch * C;
        const int cn = min(C, len - t0);
        fence_async_smem();
        fence_before_sync();  // the previous state pass (or the initial state) wrote TMEM
        // concurrent form: has the pre-pass already formed this chunk's T diag(beta) and P?
        // (read once, never waited for: otherwise this CTA forms them itself, as always)
        size_t blob_idx = 0;
        if (tp.flags) {
            blob_idx = (size_t)blob_slot(bos, n, ch) * H + h;
            if (tid == 0) {
                st_relaxed_gpu(tp.progress + unit, (uint32_t)ch + 1u);
                reinterpret_cast<volatile uint32_t *>(fs)[F_BLOB] = ld_acquire_gpu(tp.flags + blob_idx);
            }
        }
        // ---- operand tiles of this chunk and S(n-1) are ready
        const int fallback = __syncthreads_or(oor_next);
        // a wide-decay chunk keeps its exact path (its Kg^T is formed there too)
        const bool use_blob = tp.flags && !fallback && reinterpret_cast<volatile uint32_t *>(fs)[F_BLOB] != 0u;

        // ================= gram [-Kd;Qd] [Km_hi;Km_lo]^T (+ lo x hi), or the blob
        if (tid == 0) {
            fence_after_sync();
            if (use_blob) {
                // T diag(beta) hi/lo and P hi/lo straight into their operand tiles: T diag(beta)
                // was last read by the previous D product, P by the previous O/S product
                fence_proxy_async_global();
                const uint8_t *blob = tp.ws + blob_idx * kBlobBytes;
                mbar_arrive_expect_tx(blob_bar, kBlobBytes);
                bulk_load(sb + S_TBH, blob, 16384, blob_bar);
                bulk_load(sb + S_PKGH, blob + 16384, 8192, blob_bar);
                bulk_load(sb + S_PKGL, blob + 24576, 8192, blob_bar);
                b_pending = (int)(n_blobs++ & 1);
                atomicAdd(&g_chunk_tc_blob_chunks, 1ull);
            } else if (!fallback) {
                const uint32_t id128 = idesc_bf16(128, 128, false, false);
                const uint32_t id64 = idesc_bf16(128, 64, false, false);
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // [-Kd;Qd]_hi x [Km_hi;Km_lo]^T
                    const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_ss(tb + T_G, sdesc_at(sb16, S_KQH + koff, 16, 1024), sdesc_at(sb16, S_KM + koff, 16, 1024), id128,
                           s ? 1u : 0u);
                }
#pragma unroll 1
                for (int s = 0; s < 8; ++s) {  // [-Kd;Qd]_lo x Km_hi^T into the first half
                    const uint32_t koff = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_ss(tb + T_G, sdesc_at(sb16, S_KQL + koff, 16, 1024), sdesc_at(sb16, S_KM + koff, 16, 1024), id64, 1u);
                }
            }
            mma_commit(bar_g);  // an empty commit on fallback chunks
        }
        __syncwarp();
        // this chunk's Kg^T tile (the previous O/S product has read the old one; the gram
        // does not read it)
        st_kg(kgv);
        fence_async_smem();
        // warps 1-15 start loading the next chunk while waiting for the gram (warp 0 loads
        // its tokens after the gram pass)
        if (warp > 0 && ch + 1 < nchunks) load_chunk<GL>(p, cr, bos, t0 + C, min(C, len - t0 - C), h, warp, l4);
        if (!wait_group(bar_g, par)) failed = 1;
        if (use_blob) {
            // nothing to form: the pre-pass did the gram pass and the solve
        } else if (!fallback) {
            uint32_t r1[16], r2[16];
            tmem_ld16(tb + lane_off + T_G + wg * 16, r1);
            tmem_ld16(tb + lane_off + T_G + 64 + wg * 16, r2);
            tmem_wait_ld();
            const int j0 = wg * 16;
            if (m < 64) {
                const int i = m;
                const float b = -fs[F_BETA + i];  // gram rows hold -Kd Km^T
                float4 *dst = reinterpret_cast<float4 *>(Asm + i * AP + j0);
                const float2 b2 = make_float2(b, b);
#pragma unroll
                for (int c = 0; c < 16; c += 4) {
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
                float x[16];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float2 v = __fadd2_rn(make_float2(__uint_as_float(r1[c]), __uint_as_float(r1[c + 1])),
                                                make_float2(__uint_as_float(r2[c]), __uint_as_float(r2[c + 1])));
                    x[c] = (j0 + c <= i) ? v.x : 0.f;
                    x[c + 1] = (j0 + c + 1 <= i) ? v.y : 0.f;
                }
                st_tile8(sb + S_PKGH, sb + S_PKGL, 192, i, j0, x);
                st_tile8(sb + S_PKGH, sb + S_PKGL, 192, i, j0 + 8, x + 8);
            }
        } else {
            // exact grams with pairwise exponentials (decay range too wide for Km)
            float *Gs = reinterpret_cast<float *>(sm + S_FB_G);
            const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(p.q);
            const __nv_bfloat16 *kgl = reinterpret_cast<const __nv_bfloat16 *>(p.k);
            if (tid < 128) {  // G for every token and channel, from the inputs again
                float acc = 0.f;
                for (int i = 0; i < C; ++i) {
                    if (i < cn) acc += load_g(p, ((size_t)(bos + t0 + i) * H + h) * DK + tid, h, tid);
                    Gs[i * 128 + tid] = acc;
                }
            }
            __syncthreads();
            {  // Kg from the exact G (the fast formula overflows here)
                float kg[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = warp * 4 + r;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float kv = i < cn ? __bfloat162float(kgl[((size_t)(bos + t0 + i) * H + h) * DK + l4 + c]) : 0.f;
                        kg[r][c] = kv * fs[F_RK + i] * __expf(Gs[63 * 128 + l4 + c] - Gs[i * 128 + l4 + c]);
                    }
                }
                st_kgt(sb + S_PKGH, sb + S_PKGL, l4, warp * 4, kg);
            }
            float *Pf = Tsm;  // P in fp32, converted to the tile below
            for (int i = warp; i < C; i += 16) {
                const size_t ri = ((size_t)(bos + t0 + i) * H + h) * DK;
                float qi[4], ki[4], gi[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int ch_ = lane + 32 * c;
                    qi[c] = i < cn ? __bfloat162float(qg[ri + ch_]) : 0.f;
                    ki[c] = i < cn ? __bfloat162float(kgl[ri + ch_]) : 0.f;
                    gi[c] = Gs[i * 128 + ch_];
                }
                for (int j = 0; j <= i; ++j) {
                    const size_t rj = ((size_t)(bos + t0 + j) * H + h) * DK;
                    float a = 0.f, b = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int ch_ = lane + 32 * c;
                        const float kj = (j < cn ? __bfloat162float(kgl[rj + ch_]) : 0.f) * __expf(gi[c] - Gs[j * 128 + ch_]);
                        a = fmaf(ki[c], kj, a);
                        b = fmaf(qi[c], kj, b);
                    }
                    a = warp_sum(a) * fs[F_RK + i] * fs[F_RK + j];
                    b = warp_sum(b) * fs[F_RQ + i] * fs[F_RK + j];
                    if (lane == 0) {
                        Asm[i * AP + j] = (j < i) ? fs[F_BETA + i] * a : 0.f;
                        Pf[i * AP + j] = b;
                    }
                }
                if (lane == 0)
                    for (int j = i + 1; j < C; ++j) {
                        Asm[i * AP + j] = 0.f;
                        Pf[i * AP + j] = 0.f;
                    }
            }
            __syncthreads();
            {
                const int i = tid >> 3, j0 = (tid & 7) * 8;
                float x[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) x[c] = Pf[i * AP + j0 + c];
                st_tile8(sb + S_PKGH, sb + S_PKGL, 192, i, j0, x);
            }
            // every thread wrote P / Kg rows the tensor core reads (warp 0 does not reach
            // the solve's fence); on regular chunks only warps 1-15 write P and fence there
            fence_async_smem();
        }
        __syncthreads();

        if (warp == 0) {
            if (lane == 0 && ch + 1 < nchunks && !failed) {  // the gram has read Km (and the exact path its G scratch)
                issue_g(ch + 1);
                g_pending = ch + 1;
            }
            if (ch + 1 < nchunks) load_chunk<GL>(p, cr, bos, t0 + C, min(C, len - t0 - C), h, warp, l4);
        }
        if (tid == 0) {
            // ================= R^T = V^T I + S^T (-Kd)^T, O^T = S^T Qd^T (while warps 1-15 solve T)
            if (mbar_wait(tma_bar, (uint32_t)par, p.polls))
                v_pending = -1;
            else
                failed = 1;
            fence_after_sync();
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
        } else if (warp > 0 && !use_blob) {
            // ================= T = (I + A)^-1, blocked with 16 x 16 diagonal blocks (warps 1-15)
            const int ctid = tid - 32;
            if (tid >= kThreads - 64) {
                const int t = tid - (kThreads - 64), b = t >> 4, c = t & 15, o = 16 * b;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a[16];
#pragma unroll
                    for (int j4 = 0; j4 < i; j4 += 4) {  // row i of the block, 16 B at a time
                        const float4 v = *reinterpret_cast<const float4 *>(Asm + (o + i) * AP + o + j4);
                        a[j4] = v.x; a[j4 + 1] = v.y; a[j4 + 2] = v.z; a[j4 + 3] = v.w;
                    }
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < i; ++j) acc = fmaf(a[j], x[j], acc);
                    x[i] = (i < c) ? 0.f : (i == c ? 1.f : -acc);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) Tsm[(o + i) * AP + o + c] = x[i];
            }
            tbar();
            tri_offdiag(Asm, Tsm, ctid);
            {  // T diag(beta) -> hi/lo tile (rows i, K = j): only the 288 blocks of 8 columns on or
               // below the diagonal (the rest stays zero from the setup), one per thread: the
               // threads whose block lies above it take rows 60-63
                int i = ctid >> 3, jb = ctid & 7;
                if (jb == 7 && i < 32) {
                    jb = i & 7;
                    i = 60 + (i >> 3);
                }
                const int j0 = jb * 8;
                if (j0 <= i) {
                float x[8];
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    const float2 v = __fmul2_rn(make_float2(Tsm[i * AP + j0 + c], Tsm[i * AP + j0 + c + 1]),
                                                make_float2(fs[F_BETA + j0 + c], fs[F_BETA + j0 + c + 1]));
                    x[c] = (j0 + c <= i) ? v.x : 0.f;
                    x[c + 1] = (j0 + c + 1 <= i) ? v.y : 0.f;
                }
                st_tile8(sb + S_TBH, sb + S_TBL, 64, i, j0, x);
                }
            }
            fence_async_smem();
        }
        __syncwarp();
        // warp 0, idle while the solve runs (g and beta given): the next chunk's norms for its own tokens
        if (!GL && warp == 0 && ch + 1 < nchunks) prep_norms(cr, min(C, len - t0 - C), ch + 1);
        __syncthreads();

        // ================= R pass: R^T (lane v, column j) -> hi/lo operand in TMEM
        if (!wait_group(bar_r, par)) failed = 1;
        if (tid == 0 && ch + 1 < nchunks && !failed) {  // the V tile has been read
            issue_v(ch + 1);
            v_pending = ch + 1;
        }
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
        if (NORM) fence_async_smem();  // the A buffer (written in the gram pass) takes the gate tile next
        fence_before_sync();
        // ---- T diag(beta) tile and R^T hi/lo are ready
        if (__syncthreads_or(failed)) break;
        // fused norm, bf16 gate: this chunk's gate tile (64 tokens x 128 values) into the A
        // buffer, free from the end of the solve to the next gram pass, read by the O pass
        if (NORM && tid == 0 && p.gate_bf16) {
            mbar_arrive_expect_tx(gate_bar, C * DV * 2);
            tma_load_3d(sb + S_A, &tmap_gate, gate_bar, 0, h, bos + t0);
            q_pending = ch;
        }

        // ================= D^T = R^T (T diag beta)^T
        if (tid == 0) {
            if (use_blob) {  // the blob's tiles have landed (the O/S product reads P after this too)
                if (mbar_wait(blob_bar, (uint32_t)b_pending, p.polls))
                    b_pending = -1;
                else
                    failed = 1;
            }
            fence_after_sync();
            // R^T_hi [T diag(beta)_hi ; _lo]^T (N = 128: the two tiles are contiguous) into
            // [D_a | D_b], then R^T_lo (T diag beta)_hi^T onto D_a
            const uint32_t id128 = idesc_bf16(128, 128, false, false), id64 = idesc_bf16(128, 64, false, false);
#pragma unroll 1
            for (int s = 0; s < 4; ++s)
                mma_ts(tb + T_G, tb + T_R + s * 16, sdesc_at(sb16, S_TBH + s * 32, 16, 1024), id128, s ? 1u : 0u);
#pragma unroll 1
            for (int s = 0; s < 4; ++s)
                mma_ts(tb + T_G, tb + T_R + s * 16 + 8, sdesc_at(sb16, S_TBH + s * 32, 16, 1024), id64, 1u);
            mma_commit(bar_d);
        }
        __syncwarp();
        // while D runs: the next chunk's norms, beta and decay totals
        if (ch + 1 < nchunks) {
            if (GL || warp > 0) {
                prep_norms(cr, min(C, len - t0 - C), ch + 1);
            } else {
                beta0_publish();
            }
        }
        // ================= D pass (hi/lo into TMEM) and S decay by exp(gamma)
        if (!wait_group(bar_d, par)) failed = 1;
        {
            uint32_t r[16], s1[16], s2[16], hi[8], lo[8];
            const int c0 = wg * 32;
            {
                uint32_t rb[16];
                tmem_ld16(tb + lane_off + T_G + wg * 16, r);
                tmem_ld16(tb + lane_off + T_G + 64 + wg * 16, rb);
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
            tmem_st8(tb + lane_off + T_G + wg * 16, hi);  // in place: tokens 16 wg.. as hi, then lo
            tmem_st8(tb + lane_off + T_G + wg * 16 + 8, lo);
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
        // ---- D^T hi/lo ready, S^T decayed
        if (__syncthreads_or(failed)) break;

        // ================= [O|S]^T += D^T [P^T | Kg]
        if (tid == 0) {
            fence_after_sync();
            const uint32_t id192 = idesc_bf16(128, 192, false, false);
#pragma unroll
            for (int cb = 0; cb < 3; ++cb)
#pragma unroll 1
                for (int s = 0; s < 4; ++s)
                    mma_ts(tb + T_O, tb + T_G + s * 16 + (combo_a(cb) ? 8 : 0),
                           sdesc_at(sb16, (combo_b(cb) ? S_PKGL : S_PKGH) + s * 32, 16, 1024), id192, 1u);
            mma_commit(bar_s);
        }
        __syncwarp();
        // while O and S update: the next chunk's operand tiles (its Kg waits for this MMA)
        if (ch + 1 < nchunks) {
            if (warp > 0)
                scan_prefix();
            else if (!mbar_wait(pre_bar, (uint32_t)(ch & 1), kPolls))  // warp 0, after its O/S issue
                failed = 1;
            oor_next = prep_tiles(cr, kgv, true);
        }
        // ================= O pass (+ gated norm) and state pass
        if (!wait_group(bar_s, par)) failed = 1;
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
                const float w = norm_wv;
                // sigmoid of the gates before the barrier, where the warps wait for the last
                // one (a fast reciprocal: 2 ulp).  A bf16 gate comes from the tile in shared
                // memory; an fp32 one from global memory
                float sg[16];
                if (p.gate_bf16) {
                    if (!mbar_wait(gate_bar, (uint32_t)(ch & 1), p.polls))
                        failed = 1;
                    else if (tid == 0)
                        q_pending = -1;
                    const uint16_t *gs = reinterpret_cast<const uint16_t *>(sm + S_A) + i0 * DV + v;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        sg[c] = __fdividef(1.0f, 1.0f + __expf(-__uint_as_float((uint32_t)gs[c * DV] << 16)));
                } else {
                    const float *gp = reinterpret_cast<const float *>(p.gate) + ((size_t)(bos + t0) * H + h) * DV + v;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        sg[c] = __fdividef(1.0f, 1.0f + __expf(-__ldg(gp + (size_t)min(i0 + c, cn - 1) * H * DV)));
                }
                // a row's statistics come from the 4 warps of its warpgroup only: the other
                // warpgroups need not wait for warp 0, the tensor-core issuer and last here
                wg_bar(wg);
                // lane l forms 1 / rms of row l % 16 once; the others take it by shuffle
                const int cl = lane & 15;
                const float ssl = red[(wg * 4 + 0) * 16 + cl] + red[(wg * 4 + 1) * 16 + cl] +
                                  red[(wg * 4 + 2) * 16 + cl] + red[(wg * 4 + 3) * 16 + cl];
                const float invl = rsqrtf(ssl * (1.f / DV) + p.eps);
                // rows i0.. of this head: one base address and a constant row stride, the output
                // type chosen once for the pass
                const size_t base = ((size_t)(bos + t0 + i0) * H + h) * DV + v, stride = (size_t)H * DV;
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
                const size_t base = ((size_t)(bos + t0 + i0) * H + h) * DV + v, stride = (size_t)H * DV;
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
            atomicAdd(&g_chunk_tc_timeouts, 1);
            mma_commit(drain_bar);  // arrives once the tensor-core work already issued has drained
            if (v_pending >= 0) mbar_wait(tma_bar, (uint32_t)(v_pending & 1), kPolls);  // V copy in flight
            if (g_pending >= 0) mbar_wait(gt_bar, (uint32_t)(g_pending & 1), kPolls);   // g copy in flight
            if (q_pending >= 0) mbar_wait(gate_bar, (uint32_t)(q_pending & 1), kPolls);  // gate copy in flight
            if (b_pending >= 0) mbar_wait(blob_bar, (uint32_t)b_pending, kPolls);       // blob copy in flight
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

// ---------------------------------------------------------------------------
// host side

EncodeTiledFn encode_fn() { return reinterpret_cast<EncodeTiledFn>(tensor_map_encoder()); }

}  // namespace

void *tensor_map_encoder() {
    static void *fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = ptr;
    }
    return fn;
}

int take_chunk_tc_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_chunk_tc_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_chunk_tc_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("chunk_tc: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

long long take_chunk_blob_chunks(cudaStream_t st) {
    unsigned long long n = 0;
    const unsigned long long zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_chunk_tc_blob_chunks, sizeof(n), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_chunk_tc_blob_chunks, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("chunk_tc: cannot read the blob counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return (long long)n;
}

bool chunk_tc_supported(int K, int V, int chunk) { return K == DK && V == DV && chunk == C; }

kda_status launch_chunk_tc(const SeqParams &p_in, int K, int V, int chunk, cudaStream_t st, const void *ws) {
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
    CUresult cres = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p_in.v), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cres != CUDA_SUCCESS) {
        set_error("chunk_tc: cuTensorMapEncodeTiled failed (%d)", (int)cres);
        return KDA_ERR_CUDA;
    }
    CUtensorMap tmap_g;
    {
        const bool gb = p_in.g_logits && p_in.g_logits_bf16;
        const cuuint64_t es = gb ? 2 : 4;
        const void *gsrc = p_in.g_logits ? p_in.g_logits : (const void *)p_in.g;
        const cuuint64_t gdims[3] = {(cuuint64_t)DK, (cuuint64_t)p_in.H, (cuuint64_t)rows};
        const cuuint64_t gstrides[2] = {(cuuint64_t)DK * es, (cuuint64_t)p_in.H * DK * es};
        const cuuint32_t gbox[3] = {(cuuint32_t)DK, 1, (cuuint32_t)C};
        cres = enc(&tmap_g, gb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<void *>(gsrc), gdims, gstrides, gbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cres != CUDA_SUCCESS) {
            set_error("chunk_tc: cuTensorMapEncodeTiled failed for g (%d)", (int)cres);
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
        cres = enc(&tmap_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p_in.gate), qdims, qstrides,
                   qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cres != CUDA_SUCCESS) {
            set_error("chunk_tc: cuTensorMapEncodeTiled failed for the gate (%d)", (int)cres);
            return KDA_ERR_CUDA;
        }
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
    static DeviceOnce configured;
    const int dev = current_device();
    if (!configured.done(dev)) {
        for (void *fn : {(void *)chunk_tc_kernel<false, false>, (void *)chunk_tc_kernel<true, false>,
                         (void *)chunk_tc_kernel<false, true>, (void *)chunk_tc_kernel<true, true>}) {
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            if (e != cudaSuccess) {
                set_error("chunk_tc: cannot reserve %u bytes of shared memory: %s", SMEM_BYTES, cudaGetErrorString(e));
                return KDA_ERR_CUDA;
            }
        }
        configured.set(dev);
    }
    auto kern = p_in.g_logits ? (p_in.gate ? chunk_tc_kernel<true, true> : chunk_tc_kernel<true, false>)
                              : (p_in.gate ? chunk_tc_kernel<false, true> : chunk_tc_kernel<false, false>);
    if (!ws) {
        kern<<<units, kThreads, SMEM_BYTES, st>>>(tmap, tmap_g, tmap_gate, tp);
        note_launch();
        return check_launch("chunk_tc_kernel");
    }
    // concurrent form: this kernel's CTAs must take their SMs before the pre-pass's, which
    // is launched right after on another stream, so it runs at the highest priority
    const WorkspaceLayout L(rows, p_in.N, p_in.H);
    tp.ws = static_cast<const uint8_t *>(ws);
    tp.flags = reinterpret_cast<const uint32_t *>(tp.ws + L.flags);
    tp.progress = reinterpret_cast<uint32_t *>(const_cast<uint8_t *>(tp.ws) + L.progress);
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) {
        cudaGetLastError();
        greatest = 0;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(units, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributePriority;
    attr[0].val.priority = greatest;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmap, tmap_g, tmap_gate, tp);
    note_launch();
    if (e != cudaSuccess) {
        set_error("chunk_tc_kernel: %s", cudaGetErrorString(e));
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return check_launch("chunk_tc_kernel");
}

kda_status launch_chunk_concurrent(const SeqParams &p, void *ws, cudaStream_t st) {
    const int units = p.N * p.H, sms = sm_count();
    const int64_t rows = p.cu_seqlens ? (int64_t)p.T : (int64_t)p.N * p.T;
    if (units >= sms || rows <= 0) return launch_chunk_tc(p, DK, DV, C, st);  // no SM would be left over
    kda_status s = configure_chunk_prep();  // before the fused kernel is launched
    if (s != KDA_OK) return s;
    const WorkspaceLayout L(rows, p.N, p.H);
    cudaStream_t side = nullptr;
    cudaEvent_t ready = nullptr, done = nullptr;
    auto cuda_fail = [&](const char *what, cudaError_t e) {
        set_error("chunk (concurrent form): %s failed: %s", what, cudaGetErrorString(e));
        cudaGetLastError();
        s = KDA_ERR_CUDA;
    };
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking)) != cudaSuccess) {
        cuda_fail("creating a stream", e);
        return s;
    }
    if ((e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&done, cudaEventDisableTiming)) != cudaSuccess) {
        cuda_fail("creating an event", e);
    } else if ((e = cudaMemsetAsync(static_cast<uint8_t *>(ws) + L.flags, 0, L.bytes - L.flags, st)) != cudaSuccess) {
        cuda_fail("clearing the flags", e);
    } else if ((e = cudaEventRecord(ready, st)) != cudaSuccess || (e = cudaStreamWaitEvent(side, ready, 0)) != cudaSuccess) {
        cuda_fail("ordering the streams", e);
    } else if ((s = launch_chunk_tc(p, DK, DV, C, st, ws)) == KDA_OK) {
        PrepConcurrent cc;
        cc.grid = 2 * (sms - units);  // two pre-pass CTAs per idle SM
        cc.lead = 2;
        s = launch_chunk_prep(p, ws, side, &cc);
        // the caller's stream covers the pre-pass too, even after a failed launch
        if ((e = cudaEventRecord(done, side)) != cudaSuccess || (e = cudaStreamWaitEvent(st, done, 0)) != cudaSuccess)
            cuda_fail("joining the streams", e);
    }
    if (ready) cudaEventDestroy(ready);
    if (done) cudaEventDestroy(done);
    cudaStreamDestroy(side);  // released once its work completes
    return s;
}

}  // namespace kda
