// kda_recurrent.cu -- the token-by-token KDA kernel (decode step and multi-token form).
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (a decode step
// runs the token-by-token kernel), section 03 "Kimi Delta Attention decays each
// key channel" and section 04 (decay per key channel before each delta-rule
// update; q, k L2-normalised in the kernel).  Kimi-K3 atlas "gate-project
// (decode, P = 1000)" for the fused sigmoid-gated RMSNorm.
//
// One CTA per (sequence, head).  The fp32 state S[K][V] lives in registers for
// the whole call: warp w owns rows [w*K/NW, (w+1)*K/NW), lane l owns columns
// [l*V/32, (l+1)*V/32) of every one of them, so each row is read and written as
// one coalesced 128-bit-per-lane transaction (V = 128).  Per token:
//   S' = Diag(exp g) S           (each thread scales its own rows)
//   u  = S'^T k^,  p = S'^T q^   (per-thread partials over rows, then a
//                                 cross-warp sum in shared memory)
//   D  = beta (v - u)
//   o  = scale (p + (k^.q^) D)   = scale S^T q^ after the write
//   S  = S' + k^ D^T
// so the state crosses HBM exactly once in each direction per call.  For decode
// (T = 1) that is the whole cost: 2 x 64 KiB per (sequence, head) at d = 128.
#include <math.h>

#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int VPL>
struct VecF;
template <>
struct VecF<1> {
    float x[1];
};
template <>
struct VecF<2> {
    float x[2];
};
template <>
struct VecF<4> {
    float x[4];
};

template <int VPL>
__device__ __forceinline__ void ld_row(const float *p, float (&r)[VPL]) {
    if constexpr (VPL == 4) {
        float4 t = __ldcs(reinterpret_cast<const float4 *>(p));
        r[0] = t.x; r[1] = t.y; r[2] = t.z; r[3] = t.w;
    } else if constexpr (VPL == 2) {
        float2 t = __ldcs(reinterpret_cast<const float2 *>(p));
        r[0] = t.x; r[1] = t.y;
    } else {
        r[0] = __ldcs(p);
    }
}

template <int VPL>
__device__ __forceinline__ void st_row(float *p, const float (&r)[VPL]) {
    if constexpr (VPL == 4) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(r[0], r[1], r[2], r[3]));
    } else if constexpr (VPL == 2) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(r[0], r[1]));
    } else {
        __stcs(p, r[0]);
    }
}

// GL: g and beta come from their logits (a compile-time choice, so the plain path keeps
// its schedule).
template <int K, int V, bool GL>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(const SeqParams p) {
    constexpr int RPW = K / kWarps;  // rows per warp
    constexpr int VPL = V / 32;      // columns per lane
    static_assert(K % kWarps == 0 && V % 32 == 0 && K <= kThreads && V <= 128, "shape");

    __shared__ float sq[K], sk[K], se[K];
    __shared__ float sv[V], sd[V];
    __shared__ float red_u[kWarps][V], red_q[kWarps][V];
    __shared__ float misc[kWarps][4];

    const int H = p.H;
    const int unit = blockIdx.x;
    const int n = unit / H, h = unit % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int bos, len;
    seq_range(p, n, bos, len);

    const size_t state_off = (size_t)unit * K * V;
    float s[RPW][VPL];
    // Issue every state load first so they are in flight during the q/k prologue.
    if (p.s0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            ld_row<VPL>(p.s0 + state_off + (size_t)(warp * RPW + r) * V + lane * VPL, s[r]);
    } else {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int c = 0; c < VPL; ++c) s[r][c] = 0.f;
    }

    for (int t = 0; t < len; ++t) {
        const size_t row = (size_t)(bos + t);
        const size_t hk = (row * H + h) * K, hv = (row * H + h) * V;
        // -- prologue: load q, k, exp(g), v; partial norms
        float pq = 0.f, pk = 0.f, pqk = 0.f;
        if (tid < K) {
            const float qv = ld_in(p.q, hk + tid, p.qkv_bf16);
            const float kv = ld_in(p.k, hk + tid, p.qkv_bf16);
            sq[tid] = qv;
            sk[tid] = kv;
            se[tid] = __expf(GL ? load_g(p, hk + tid, h, tid) : p.g[hk + tid]);
            pq = qv * qv;
            pk = kv * kv;
            pqk = qv * kv;
        }
        if (tid >= kThreads - V) sv[tid - (kThreads - V)] = ld_in(p.v, hv + tid - (kThreads - V), p.qkv_bf16);
        pq = warp_sum(pq);
        pk = warp_sum(pk);
        pqk = warp_sum(pqk);
        if (lane == 0) {
            misc[warp][0] = pq;
            misc[warp][1] = pk;
            misc[warp][2] = pqk;
        }
        __syncthreads();
        float ssq = 0.f, ssk = 0.f, sqk = 0.f;
#pragma unroll
        for (int w = 0; w < (K + 31) / 32; ++w) {
            ssq += misc[w][0];
            ssk += misc[w][1];
            sqk += misc[w][2];
        }
        const float rq = p.l2norm ? rsqrtf(ssq + 1e-6f) : 1.f;
        const float rk = p.l2norm ? rsqrtf(ssk + 1e-6f) : 1.f;
        const float kq = sqk * rq * rk;  // k^ . q^

        // -- decay rows, partial u = S'^T k^ and p = S'^T q^
        float pu[VPL], pp[VPL];
#pragma unroll
        for (int c = 0; c < VPL; ++c) pu[c] = pp[c] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int i = warp * RPW + r;
            const float e = se[i], ki = sk[i] * rk, qi = sq[i] * rq;
#pragma unroll
            for (int c = 0; c < VPL; ++c) {
                s[r][c] *= e;
                pu[c] = fmaf(ki, s[r][c], pu[c]);
                pp[c] = fmaf(qi, s[r][c], pp[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
            red_u[warp][lane * VPL + c] = pu[c];
            red_q[warp][lane * VPL + c] = pp[c];
        }
        __syncthreads();

        // -- delta and output, one thread per value column
        float ov = 0.f;
        if (tid < V) {
            float u = 0.f, pv = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                u += red_u[w][tid];
                pv += red_q[w][tid];
            }
            const float b = GL ? load_beta(p, row * H + h) : p.beta[row * H + h];
            const float d = b * (sv[tid] - u);
            sd[tid] = d;
            ov = p.scale * fmaf(kq, d, pv);
            if (p.o) st_out(p.o, hv + tid, ov, p.o_bf16);
        }
        if (p.gate) {
            // sigmoid-gated RMSNorm over the V outputs of this head
            float sq2 = warp_sum(tid < V ? ov * ov : 0.f);
            if (lane == 0) misc[warp][3] = sq2;
        }
        __syncthreads();
        if (p.gate && tid < V) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < V / 32; ++w) ss += misc[w][3];
            const float inv = rsqrtf(ss / (float)V + p.eps);
            const float gt = ld_in(p.gate, hv + tid, p.gate_bf16);
            st_out(p.y, hv + tid, ov * inv * p.norm_w[tid] * sigmoidf_(gt), p.o_bf16);
        }

        // -- rank-one write
        float dl[VPL];
#pragma unroll
        for (int c = 0; c < VPL; ++c) dl[c] = sd[lane * VPL + c];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float ki = sk[warp * RPW + r] * rk;
#pragma unroll
            for (int c = 0; c < VPL; ++c) s[r][c] = fmaf(ki, dl[c], s[r][c]);
        }
        if (p.states) {
            const size_t so = row * H * (size_t)K * V + (size_t)h * K * V;
#pragma unroll
            for (int r = 0; r < RPW; ++r)
                st_row<VPL>(p.states + so + (size_t)(warp * RPW + r) * V + lane * VPL, s[r]);
        }
        __syncthreads();  // shared buffers are rewritten by the next token
    }

    if (p.sT) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
            st_row<VPL>(p.sT + state_off + (size_t)(warp * RPW + r) * V + lane * VPL, s[r]);
    }
}

// ---------------------------------------------------------------------------
// Decode step (one token per sequence, dense batch, K = V = 128).  The same arithmetic
// and thread mapping as recurrent_kernel, but persistent: two CTAs per SM walk the
// (sequence, head) units with the grid as stride.  While one unit is computed from
// registers, the next unit's 64 KiB state and its q, k, v, g and gate rows are already
// on their way into shared memory (bulk copies on an mbarrier), so each SM keeps about
// 128 KiB of reads in flight instead of stalling at every CTA's start.

constexpr int kDK = 128;                 // K = V
// One unit's staging buffer: state [128][128] fp32, then the q, k, v, g and gate rows; with
// the fused short convolutions also the three filters' weights (128 channels x up to 4
// taps each) and their histories (up to 3 rows of 128 channels each).
constexpr uint32_t S_Q = 65536, S_K = S_Q + 512, S_V = S_K + 512, S_G = S_V + 512, S_GATE = S_G + 512;
constexpr uint32_t S_CW = S_GATE + 512, S_CS = S_CW + 3 * 2048;
constexpr uint32_t kDecodePolls = 1u << 26;
template <bool CV>
constexpr uint32_t kStage = CV ? S_CS + 9 * 512 : S_CW;

// Shared-memory layout of the decode kernel with NW warps and NS staging buffers.
template <int NW, int NS, bool CV>
struct DecodeSmem {
    static constexpr uint32_t arr = NS * kStage<CV>;           // sq, sk, se, sv, sd: [128] floats each
    static constexpr uint32_t red = arr + 5 * 512;             // red_u, red_q: [NW][128] floats each
    static constexpr uint32_t misc = red + 2 * NW * 512;       // [NW][4] floats
    static constexpr uint32_t bar = misc + NW * 16;            // NS mbarriers
    static constexpr uint32_t bytes = bar + NS * 8;
};

// Set by a CTA whose bounded wait on its copies gave up; that unit and every later unit
// the CTA owned get NaN in their state, o and y.
__device__ int g_decode_timeouts = 0;

__device__ __forceinline__ float in_elem(const uint8_t *base, int i, int is_bf16) {
    return is_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i])
                   : reinterpret_cast<const float *>(base)[i];
}

// Fused short convolution of channel c through filter f of a staged unit:
//   z = sum_{j < W-1} w[j] * hist[j] + w[W-1] * x,   returns SiLU(z) = z / (1 + e^-z)
// (hist = the W-1 inputs before this token, oldest first; zero without history), and
// writes the channel's new history (hist[1..], x) to out, rows out_stride floats apart.
__device__ __forceinline__ float conv_silu(const uint8_t *buf, int f, int c, float x, int W, bool hist, float *out,
                                           size_t out_stride) {
    const float *w = reinterpret_cast<const float *>(buf + S_CW + f * 2048) + c * W;
    const float *h = reinterpret_cast<const float *>(buf + S_CS + f * 3 * 512) + c;
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        if (j >= W - 1) break;
        const float hj = hist ? h[j * kDK] : 0.f;
        z = fmaf(w[j], hj, z);
        out[j * out_stride] = j + 1 < W - 1 ? (hist ? h[(j + 1) * kDK] : 0.f) : x;
    }
    z = fmaf(w[W - 1], x, z);
    return __fdividef(z, 1.f + __expf(-z));
}

// NW warps (warp w owns rows [w * 128 / NW, (w + 1) * 128 / NW) of the state, lane l the
// columns 4l .. 4l+3) and NS staging buffers: the copies of the NS units after the one
// being computed are in flight.  CV: q, k and v pass through their short convolutions
// (+ SiLU) first, with the filters and histories staged alongside the unit.
template <bool GL, bool CV, int NW, int NS>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) decode_kernel(const SeqParams p) {
    using L = DecodeSmem<NW, NS, CV>;
    constexpr uint32_t kStg = kStage<CV>;
    static_assert(!CV || NW * 32 >= 2 * kDK, "the fused convolutions give q, k and v to disjoint threads");
    constexpr int NT = NW * 32, RPW = kDK / NW, VPL = kDK / 32;
    extern __shared__ __align__(1024) uint8_t dsm[];
    const uint32_t sb = tc::smem_u32(dsm);
    float *sq = reinterpret_cast<float *>(dsm + L::arr), *sk = sq + kDK, *se = sk + kDK, *sv = se + kDK,
          *sd = sv + kDK;
    float(*red_u)[kDK] = reinterpret_cast<float(*)[kDK]>(dsm + L::red);
    float(*red_q)[kDK] = reinterpret_cast<float(*)[kDK]>(dsm + L::red + NW * 512);
    float(*misc)[4] = reinterpret_cast<float(*)[4]>(dsm + L::misc);
    uint64_t *bars = reinterpret_cast<uint64_t *>(dsm + L::bar);

    const int H = p.H, units = p.N * p.H, stride = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t eq = p.qkv_bf16 ? 2 : 4;
    const void *gsrc = GL ? p.g_logits : static_cast<const void *>(p.g);
    const uint32_t eg = GL && p.g_logits_bf16 ? 2 : 4, eo = p.gate_bf16 ? 2 : 4;
    const int W = CV ? p.conv_w : 0;
    const bool hist = CV && p.cs_in[0];
    const size_t cD = (size_t)H * kDK;  // channels of each convolution
    const uint32_t tx = (p.s0 ? 65536u : 0u) + 3u * kDK * eq + kDK * eg + (p.gate ? kDK * eo : 0u) +
                        (CV ? 3u * kDK * 4u * W + (hist ? 3u * (W - 1) * 512u : 0u) : 0u);
    auto issue = [&](int u, int st) {  // thread 0: every copy of unit u into buffer st
        uint64_t *bar = bars + st;
        const uint32_t d = sb + (uint32_t)st * kStg;
        tc::mbar_arrive_expect_tx(bar, tx);
        if (p.s0) tc::bulk_load(d, p.s0 + (size_t)u * kDK * kDK, 65536u, bar);
        tc::bulk_load(d + S_Q, static_cast<const uint8_t *>(p.q) + (size_t)u * kDK * eq, kDK * eq, bar);
        tc::bulk_load(d + S_K, static_cast<const uint8_t *>(p.k) + (size_t)u * kDK * eq, kDK * eq, bar);
        tc::bulk_load(d + S_V, static_cast<const uint8_t *>(p.v) + (size_t)u * kDK * eq, kDK * eq, bar);
        tc::bulk_load(d + S_G, static_cast<const uint8_t *>(gsrc) + (size_t)u * kDK * eg, kDK * eg, bar);
        if (p.gate)
            tc::bulk_load(d + S_GATE, static_cast<const uint8_t *>(p.gate) + (size_t)u * kDK * eo, kDK * eo, bar);
        if constexpr (CV) {
            const int n = u / H, h = u - n * H;
            for (int f = 0; f < 3; ++f) {
                tc::bulk_load(d + S_CW + f * 2048, p.cw[f] + (size_t)h * kDK * W, kDK * 4u * W, bar);
                if (hist)
                    for (int j = 0; j < W - 1; ++j)
                        tc::bulk_load(d + S_CS + (f * 3 + j) * 512,
                                      p.cs_in[f] + ((size_t)n * (W - 1) + j) * cD + (size_t)h * kDK, 512u, bar);
            }
        }
    };
    // beta (or its logit) and, with logits, the head's A_log and this thread's dt_bias:
    // loaded one unit ahead, into registers
    auto pre_beta = [&](int u) {
        if (u >= units) return 0.f;
        return GL ? ld_in(p.beta_logits, (size_t)u, p.beta_logits_bf16) : __ldg(p.beta + u);
    };
    auto pre_alog = [&](int u) { return GL && u < units ? __ldg(p.A_log + u % H) : 0.f; };
    auto pre_db = [&](int u) {
        return GL && u < units && p.dt_bias && tid < kDK ? __ldg(p.dt_bias + (size_t)(u % H) * kDK + tid) : 0.f;
    };

    if (tid == 0) {
        for (int st = 0; st < NS; ++st) tc::mbar_init(bars + st, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    int u = blockIdx.x;
    if (tid == 0)
        for (int st = 0; st < NS; ++st)
            if (u + st * stride < units) issue(u + st * stride, st);
    const float nw = p.gate && tid < kDK ? p.norm_w[tid] : 0.f;
    float b_cur = pre_beta(u), al_cur = pre_alog(u), db_cur = pre_db(u);
    int it = 0;
    bool failed = false;
    for (; u < units; u += stride, ++it) {
        const int st = it % NS;
        const uint8_t *buf = dsm + (uint32_t)st * kStg;
        failed = __syncthreads_or(!tc::mbar_wait(bars + st, (uint32_t)((it / NS) & 1), p.polls));
        if (failed) break;  // the copies did not arrive in time: this unit and the rest are poisoned below
        float s[RPW][VPL];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            if (p.s0) {
                const float4 t = *reinterpret_cast<const float4 *>(buf + ((warp * RPW + r) * kDK + lane * VPL) * 4);
                s[r][0] = t.x; s[r][1] = t.y; s[r][2] = t.z; s[r][3] = t.w;
            } else {
#pragma unroll
                for (int c = 0; c < VPL; ++c) s[r][c] = 0.f;
            }
        }
        // -- prologue from the staged rows: q, k, exp(g), v, the gate; partial norms
        float pq = 0.f, pk = 0.f, pqk = 0.f, gt = 0.f;
        // the unit's row of each new convolution history: channel c of row j at [j * cD + c]
        const size_t cs_row = CV ? ((size_t)(u / H) * (W - 1)) * cD + (size_t)(u % H) * kDK : 0;
        if (tid < kDK) {
            float qv = in_elem(buf + S_Q, tid, p.qkv_bf16), kv = in_elem(buf + S_K, tid, p.qkv_bf16);
            if constexpr (CV) {
                qv = conv_silu(buf, 0, tid, qv, W, hist, p.cs_out[0] + cs_row + tid, cD);
                kv = conv_silu(buf, 1, tid, kv, W, hist, p.cs_out[1] + cs_row + tid, cD);
            }
            const float z = in_elem(buf + S_G, tid, GL ? p.g_logits_bf16 : 0);
            sq[tid] = qv;
            sk[tid] = kv;
            se[tid] = __expf(GL ? gate_of_logit(z + db_cur, __expf(al_cur), p.g_lower) : z);
            pq = qv * qv;
            pk = kv * kv;
            pqk = qv * kv;
            if (p.gate) gt = in_elem(buf + S_GATE, tid, p.gate_bf16);
        }
        if (tid >= NT - kDK) {
            const int c = tid - (NT - kDK);
            float vv = in_elem(buf + S_V, c, p.qkv_bf16);
            if constexpr (CV) vv = conv_silu(buf, 2, c, vv, W, hist, p.cs_out[2] + cs_row + c, cD);
            sv[c] = vv;
        }
        pq = warp_sum(pq);
        pk = warp_sum(pk);
        pqk = warp_sum(pqk);
        if (lane == 0) {
            misc[warp][0] = pq;
            misc[warp][1] = pk;
            misc[warp][2] = pqk;
        }
        tc::fence_async_smem();  // these reads of the buffer come before the next copies into it
        __syncthreads();         // the staged rows are consumed: the buffer takes unit u + NS * stride
        if (tid == 0 && u + NS * stride < units) issue(u + NS * stride, st);
        const int un = u + stride;
        const float b_next = pre_beta(un), al_next = pre_alog(un), db_next = pre_db(un);
        float ssq = 0.f, ssk = 0.f, sqk = 0.f;
#pragma unroll
        for (int w = 0; w < kDK / 32; ++w) {
            ssq += misc[w][0];
            ssk += misc[w][1];
            sqk += misc[w][2];
        }
        const float rq = p.l2norm ? rsqrtf(ssq + 1e-6f) : 1.f;
        const float rk = p.l2norm ? rsqrtf(ssk + 1e-6f) : 1.f;
        const float kq = sqk * rq * rk;  // k^ . q^

        // -- decay rows, partial u = S'^T k^ and p = S'^T q^
        float pu[VPL], pp[VPL];
#pragma unroll
        for (int c = 0; c < VPL; ++c) pu[c] = pp[c] = 0.f;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const int i = warp * RPW + r;
            const float e = se[i], ki = sk[i] * rk, qi = sq[i] * rq;
#pragma unroll
            for (int c = 0; c < VPL; ++c) {
                s[r][c] *= e;
                pu[c] = fmaf(ki, s[r][c], pu[c]);
                pp[c] = fmaf(qi, s[r][c], pp[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < VPL; ++c) {
            red_u[warp][lane * VPL + c] = pu[c];
            red_q[warp][lane * VPL + c] = pp[c];
        }
        __syncthreads();

        // -- delta and output, one thread per value column
        const size_t hv = (size_t)u * kDK;
        float ov = 0.f;
        if (tid < kDK) {
            float uu = 0.f, pv = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                uu += red_u[w][tid];
                pv += red_q[w][tid];
            }
            const float b = GL ? beta_of_logit(b_cur) : b_cur;
            const float d = b * (sv[tid] - uu);
            sd[tid] = d;
            ov = p.scale * fmaf(kq, d, pv);
            if (p.o) st_out(p.o, hv + tid, ov, p.o_bf16);
        }
        if (p.gate) {
            const float sq2 = warp_sum(tid < kDK ? ov * ov : 0.f);
            if (lane == 0) misc[warp][3] = sq2;
        }
        __syncthreads();
        if (p.gate && tid < kDK) {
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < kDK / 32; ++w) ss += misc[w][3];
            const float inv = rsqrtf(ss / (float)kDK + p.eps);
            st_out(p.y, hv + tid, ov * inv * nw * sigmoidf_(gt), p.o_bf16);
        }

        // -- rank-one write, straight from registers to the state output
        float dl[VPL];
#pragma unroll
        for (int c = 0; c < VPL; ++c) dl[c] = sd[lane * VPL + c];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float ki = sk[warp * RPW + r] * rk;
#pragma unroll
            for (int c = 0; c < VPL; ++c) s[r][c] = fmaf(ki, dl[c], s[r][c]);
            st_row<VPL>(p.sT + (size_t)u * kDK * kDK + (size_t)(warp * RPW + r) * kDK + lane * VPL, s[r]);
        }
        b_cur = b_next;
        al_cur = al_next;
        db_cur = db_next;
        __syncthreads();  // shared arrays are rewritten by the next unit
    }
    if (!failed) return;
    // After a failure: the copies still in flight (iterations it .. it + NS - 1) get their
    // full bounded time to land, then unit u and every later unit of this CTA is poisoned,
    // so that no output of the call keeps an old value that would pass for a result (with
    // the state updated in place, an unwritten unit would still hold its previous state).
    if (tid == 0) {
        atomicAdd(&g_decode_timeouts, 1);
        for (int k = 0; k < NS; ++k) {
            const int j = it + k, uj = blockIdx.x + j * stride;
            if (uj < units) tc::mbar_wait(bars + j % NS, (uint32_t)((j / NS) & 1), kDecodePolls);
        }
    }
    __syncthreads();
    const float nan = __int_as_float(0x7fc00000);
    for (; u < units; u += stride) {
        for (int e = tid; e < kDK * kDK; e += NT) p.sT[(size_t)u * kDK * kDK + e] = nan;
        if (tid < kDK) {
            if (p.o) st_out(p.o, (size_t)u * kDK + tid, nan, p.o_bf16);
            if (p.gate) st_out(p.y, (size_t)u * kDK + tid, nan, p.o_bf16);
            if constexpr (CV) {
                const size_t row = ((size_t)(u / H) * (W - 1)) * cD + (size_t)(u % H) * kDK + tid;
                for (int f = 0; f < 3; ++f)
                    for (int j = 0; j < W - 1; ++j) p.cs_out[f][row + j * cD] = nan;
            }
        }
    }
}

// Decode configuration: NW warps per CTA, NS staging buffers (CTAs per SM follow from
// the registers and shared memory: 2 for 8 warps and one buffer, 1 for 16 warps and 2
// or 3).  Measured at B = 256: 8 warps / 1 buffer 0.515 ms, 16 / 2 0.527 ms, 16 / 3
// 0.530 ms.
constexpr int kDecNW = 8, kDecNS = 1;

template <int K, int V>
kda_status launch_kv(const SeqParams &p, cudaStream_t st) {
    const int units = p.N * p.H;
    if (units == 0) return KDA_OK;
    if (K == kDK && V == kDK && p.T == 1 && !p.cu_seqlens && !p.states && p.sT) {
        using L = DecodeSmem<kDecNW, kDecNS, false>;
        using LC = DecodeSmem<kDecNW, kDecNS, true>;
        static DeviceOnce configured;
        const int dev = current_device();
        if (!configured.done(dev)) {
            const struct {
                const void *fn;
                uint32_t bytes;
            } fns[] = {{(const void *)decode_kernel<false, false, kDecNW, kDecNS>, L::bytes},
                       {(const void *)decode_kernel<true, false, kDecNW, kDecNS>, L::bytes},
                       {(const void *)decode_kernel<false, true, kDecNW, kDecNS>, LC::bytes},
                       {(const void *)decode_kernel<true, true, kDecNW, kDecNS>, LC::bytes}};
            for (const auto &f : fns) {
                const cudaError_t e = cudaFuncSetAttribute(f.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, f.bytes);
                if (e != cudaSuccess) {
                    set_error("decode: cannot reserve %u bytes of shared memory: %s", f.bytes, cudaGetErrorString(e));
                    return KDA_ERR_CUDA;
                }
            }
            configured.set(dev);
        }
        const int per_sm = kDecNW == 8 ? 2 : 1;
        const int grid = units < per_sm * sm_count() ? units : per_sm * sm_count();
        if (p.conv_w) {
            if (p.g_logits)
                decode_kernel<true, true, kDecNW, kDecNS><<<grid, kDecNW * 32, LC::bytes, st>>>(p);
            else
                decode_kernel<false, true, kDecNW, kDecNS><<<grid, kDecNW * 32, LC::bytes, st>>>(p);
        } else if (p.g_logits) {
            decode_kernel<true, false, kDecNW, kDecNS><<<grid, kDecNW * 32, L::bytes, st>>>(p);
        } else {
            decode_kernel<false, false, kDecNW, kDecNS><<<grid, kDecNW * 32, L::bytes, st>>>(p);
        }
        note_launch();
        return check_launch("decode_kernel");
    }
    if (p.conv_w) {
        set_error("recurrent: the fused short convolutions need the decode step (K = V = 128, T = 1, dense)");
        return KDA_ERR_UNSUPPORTED;
    }
    if (p.g_logits)
        recurrent_kernel<K, V, true><<<units, kThreads, 0, st>>>(p);
    else
        recurrent_kernel<K, V, false><<<units, kThreads, 0, st>>>(p);
    note_launch();
    return check_launch("recurrent_kernel");
}

}  // namespace

int take_decode_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_decode_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_decode_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("decode: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

kda_status launch_recurrent(const SeqParams &p, int K, int V, cudaStream_t st) {
#define KDA_CASE(KK, VV) \
    if (K == KK && V == VV) return launch_kv<KK, VV>(p, st);
    KDA_CASE(128, 128)
    KDA_CASE(64, 64)
    KDA_CASE(32, 32)
    KDA_CASE(128, 64)
    KDA_CASE(64, 128)
    KDA_CASE(128, 32)
    KDA_CASE(32, 128)
    KDA_CASE(64, 32)
    KDA_CASE(32, 64)
#undef KDA_CASE
    set_error("recurrent: K=%d V=%d not built (K, V in {32, 64, 128})", K, V);
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
