// kda_chunk_fp32.cu -- chunked KDA prefill in fp32 on CUDA cores.
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (a prompt runs
// a chunked kernel that carries the state from one 64-token chunk to the next),
// sections 03/04 for the recurrence itself (per-key-channel decay before each
// delta-rule update, in-kernel L2 norm of q and k).
//
// Chunk algebra (derived from the recurrence; exact in real arithmetic).  For a
// chunk of C tokens starting from state S, with G_i = sum_{s<=i} g_s (inclusive
// cumulative log decay inside the chunk, a K-vector) and gamma = G_{C-1}:
//   A[i][j] = beta_i sum_c k^_i[c] k^_j[c] exp(G_i[c] - G_j[c])      (j < i)
//   P[i][j] =        sum_c q^_i[c] k^_j[c] exp(G_i[c] - G_j[c])      (j <= i)
//   T       = (I + A)^-1                         (unit lower triangular)
//   Kd = k^ * exp(G),  Qd = q^ * exp(G),  Kg = k^ * exp(gamma - G)
//   D       = T diag(beta) (V - Kd S)            (the chunk's write residuals)
//   O       = Qd S + P D
//   S'      = Diag(exp gamma) S + Kg^T D
// Every exponential here has a non-positive argument, so nothing overflows for
// any g <= 0.  Pairwise exponentials make this path slow; it is the fp32
// reference mode of the library and the path for small head sizes / chunks.
//
// One CTA per (sequence, head, 32-wide slice of V): value columns evolve
// independently, so slices only repeat the key-side work.
#include <math.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int VS = 32;  // value columns per CTA

template <int K, int C>
struct Smem {
    // padded rows avoid bank conflicts on column walks
    static constexpr int KP = K + 1, CP = C + 1, VP = VS + 1;
    static constexpr size_t qh = 0;                        // [C][KP]  q^ (scaled) -> Qd
    static constexpr size_t kh = qh + C * KP;              // [C][KP]  k^ -> Kd
    static constexpr size_t G = kh + C * KP;               // [C][KP]  G -> Kg
    static constexpr size_t A = G + C * KP;                // [C][CP]
    static constexpr size_t Tm = A + C * CP;               // [C][CP]
    static constexpr size_t P = Tm + C * CP;               // [C][CP]
    static constexpr size_t S = P + C * CP;                // [K][VP]
    static constexpr size_t R = S + K * VP;                // [C][VP]  rhs, then D
    static constexpr size_t D = R + C * VP;                // [C][VP]
    static constexpr size_t gam = D + C * VP;              // [K]  exp(gamma)
    static constexpr size_t bet = gam + K;                 // [C]
    static constexpr size_t total = bet + C;
    static constexpr size_t bytes = total * sizeof(float);
};

template <int K, int C>
__global__ void __launch_bounds__(kThreads) chunk_fp32_kernel(const SeqParams p, const int V,
                                                              const int *order) {
    using L = Smem<K, C>;
    extern __shared__ float sm[];
    float *qh = sm + L::qh, *kh = sm + L::kh, *G = sm + L::G;
    float *A = sm + L::A, *Tm = sm + L::Tm, *P = sm + L::P, *S = sm + L::S;
    float *R = sm + L::R, *D = sm + L::D, *gam = sm + L::gam, *bet = sm + L::bet;
    constexpr int KP = L::KP, CP = L::CP, VP = L::VP;

    const int nslices = V / VS;
    const int H = p.H;
    int unit = blockIdx.x / nslices;
    const int slice = blockIdx.x % nslices;
    if (order) unit = order[unit];
    const int n = unit / H, h = unit % H;
    const int c0 = slice * VS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int bos, len;
    seq_range(p, n, bos, len);

    // state slice S[K][VS]
    for (int e = tid; e < K * VS; e += kThreads) {
        const int i = e / VS, j = e % VS;
        S[i * VP + j] = p.s0 ? p.s0[((size_t)unit * K + i) * V + c0 + j] : 0.f;
    }

    for (int t0 = 0; t0 < len; t0 += C) {
        const int cn = min(C, len - t0);  // valid tokens in this chunk
        __syncthreads();
        // -- load: normalise q, k per token (one warp per token), stage g and beta
        for (int i = warp; i < C; i += kWarps) {
            const size_t row = (size_t)(bos + t0 + i);
            const size_t hk = (row * H + h) * K;
            float aq = 0.f, ak = 0.f;
            for (int c = lane; c < K; c += 32) {
                float qv = 0.f, kv = 0.f, gv = 0.f;
                if (i < cn) {
                    qv = ld_in(p.q, hk + c, p.qkv_bf16);
                    kv = ld_in(p.k, hk + c, p.qkv_bf16);
                    gv = load_g(p, hk + c, h, c);
                }
                qh[i * KP + c] = qv;
                kh[i * KP + c] = kv;
                G[i * KP + c] = gv;
                aq += qv * qv;
                ak += kv * kv;
            }
            aq = warp_sum(aq);
            ak = warp_sum(ak);
            const float rq = (p.l2norm ? rsqrtf(aq + 1e-6f) : 1.f) * p.scale;
            const float rk = p.l2norm ? rsqrtf(ak + 1e-6f) : 1.f;
            for (int c = lane; c < K; c += 32) {
                qh[i * KP + c] *= rq;
                kh[i * KP + c] *= rk;
            }
            if (lane == 0) bet[i] = i < cn ? load_beta(p, row * H + h) : 0.f;
        }
        __syncthreads();
        // -- inclusive cumulative decay G (one thread per key channel)
        for (int c = tid; c < K; c += kThreads) {
            float acc = 0.f;
            for (int i = 0; i < C; ++i) {
                acc += G[i * KP + c];
                G[i * KP + c] = acc;
            }
            gam[c] = acc;
        }
        __syncthreads();
        // -- grams A (strict lower, beta-scaled) and P (lower incl. diagonal): one warp per pair
        for (int pr = warp; pr < C * C; pr += kWarps) {
            const int i = pr / C, j = pr % C;
            if (j > i) {
                if (lane == 0) {
                    A[i * CP + j] = 0.f;
                    P[i * CP + j] = 0.f;
                }
                continue;
            }
            float a = 0.f, b = 0.f;
            for (int c = lane; c < K; c += 32) {
                const float e = __expf(G[i * KP + c] - G[j * KP + c]);
                const float kj = kh[j * KP + c] * e;
                a = fmaf(kh[i * KP + c], kj, a);
                b = fmaf(qh[i * KP + c], kj, b);
            }
            a = warp_sum(a);
            b = warp_sum(b);
            if (lane == 0) {
                A[i * CP + j] = (j < i) ? bet[i] * a : 0.f;
                P[i * CP + j] = b;
            }
        }
        __syncthreads();
        // -- Qd, Kd, Kg in place (each element touched by one thread)
        for (int e = tid; e < C * K; e += kThreads) {
            const int i = e / K, c = e % K;
            const float gi = G[i * KP + c];
            const float ed = __expf(gi), eg = __expf(gam[c] - gi);
            const float kv = kh[i * KP + c];
            qh[i * KP + c] *= ed;
            kh[i * KP + c] = kv * ed;
            G[i * KP + c] = kv * eg;
        }
        // -- T = (I + A)^-1 by forward substitution, one thread per column
        for (int i = 0; i < C; ++i) {
            if (tid < C) {
                const int col = tid;
                float x = (i == col) ? 1.f : 0.f;
                for (int j = col; j < i; ++j) x = fmaf(-A[i * CP + j], Tm[j * CP + col], x);
                Tm[i * CP + col] = (col <= i) ? x : 0.f;
            }
            __syncthreads();
        }
        // -- R = diag(beta) (V - Kd S)
        for (int e = tid; e < C * VS; e += kThreads) {
            const int i = e / VS, j = e % VS;
            float acc = 0.f;
            for (int c = 0; c < K; ++c) acc = fmaf(kh[i * KP + c], S[c * VP + j], acc);
            float vv = 0.f;
            if (i < cn) vv = ld_in(p.v, ((size_t)(bos + t0 + i) * H + h) * V + c0 + j, p.qkv_bf16);
            R[i * VP + j] = bet[i] * (vv - acc);
        }
        __syncthreads();
        // -- D = T R
        for (int e = tid; e < C * VS; e += kThreads) {
            const int i = e / VS, j = e % VS;
            float acc = 0.f;
            for (int m = 0; m <= i; ++m) acc = fmaf(Tm[i * CP + m], R[m * VP + j], acc);
            D[i * VP + j] = acc;
        }
        __syncthreads();
        // -- O = Qd S + P D  (written straight to global)
        if (p.o) {
            for (int e = tid; e < C * VS; e += kThreads) {
                const int i = e / VS, j = e % VS;
                if (i >= cn) continue;
                float acc = 0.f;
                for (int c = 0; c < K; ++c) acc = fmaf(qh[i * KP + c], S[c * VP + j], acc);
                for (int m = 0; m <= i; ++m) acc = fmaf(P[i * CP + m], D[m * VP + j], acc);
                st_out(p.o, ((size_t)(bos + t0 + i) * H + h) * V + c0 + j, acc, p.o_bf16);
            }
        }
        __syncthreads();
        // -- S = Diag(exp gamma) S + Kg^T D
        for (int e = tid; e < K * VS; e += kThreads) {
            const int c = e / VS, j = e % VS;
            float acc = __expf(gam[c]) * S[c * VP + j];
            for (int m = 0; m < C; ++m) acc = fmaf(G[m * KP + c], D[m * VP + j], acc);
            S[c * VP + j] = acc;
        }
    }
    __syncthreads();
    if (p.sT) {
        for (int e = tid; e < K * VS; e += kThreads) {
            const int i = e / VS, j = e % VS;
            p.sT[((size_t)unit * K + i) * V + c0 + j] = S[i * VP + j];
        }
    }
}

template <int K, int C>
kda_status launch_kc(const SeqParams &p, int V, const int *order, cudaStream_t st) {
    using L = Smem<K, C>;
    const int units = p.N * p.H;
    if (units == 0) return KDA_OK;
    static DeviceOnce configured;  // benign race: the attribute call is idempotent
    const int dev = current_device();
    if (!configured.done(dev)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_fp32_kernel<K, C>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
        if (e != cudaSuccess) {
            set_error("chunk_fp32: cannot reserve %zu bytes of shared memory: %s", L::bytes,
                      cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
        configured.set(dev);
    }
    chunk_fp32_kernel<K, C><<<units * (V / VS), kThreads, L::bytes, st>>>(p, V, order);
    note_launch();
    return check_launch("chunk_fp32_kernel");
}

}  // namespace

kda_status launch_chunk_fp32(const SeqParams &p, int K, int V, int chunk, const int *order,
                             cudaStream_t st) {
    if (V % VS != 0) {
        set_error("chunk_fp32: V=%d must be a multiple of %d", V, VS);
        return KDA_ERR_UNSUPPORTED;
    }
#define KDA_CASE(KK, CC) \
    if (K == KK && chunk == CC) return launch_kc<KK, CC>(p, V, order, st);
    KDA_CASE(128, 64)
    KDA_CASE(128, 32)
    KDA_CASE(128, 16)
    KDA_CASE(64, 64)
    KDA_CASE(64, 32)
    KDA_CASE(64, 16)
    KDA_CASE(32, 64)
    KDA_CASE(32, 32)
    KDA_CASE(32, 16)
#undef KDA_CASE
    set_error("chunk_fp32: K=%d chunk=%d not built (K in {32,64,128}, chunk in {16,32,64})", K, chunk);
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
