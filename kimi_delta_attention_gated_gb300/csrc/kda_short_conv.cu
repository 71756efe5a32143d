// kda_short_conv.cu -- causal depthwise short convolution (+ SiLU) of q, k and v.
//
// Pages: nnterp encyclopedia "Kimi-Linear", section "Printout" (the layer's conv1d
// is Conv1d(12288, 12288, kernel_size=(4,), padding=(3,), groups=12288,
// bias=False): one 4-tap filter per channel along the sequence, padded by 3
// before the first token, the first T outputs kept); Kimi-K3 atlas "gate-project
// (decode, P = 1000)", section "Code" (q_conv1d, k_conv1d, v_conv1d =
// ShortConvolution(hidden_size, kernel_size=4, activation='silu')).
//
//   y[t][c] = act( bias[c] + sum_{w<W} weight[c][w] * x[t - (W-1) + w][c] )
//
// with positions before a sequence taken from its conv state (the W-1 inputs
// before it, oldest first) or zero.  The state after the call is the last W-1
// inputs of each sequence.
//
// HBM-bound: every input is read once and every output written once.
//  * Prompts: persistent CTAs (as many as fit on the SMs) walk over tiles of 256
//    channels x 64 tokens of the packed token axis.  One thread keeps two tiles in
//    flight with TMA: each tile, with the W-1 rows before it (rows before 0 read as
//    zero), lands in one of two shared-memory buffers and completes on its own
//    mbarrier, so the next tile loads while this one is computed.  The 256 threads
//    each own 4 channels x 16 tokens of a tile, slide the W-1 previous inputs in
//    registers and store y with 8-byte stores (a warp covers 128 contiguous
//    channels of one row).  A sequence that starts inside the tile (varlen)
//    restarts the window from its own state; the thread that handles a sequence's
//    last token writes its new state.
//  * Decode (one token per sequence): one thread per (sequence, 4 channels) issues
//    its W-1 state loads and its input load together, then writes y and the
//    shifted state (in place allowed: each thread reads its state before writing it).
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_tc_ptx.cuh"

#include <string.h>

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;    // tokens per tile
constexpr int kCh = 256;     // channels per tile (the TMA box width)
constexpr int kVec = 4;      // channels per thread
constexpr int kTokPer = 16;  // tokens per thread: 64 channel groups x 4 token quarters = 256 threads
constexpr uint32_t kPolls = 1u << 24;  // bound on the wait that drains a tile still in flight
static_assert((kCh / kVec) * (kTile / kTokPer) == kThreads && kVec == 4, "thread map");

// Set by a CTA whose wait for its TMA tile gave up (its outputs, and the state of every
// sequence ending in one of its remaining tiles, are then NaN).
__device__ int g_short_conv_timeouts = 0;

struct ConvParams {
    const void *x;
    void *y;
    const float *w;     // [D, W]
    const float *bias;  // [D] or null
    const float *s0;    // [N, W-1, D] or null
    float *sT;          // [N, W-1, D] or null
    const int32_t *cu;  // [N + 1] device or null (dense: sequence n = rows [n T, n T + T))
    int64_t rows;       // packed tokens
    int N, T, D, act;
    uint32_t polls;     // bound on the wait for each tile
};

__device__ __forceinline__ int64_t clamp_row(int64_t v, int64_t rows) { return v < 0 ? 0 : (v > rows ? rows : v); }

// Sequence holding packed token t: the last n with cu[n] <= t (so its end lies past t
// for a valid cu_seqlens; a malformed one gives wrong but in-bounds results).
__device__ __forceinline__ void seq_of(const ConvParams &p, int64_t t, int &n, int64_t &bos, int64_t &eos) {
    if (!p.cu) {
        n = (int)(t / p.T);
        bos = (int64_t)n * p.T;
        eos = bos + p.T;
        return;
    }
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (clamp_row(p.cu[mid], p.rows) <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    n = lo;
    bos = clamp_row(p.cu[n], p.rows);
    eos = clamp_row(p.cu[n + 1], p.rows);
    if (bos > t) bos = t;      // only for a malformed cu_seqlens
    if (eos <= t) eos = t + 1;
}

// Vectors of kVec consecutive channels (4: 8 bytes of bf16 or 16 bytes of fp32).
template <bool BF16>
__device__ __forceinline__ void unpack_bf16(const uint32_t *w, float (&v)[kVec]) {
#pragma unroll
    for (int i = 0; i < kVec / 2; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <bool BF16>
__device__ __forceinline__ void ld_vec(const void *x, size_t idx, float (&v)[kVec]) {  // global, read-only
    if constexpr (BF16) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(x) + idx));
        const uint32_t w[2] = {u.x, u.y};
        unpack_bf16<true>(w, v);
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + idx));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
}

template <bool BF16>
__device__ __forceinline__ void lds_vec(const uint8_t *tile, size_t eidx, float (&v)[kVec]) {  // shared
    if constexpr (BF16) {
        const uint2 u = *reinterpret_cast<const uint2 *>(tile + eidx * 2);
        const uint32_t w[2] = {u.x, u.y};
        unpack_bf16<true>(w, v);
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(tile + eidx * 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    }
}

template <bool BF16>
__device__ __forceinline__ void st_vec(void *y, size_t idx, const float (&v)[kVec]) {  // global, streaming
    if constexpr (BF16) {
        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
        __stcs(reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(y) + idx),
               make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1)));
    } else {
        __stcs(reinterpret_cast<float4 *>(reinterpret_cast<float *>(y) + idx), make_float4(v[0], v[1], v[2], v[3]));
    }
}

__device__ __forceinline__ void ld_state(const float *s, size_t idx, float (&v)[kVec]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(s + idx));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}

__device__ __forceinline__ void st_state(float *s, size_t idx, const float (&v)[kVec]) {
    *reinterpret_cast<float4 *>(s + idx) = make_float4(v[0], v[1], v[2], v[3]);
}

template <int W>
__device__ __forceinline__ void load_filter(const ConvParams &p, int c0, float (&wv)[W][kVec], float (&bv)[kVec]) {
    const float4 *wp = reinterpret_cast<const float4 *>(p.w + (size_t)c0 * W);  // kVec W floats
    float wt[kVec * W];
#pragma unroll
    for (int i = 0; i < kVec * W / 4; ++i) {
        const float4 f = __ldg(wp + i);
        wt[4 * i] = f.x; wt[4 * i + 1] = f.y; wt[4 * i + 2] = f.z; wt[4 * i + 3] = f.w;
    }
#pragma unroll
    for (int e = 0; e < kVec; ++e)
#pragma unroll
        for (int w = 0; w < W; ++w) wv[w][e] = wt[e * W + w];
#pragma unroll
    for (int e = 0; e < kVec; ++e) bv[e] = p.bias ? __ldg(p.bias + c0 + e) : 0.f;
}

// SiLU as z / (1 + e^-z) with the fast divide: for z below about -88 the
// denominator is infinite and the result is -0, the correctly rounded limit.
template <int W, bool ACT>
__device__ __forceinline__ void conv_point(const float (&wv)[W][kVec], const float (&bv)[kVec],
                                           const float (&win)[W - 1][kVec], const float (&xv)[kVec],
                                           float (&z)[kVec]) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        float a = fmaf(wv[W - 1][e], xv[e], bv[e]);
#pragma unroll
        for (int j = 0; j < W - 1; ++j) a = fmaf(wv[j][e], win[j][e], a);
        z[e] = ACT ? __fdividef(a, 1.f + __expf(-a)) : a;
    }
}

// The tokens [ta, tb) of one tile for this thread's kVec channels: the window of the
// W-1 previous inputs slides in registers; sequence boundaries are counted down.
template <int W, bool XB, bool YB, bool ACT>
__device__ __forceinline__ void conv_tokens(const ConvParams &p, const uint8_t *tile, int64_t t0, int64_t ta,
                                            int64_t tb, int ch, int c0) {
    constexpr int NH = W - 1;
    constexpr int ES = XB ? 2 : 4, YS = YB ? 2 : 4;
    const size_t D = (size_t)p.D;
    float wv[W][kVec], bv[kVec];
    load_filter<W>(p, c0, wv, bv);
    int n;
    int64_t bos, eos;
    seq_of(p, ta, n, bos, eos);
    float win[NH][kVec];
    auto start_window = [&](int64_t t) {  // inputs t-NH .. t-1 of sequence n
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            const int64_t src = t - NH + j;
            if (src >= bos) {
                lds_vec<XB>(tile, (size_t)(src - (t0 - NH)) * kCh + ch, win[j]);
            } else if (p.s0) {
                ld_state(p.s0, ((size_t)n * NH + (NH - (bos - src))) * D + c0, win[j]);
            } else {
#pragma unroll
                for (int e = 0; e < kVec; ++e) win[j][e] = 0.f;
            }
        }
    };
    start_window(ta);
    const uint8_t *xs = tile + ((size_t)(ta - (t0 - NH)) * kCh + ch) * ES;
    uint8_t *yp = reinterpret_cast<uint8_t *>(p.y) + ((size_t)ta * D + c0) * YS;
    const size_t ystride = D * YS;
    if (tb - ta == kTokPer && eos >= tb) {
        // fast path: all kTokPer tokens in one sequence; unrolled, the window slides by renaming
        float xw[kTokPer + NH][kVec];
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int e = 0; e < kVec; ++e) xw[j][e] = win[j][e];
#pragma unroll
        for (int k = 0; k < kTokPer; ++k) lds_vec<XB>(xs + (size_t)k * kCh * ES, 0, xw[NH + k]);
#pragma unroll
        for (int k = 0; k < kTokPer; ++k) {
            float z[kVec];
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
                float a = fmaf(wv[W - 1][e], xw[NH + k][e], bv[e]);
#pragma unroll
                for (int j = 0; j < NH; ++j) a = fmaf(wv[j][e], xw[k + j][e], a);
                z[e] = ACT ? __fdividef(a, 1.f + __expf(-a)) : a;
            }
            st_vec<YB>(yp + (size_t)k * ystride, 0, z);
        }
        if (eos == tb && p.sT) {
#pragma unroll
            for (int j = 0; j < NH; ++j) st_state(p.sT, ((size_t)n * NH + j) * D + c0, xw[kTokPer + j]);
        }
        return;
    }
    int left = (int)(eos - ta < kTile + 1 ? eos - ta : kTile + 1);  // tokens until the sequence ends
    const int cnt = (int)(tb - ta);
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
        if (left == 0) {  // a sequence starts inside the tile
            const int64_t t = ta + k;
            seq_of(p, t, n, bos, eos);
            start_window(t);
            left = (int)(eos - t < kTile + 1 ? eos - t : kTile + 1);
        }
        float xv[kVec], z[kVec];
        lds_vec<XB>(xs, 0, xv);
        xs += kCh * ES;
        conv_point<W, ACT>(wv, bv, win, xv, z);
        st_vec<YB>(yp, 0, z);
        yp += ystride;
#pragma unroll
        for (int j = 0; j + 1 < NH; ++j)
#pragma unroll
            for (int e = 0; e < kVec; ++e) win[j][e] = win[j + 1][e];
#pragma unroll
        for (int e = 0; e < kVec; ++e) win[NH - 1][e] = xv[e];
        if (--left == 0 && p.sT) {
#pragma unroll
            for (int j = 0; j < NH; ++j) st_state(p.sT, ((size_t)n * NH + j) * D + c0, win[j]);
        }
    }
}

template <int W, bool XB, bool YB>
__global__ void __launch_bounds__(kThreads) short_conv_tile_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                   const ConvParams p, int n_cb, int64_t n_tiles) {
    constexpr int NH = W - 1;  // inputs carried between tokens
    constexpr int ES = XB ? 2 : 4;
    constexpr uint32_t kBuf = (kTile + NH) * kCh * ES;  // one staged tile
    extern __shared__ __align__(128) uint8_t smem[];      // two tiles: (kTile + NH) rows x kCh channels each
    __shared__ __align__(8) uint64_t bar[2];
    const int tid = threadIdx.x;
    const int g = tid & 63, qt = tid >> 6;
    const int ch = g * kVec;  // channel offset inside the tile
    const size_t D = (size_t)p.D;

    // empty sequences hand their state through
    if (p.sT && (p.cu || p.T == 0) && qt == 0) {
        for (int cb = blockIdx.x; cb < n_cb; cb += gridDim.x) {
            const int c0 = cb * kCh + ch;
            if (c0 >= p.D) continue;
            for (int n = 0; n < p.N; ++n) {
                const int64_t len = p.cu ? clamp_row(p.cu[n + 1], p.rows) - clamp_row(p.cu[n], p.rows) : 0;
                if (len > 0) continue;
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    float v[kVec];
                    if (p.s0)
                        ld_state(p.s0, ((size_t)n * NH + j) * D + c0, v);
                    else
#pragma unroll
                        for (int e = 0; e < kVec; ++e) v[e] = 0.f;
                    st_state(p.sT, ((size_t)n * NH + j) * D + c0, v);
                }
            }
        }
    }
    if (p.rows == 0) return;

    // tile id -> (channel block, token tile); consecutive ids share a token tile.
    // Thread 0 counts, per buffer, the copies issued and the completions seen.
    int n_issued[2] = {0, 0}, n_seen[2] = {0, 0};
    auto issue = [&](int64_t id, int b) {
        ++n_issued[b];
        const int cb = (int)(id % n_cb);
        const int64_t t0 = (id / n_cb) * kTile;
        tc::mbar_arrive_expect_tx(&bar[b], kBuf);
        tc::tma_load_2d(tc::smem_u32(smem + b * kBuf), &tmx, &bar[b], cb * kCh, (int)(t0 - NH));
    };
    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        tc::fence_mbar_init();
        if ((int64_t)blockIdx.x < n_tiles) issue(blockIdx.x, 0);
        if ((int64_t)blockIdx.x + gridDim.x < n_tiles) issue(blockIdx.x + gridDim.x, 1);
    }
    __syncthreads();  // the barriers are initialised before anyone polls them

    int it = 0;
    bool ok = true;
    int64_t first_bad = n_tiles;
    for (int64_t id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
        const int b = it & 1;
        const uint8_t *tile = smem + b * kBuf;
        const int cb = (int)(id % n_cb);
        const int64_t t0 = (id / n_cb) * kTile;
        const int c0 = cb * kCh + ch;
        const bool tile_ok = tc::mbar_wait(&bar[b], (uint32_t)((it >> 1) & 1), p.polls);
        if (tile_ok) ++n_seen[b];
        const int64_t ta = t0 + qt * kTokPer;  // this thread's tokens [ta, tb)
        const int64_t t1 = t0 + kTile < p.rows ? t0 + kTile : p.rows;
        const int64_t tb = ta + kTokPer < t1 ? ta + kTokPer : t1;
        if (tile_ok && c0 < p.D && ta < tb) {
            if (p.act)
                conv_tokens<W, XB, YB, true>(p, tile, t0, ta, tb, ch, c0);
            else
                conv_tokens<W, XB, YB, false>(p, tile, t0, ta, tb, ch, c0);
        }
        ok = __syncthreads_and(tile_ok);  // every thread is done with buffer b; a timeout anywhere stops the CTA
        if (!ok) {
            first_bad = id;  // this whole tile is poisoned below, with the rest
            break;
        }
        if (tid == 0 && id + 2 * (int64_t)gridDim.x < n_tiles) issue(id + 2 * (int64_t)gridDim.x, b);
    }
    if (ok) return;
    // A tile did not arrive in time: the copies still in flight get their full bounded time
    // to land, then every tile this CTA still owned gets NaN outputs, and so does the state
    // of each sequence whose last token lies in one of them.
    if (tid == 0) {
        atomicAdd(&g_short_conv_timeouts, 1);
        for (int b = 0; b < 2; ++b)
            if (n_issued[b] > n_seen[b]) tc::mbar_wait(&bar[b], (uint32_t)(n_seen[b] & 1), kPolls);
    }
    __syncthreads();
    const float nan = __int_as_float(0x7fc00000);
    const float nan4[kVec] = {nan, nan, nan, nan};
    for (int64_t id = first_bad; id < n_tiles; id += gridDim.x) {
        const int c0 = (int)(id % n_cb) * kCh + ch;
        const int64_t ta = (id / n_cb) * kTile + qt * kTokPer;
        const int64_t t1 = (id / n_cb) * kTile + kTile < p.rows ? (id / n_cb) * kTile + kTile : p.rows;
        const int64_t tb = ta + kTokPer < t1 ? ta + kTokPer : t1;
        if (c0 >= p.D) continue;
        for (int64_t t = ta; t < tb; ++t) {
            st_vec<YB>(p.y, (size_t)t * D + c0, nan4);
            int n;
            int64_t bos, eos;
            seq_of(p, t, n, bos, eos);
            if (p.sT && eos == t + 1)
                for (int j = 0; j < NH; ++j) st_state(p.sT, ((size_t)n * NH + j) * D + c0, nan4);
        }
    }
}

// One token per sequence (dense, T = 1): thread per (sequence, 4 channels).
template <int W, bool XB, bool YB>
__global__ void __launch_bounds__(256) short_conv_step_kernel(const ConvParams p) {
    constexpr int NH = W - 1;
    const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int groups = p.D / kVec;
    const int64_t n = idx / groups;
    if (n >= p.rows) return;
    const int c0 = (int)(idx % groups) * kVec;
    const size_t D = (size_t)p.D;
    float win[NH][kVec], xv[kVec], wv[W][kVec], bv[kVec], z[kVec];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        if (p.s0)
            ld_state(p.s0, ((size_t)n * NH + j) * D + c0, win[j]);
        else
#pragma unroll
            for (int e = 0; e < kVec; ++e) win[j][e] = 0.f;
    }
    ld_vec<XB>(p.x, (size_t)n * D + c0, xv);
    load_filter<W>(p, c0, wv, bv);
    if (p.act)
        conv_point<W, true>(wv, bv, win, xv, z);
    else
        conv_point<W, false>(wv, bv, win, xv, z);
    st_vec<YB>(p.y, (size_t)n * D + c0, z);
    if (p.sT) {
#pragma unroll
        for (int j = 0; j + 1 < NH; ++j) st_state(p.sT, ((size_t)n * NH + j) * D + c0, win[j + 1]);
        st_state(p.sT, ((size_t)n * NH + NH - 1) * D + c0, xv);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int W, bool XB, bool YB>
kda_status launch_wxy(const ConvParams &p, cudaStream_t st) {
    constexpr int NH = W - 1;
    if (!p.cu && p.T == 1) {  // decode step
        const int64_t threads = p.rows * (p.D / kVec);
        short_conv_step_kernel<W, XB, YB><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(p);
        note_launch();
        return check_launch("short_conv_step_kernel");
    }
    const int64_t tiles = (p.rows + kTile - 1) / kTile;
    CUtensorMap tmap;
    memset(&tmap, 0, sizeof(tmap));
    if (p.rows > 0) {
        EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
        if (!enc) {
            set_error("short_conv: cuTensorMapEncodeTiled is not available from the driver");
            return KDA_ERR_CUDA;
        }
        const cuuint64_t dims[2] = {(cuuint64_t)p.D, (cuuint64_t)p.rows};
        const cuuint64_t strides[1] = {(cuuint64_t)p.D * (XB ? 2 : 4)};
        const cuuint32_t box[2] = {(cuuint32_t)kCh, (cuuint32_t)(kTile + NH)};
        const cuuint32_t estr[2] = {1, 1};
        const CUresult r = enc(&tmap, XB ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                               const_cast<void *>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            set_error("short_conv: cuTensorMapEncodeTiled failed (%d)", (int)r);
            return KDA_ERR_CUDA;
        }
    }
    const int smem = 2 * (kTile + NH) * kCh * (XB ? 2 : 4);
    static DeviceOnce configured;
    const int dev = current_device();
    if (!configured.done(dev)) {
        const cudaError_t e = cudaFuncSetAttribute(short_conv_tile_kernel<W, XB, YB>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            set_error("short_conv: cannot reserve %d bytes of shared memory: %s", smem, cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
        configured.set(dev);
    }
    const int n_cb = (p.D + kCh - 1) / kCh;
    const int64_t n_tiles = tiles * n_cb;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, short_conv_tile_kernel<W, XB, YB>, kThreads, smem);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int64_t grid = n_tiles < cap ? (n_tiles > 0 ? n_tiles : 1) : cap;
    short_conv_tile_kernel<W, XB, YB><<<(unsigned)grid, kThreads, smem, st>>>(tmap, p, n_cb, n_tiles);
    note_launch();
    return check_launch("short_conv_tile_kernel");
}

template <int W>
kda_status launch_w(const ConvParams &p, bool xb, bool yb, cudaStream_t st) {
    if (xb && yb) return launch_wxy<W, true, true>(p, st);
    if (xb) return launch_wxy<W, true, false>(p, st);
    if (yb) return launch_wxy<W, false, true>(p, st);
    return launch_wxy<W, false, false>(p, st);
}

}  // namespace

int take_short_conv_timeouts(cudaStream_t st) {
    int n = 0;
    const int zero = 0;
    if (cudaMemcpyFromSymbolAsync(&n, g_short_conv_timeouts, sizeof(int), 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_short_conv_timeouts, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        set_error("short_conv: cannot read the timeout counter: %s", cudaGetErrorString(cudaGetLastError()));
        return -1;
    }
    return n;
}

kda_status launch_short_conv(const void *x, int x_bf16, const float *w, const float *bias, const float *s0,
                             float *sT, void *y, int y_bf16, const int32_t *cu, int N, int64_t rows, int T,
                             int D, int W, int act, cudaStream_t st) {
    ConvParams p;
    p.x = x;
    p.y = y;
    p.w = w;
    p.bias = bias;
    p.s0 = s0;
    p.sT = sT;
    p.cu = cu;
    p.rows = rows;
    p.N = N;
    p.T = T;
    p.D = D;
    p.act = act;
    p.polls = wait_polls();
    if (rows == 0 && (!sT || N == 0)) return KDA_OK;
    switch (W) {
        case 2: return launch_w<2>(p, x_bf16, y_bf16, st);
        case 3: return launch_w<3>(p, x_bf16, y_bf16, st);
        case 4: return launch_w<4>(p, x_bf16, y_bf16, st);
        default: break;
    }
    set_error("short_conv: W=%d not built (W in {2, 3, 4})", W);
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
