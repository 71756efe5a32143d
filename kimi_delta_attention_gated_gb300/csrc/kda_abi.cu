// kda_abi.cu -- the extern "C" boundary of libkda: argument validation, path
// selection and launch bookkeeping.  Declarations and their documentation are
// in include/kda.h.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kda_internal.cuh"

namespace kda {

namespace {
thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};
std::atomic<uint32_t> g_wait_polls{kDefaultWaitPolls};
constexpr int kVersion = 10100;  // 1.1.0
}  // namespace

uint32_t wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return dev;
}

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

kda_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: %s", what, cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace kda

using kda::set_error;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool dtype_ok(int d) { return d == KDA_BF16 || d == KDA_F32; }

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

#define KDA_REQUIRE(cond, code, ...) \
    do {                             \
        if (!(cond)) {               \
            set_error(__VA_ARGS__);  \
            return code;             \
        }                            \
    } while (0)

// A byte range of one argument, for the overlap checks.
struct Span {
    const void *p;
    size_t bytes;
    const char *name;
};

bool overlaps(const Span &a, const Span &b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const char *x = static_cast<const char *>(a.p), *y = static_cast<const char *>(b.p);
    return x < y + b.bytes && y < x + a.bytes;
}

// The kernels read their inputs chunk by chunk while they write their outputs, so no
// output may share bytes with an input or with another output.  The one exception is
// the state: final_state may be initial_state itself (the same pointer), never a
// partial overlap.  Returns the first offending pair in the error message.
kda_status check_overlaps(const char *fn, const Span *in, int n_in, const Span *out, int n_out, const Span &s0,
                          const Span &sT) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            KDA_REQUIRE(!overlaps(out[i], in[j]), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn, out[i].name,
                        in[j].name);
        for (int j = i + 1; j < n_out; ++j)
            KDA_REQUIRE(!overlaps(out[i], out[j]), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn,
                        out[i].name, out[j].name);
        KDA_REQUIRE(!overlaps(out[i], s0) && !overlaps(out[i], sT), KDA_ERR_INVALID_ARG,
                    "%s: %s must not overlap the state", fn, out[i].name);
    }
    for (int j = 0; j < n_in; ++j)
        KDA_REQUIRE(!overlaps(sT, in[j]), KDA_ERR_INVALID_ARG, "%s: the final state must not overlap %s", fn,
                    in[j].name);
    KDA_REQUIRE(!overlaps(s0, sT) || s0.p == sT.p, KDA_ERR_INVALID_ARG,
                "%s: final_state may be initial_state itself but must not partly overlap it", fn);
    return KDA_OK;
}

size_t esize(int dtype) { return dtype == KDA_BF16 ? 2 : 4; }

// Overlap check of one prefill / decode call: rows tokens, N sequences.
kda_status check_call_overlaps(const char *fn, const void *q, const void *k, const void *v, int qkv_dtype,
                               const void *g, size_t g_esz, const void *beta, size_t b_esz, const float *s0,
                               const float *sT, const void *o, int o_dtype, const float *states, const void *gate,
                               int gate_dtype, const float *norm_w, const void *y, int64_t rows, int N, int H, int K,
                               int V) {
    const size_t r = (size_t)rows, hk = (size_t)H * K, hv = (size_t)H * V, st = (size_t)N * H * K * V * 4;
    const Span in[] = {{q, r * hk * esize(qkv_dtype), "q"}, {k, r * hk * esize(qkv_dtype), "k"},
                       {v, r * hv * esize(qkv_dtype), "v"}, {g, r * hk * g_esz, "g"},
                       {beta, r * H * b_esz, "beta"},      {gate, gate ? r * hv * esize(gate_dtype) : 0, "gate"},
                       {norm_w, norm_w ? (size_t)V * 4 : 0, "norm_w"}};
    const Span out[] = {{o, r * hv * esize(o_dtype), "o"},
                        {y, y ? r * hv * esize(o_dtype) : 0, "y"},
                        {states, states ? r * hk * V * 4 : 0, "states"}};
    return check_overlaps(fn, in, 7, out, 3, Span{s0, s0 ? st : 0, "initial_state"},
                          Span{sT, sT ? st : 0, "final_state"});
}


// Checks shared by the prefill entry points; fills the sequence count.
kda_status check_seq_args(const char *fn, const void *q, const void *k, const void *v, int qkv_dtype,
                          const float *g, const float *beta, const float *s0, const float *sT,
                          const void *o, int o_dtype, const int32_t *cu, const int32_t *cu_host,
                          int n_seqs, int B, int T, int H, int K, int V, float scale,
                          const void *gate, int gate_dtype, const float *norm_w, float eps,
                          const void *y, int &N) {
    // with no tokens nothing is read or written but the state (empty tensors may be NULL)
    const bool no_tokens = (int64_t)B * T == 0;
    KDA_REQUIRE(no_tokens || (q && k && v && g && beta), KDA_ERR_INVALID_ARG,
                "%s: q, k, v, g and beta must not be NULL", fn);
    KDA_REQUIRE(no_tokens || o || (gate && y), KDA_ERR_INVALID_ARG,
                "%s: o may be NULL only when the gated norm writes y", fn);
    KDA_REQUIRE(dtype_ok(qkv_dtype) && dtype_ok(o_dtype) && (!gate || dtype_ok(gate_dtype)),
                KDA_ERR_UNSUPPORTED, "%s: unsupported dtype", fn);
    KDA_REQUIRE(H > 0 && T >= 0 && B > 0, KDA_ERR_INVALID_ARG, "%s: need B > 0, T >= 0, H > 0", fn);
    KDA_REQUIRE(dim_ok(K) && dim_ok(V), KDA_ERR_UNSUPPORTED, "%s: K=%d V=%d (supported: 32, 64, 128)", fn, K, V);
    KDA_REQUIRE(std::isfinite(scale), KDA_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    KDA_REQUIRE((int64_t)B * T <= (int64_t)INT32_MAX, KDA_ERR_INVALID_ARG, "%s: B*T too large", fn);
    const void *ptrs[] = {q, k, v, g, beta, s0, sT, o, cu, gate, norm_w, y};
    for (const void *ptr : ptrs)
        KDA_REQUIRE(!ptr || aligned16(ptr), KDA_ERR_INVALID_ARG, "%s: every pointer must be 16-byte aligned", fn);
    if (gate) {
        KDA_REQUIRE(norm_w && (y || no_tokens), KDA_ERR_INVALID_ARG, "%s: the gated norm needs norm_w and y", fn);
        KDA_REQUIRE(eps > 0.f && std::isfinite(eps), KDA_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    }
    if (cu) {
        KDA_REQUIRE(B == 1, KDA_ERR_INVALID_ARG, "%s: varlen (cu_seqlens) needs B == 1", fn);
        KDA_REQUIRE(n_seqs > 0, KDA_ERR_INVALID_ARG, "%s: varlen needs n_seqs > 0", fn);
        if (cu_host) {
            KDA_REQUIRE(cu_host[0] == 0, KDA_ERR_INVALID_ARG, "%s: cu_seqlens[0] must be 0", fn);
            for (int i = 0; i < n_seqs; ++i)
                KDA_REQUIRE(cu_host[i + 1] >= cu_host[i], KDA_ERR_INVALID_ARG,
                            "%s: cu_seqlens must not decrease (entry %d)", fn, i + 1);
            KDA_REQUIRE(cu_host[n_seqs] == T, KDA_ERR_INVALID_ARG, "%s: cu_seqlens[n_seqs] = %d but T = %d", fn,
                        cu_host[n_seqs], T);
        }
        N = n_seqs;
    } else {
        KDA_REQUIRE(!cu_host, KDA_ERR_INVALID_ARG, "%s: cu_seqlens_host given without cu_seqlens", fn);
        N = B;
    }
    return KDA_OK;
}

kda::SeqParams make_params(const void *q, const void *k, const void *v, int qkv_dtype, const float *g,
                           const float *beta, const float *s0, float *sT, void *o, int o_dtype,
                           float *states, const int32_t *cu, int N, int T, int H, float scale,
                           int l2, const void *gate, int gate_dtype, const float *norm_w, float eps,
                           void *y) {
    kda::SeqParams p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.g = g;
    p.beta = beta;
    p.s0 = s0;
    p.sT = sT;
    p.o = o;
    p.states = states;
    p.cu_seqlens = cu;
    p.cu_host = nullptr;
    p.K = 0;
    p.g_logits = nullptr;
    p.A_log = nullptr;
    p.dt_bias = nullptr;
    p.beta_logits = nullptr;
    p.g_lower = -INFINITY;
    p.g_logits_bf16 = p.beta_logits_bf16 = 0;
    p.gate = gate;
    p.norm_w = norm_w;
    p.y = y;
    p.N = N;
    p.T = T;
    p.H = H;
    p.scale = scale;
    p.eps = eps;
    p.l2norm = l2 ? 1 : 0;
    p.qkv_bf16 = qkv_dtype == KDA_BF16;
    p.o_bf16 = o_dtype == KDA_BF16;
    p.gate_bf16 = gate_dtype == KDA_BF16;
    p.polls = kda::wait_polls();
    for (int f = 0; f < 3; ++f) {
        p.cw[f] = p.cs_in[f] = nullptr;
        p.cs_out[f] = nullptr;
    }
    p.conv_w = 0;
    return p;
}

using kda::GateLogits;

kda_status check_logits(const char *fn, const GateLogits &gl, bool no_tokens) {
    KDA_REQUIRE(gl.A_log, KDA_ERR_INVALID_ARG, "%s: A_log must not be NULL", fn);
    KDA_REQUIRE(no_tokens || (gl.z && gl.b), KDA_ERR_INVALID_ARG, "%s: g_logits and beta_logits must not be NULL", fn);
    KDA_REQUIRE(dtype_ok(gl.z_dtype) && dtype_ok(gl.b_dtype), KDA_ERR_UNSUPPORTED, "%s: unsupported logits dtype", fn);
    KDA_REQUIRE(!std::isnan(gl.lower) && gl.lower <= 0.f, KDA_ERR_INVALID_ARG,
                "%s: g_lower_bound must be <= 0 (-INFINITY for none)", fn);
    const void *ptrs[] = {gl.z, gl.A_log, gl.dt_bias, gl.b};
    for (const void *ptr : ptrs)
        KDA_REQUIRE(!ptr || aligned16(ptr), KDA_ERR_INVALID_ARG, "%s: every pointer must be 16-byte aligned", fn);
    return KDA_OK;
}

void set_logits(kda::SeqParams &p, const GateLogits *gl, int K) {
    p.K = K;
    p.g_logits = gl ? gl->z : nullptr;
    p.A_log = gl ? gl->A_log : nullptr;
    p.dt_bias = gl ? gl->dt_bias : nullptr;
    p.beta_logits = gl ? gl->b : nullptr;
    p.g_lower = gl ? gl->lower : -INFINITY;
    p.g_logits_bf16 = gl && gl->z_dtype == KDA_BF16;
    p.beta_logits_bf16 = gl && gl->b_dtype == KDA_BF16;
}

kda_status chunk_impl(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                      const float *g, const float *beta, const GateLogits *gl, const float *initial_state,
                      float *final_state, void *o, kda_dtype o_dtype, const int32_t *cu_seqlens,
                      const int32_t *cu_seqlens_host, int n_seqs, int B, int T, int H, int K, int V, int chunk,
                      float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                      const float *norm_w, float eps, void *y, void *workspace, size_t workspace_bytes, int mode,
                      void *stream) {
    kda::g_err[0] = 0;
    int N = 0;
    // with logits, g / beta are checked through them (the recurrence never reads g / beta then)
    const float *gchk = gl ? reinterpret_cast<const float *>(gl->z) : g;
    const float *bchk = gl ? reinterpret_cast<const float *>(gl->b) : beta;
    kda_status s = check_seq_args(fn, q, k, v, qkv_dtype, gchk, bchk, initial_state, final_state, o, o_dtype,
                                  cu_seqlens, cu_seqlens_host, n_seqs, B, T, H, K, V, scale, gate, gate_dtype,
                                  norm_w, eps, y, N);
    if (s != KDA_OK) return s;
    if (gl && (s = check_logits(fn, *gl, (int64_t)B * T == 0)) != KDA_OK) return s;
    s = check_call_overlaps(fn, q, k, v, qkv_dtype, gchk, gl ? esize(gl->z_dtype) : 4, bchk,
                            gl ? esize(gl->b_dtype) : 4, initial_state, final_state, o, o_dtype, nullptr, gate,
                            gate_dtype, norm_w, y, (int64_t)B * T, N, H, K, V);
    if (s != KDA_OK) return s;
    KDA_REQUIRE(chunk == 16 || chunk == 32 || chunk == 64, KDA_ERR_UNSUPPORTED, "%s: chunk=%d (supported: 16, 32, 64)",
                fn, chunk);
    KDA_REQUIRE(mode == KDA_MODE_AUTO || mode == KDA_MODE_TENSOR || mode == KDA_MODE_FP32 || mode == KDA_MODE_SPLIT,
                KDA_ERR_INVALID_ARG, "%s: unknown mode %d", fn, mode);
    const bool tc_ok = kda::chunk_tc_supported(K, V, chunk) && qkv_dtype == KDA_BF16;
    KDA_REQUIRE((mode != KDA_MODE_TENSOR && mode != KDA_MODE_SPLIT) || tc_ok, KDA_ERR_UNSUPPORTED,
                "%s: the tensor path needs bf16 q/k/v, K = V = 128 and chunk = 64", fn);
    KDA_REQUIRE(mode != KDA_MODE_SPLIT || workspace, KDA_ERR_INVALID_ARG,
                "%s: the split form needs a workspace (kda_chunk_workspace_size)", fn);
    cudaStream_t st = (cudaStream_t)stream;
    // an empty prompt only hands the state through: the fp32 path does that without a tensor map
    const bool use_tc = tc_ok && mode != KDA_MODE_FP32 && T > 0;
    KDA_REQUIRE(!workspace || aligned16(workspace), KDA_ERR_INVALID_ARG, "%s: the workspace must be 16-byte aligned",
                fn);
    if (use_tc) {
        kda::SeqParams p = make_params(q, k, v, qkv_dtype, g, beta, initial_state, final_state, o, o_dtype, nullptr,
                                       cu_seqlens, N, T, H, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y);
        p.cu_host = cu_seqlens_host;
        set_logits(p, gl, K);
        if (!workspace) return kda::launch_chunk_tc(p, K, V, chunk, st);
        const int64_t rows = (int64_t)B * T;
        const size_t need = kda::chunk_workspace_bytes(rows, N, H);
        KDA_REQUIRE(workspace_bytes >= need, KDA_ERR_INVALID_ARG,
                    "%s: the workspace holds %zu bytes, this call needs %zu (kda_chunk_workspace_size)", fn,
                    workspace_bytes, need);
        {  // the workspace is written while every tensor of the call is in use
            const size_t r = (size_t)rows, qkv = esize(qkv_dtype), st_bytes = (size_t)N * H * K * V * 4;
            const Span ws{workspace, need, "the workspace"};
            const Span all[] = {{q, r * H * K * qkv, "q"}, {k, r * H * K * qkv, "k"}, {v, r * H * V * qkv, "v"},
                                {gchk, r * H * K * (gl ? esize(gl->z_dtype) : 4), "g"},
                                {bchk, r * H * (gl ? esize(gl->b_dtype) : 4), "beta"},
                                {o, o ? r * H * V * esize(o_dtype) : 0, "o"},
                                {y, y ? r * H * V * esize(o_dtype) : 0, "y"},
                                {gate, gate ? r * H * V * esize(gate_dtype) : 0, "gate"},
                                {initial_state, initial_state ? st_bytes : 0, "initial_state"},
                                {final_state, final_state ? st_bytes : 0, "final_state"}};
            for (const Span &x : all)
                KDA_REQUIRE(!overlaps(ws, x), KDA_ERR_INVALID_ARG, "%s: the workspace must not overlap %s", fn, x.name);
        }
        if (mode != KDA_MODE_SPLIT) return kda::launch_chunk_concurrent(p, workspace, st);
        s = kda::launch_chunk_prep(p, workspace, st);
        if (s != KDA_OK) return s;
        return kda::launch_chunk_chain(p, workspace, st);
    }
    // fp32 path: o goes to y's buffer when o is not wanted, then the norm runs in place.
    void *o_target = o ? o : y;
    kda::SeqParams p = make_params(q, k, v, qkv_dtype, g, beta, initial_state, final_state, o_target, o_dtype,
                                   nullptr, cu_seqlens, N, T, H, scale, use_qk_l2norm, nullptr, gate_dtype, norm_w,
                                   eps, nullptr);
    set_logits(p, gl, K);
    s = kda::launch_chunk_fp32(p, K, V, chunk, nullptr, st);
    if (s != KDA_OK || !gate || (int64_t)B * T == 0) return s;
    return kda::launch_gated_rmsnorm(o_target, o_dtype == KDA_BF16, gate, gate_dtype == KDA_BF16, norm_w, eps, y,
                                     o_dtype == KDA_BF16, (int64_t)B * T, H, V, st);
}

// The fused short convolutions of kda_recurrent_step_conv.
struct ConvArgs {
    const float *const *w;       // [3]
    int W;
    const float *const *s_in;    // [3] or null
    float *const *s_out;         // [3]
};

// Arguments of the fused convolutions: shapes, alignment, and that no new history
// overlaps anything but its own old history (then exactly), and no weight or old history
// overlaps an output of the step.
kda_status check_conv(const char *fn, const ConvArgs &cv, int B, int H, int K, int V, const Span *step_in, int n_in,
                      const Span *step_out, int n_out) {
    KDA_REQUIRE(K == 128 && V == 128, KDA_ERR_UNSUPPORTED,
                "%s: the fused short convolutions are built for K = V = 128 (got K=%d V=%d)", fn, K, V);
    KDA_REQUIRE(cv.W >= 2 && cv.W <= 4, KDA_ERR_UNSUPPORTED, "%s: W=%d (supported: 2, 3, 4)", fn, cv.W);
    KDA_REQUIRE(cv.w && cv.s_out, KDA_ERR_INVALID_ARG, "%s: conv_weight and conv_state_out must not be NULL", fn);
    const bool hist = cv.s_in && cv.s_in[0];
    for (int f = 0; f < 3; ++f) {
        KDA_REQUIRE(cv.w[f] && cv.s_out[f], KDA_ERR_INVALID_ARG,
                    "%s: all three conv_weight and conv_state_out pointers are needed", fn);
        KDA_REQUIRE(!cv.s_in || (cv.s_in[f] != nullptr) == hist, KDA_ERR_INVALID_ARG,
                    "%s: conv_state_in gives all three histories or none", fn);
        KDA_REQUIRE(aligned16(cv.w[f]) && aligned16(cv.s_out[f]) && (!hist || aligned16(cv.s_in[f])),
                    KDA_ERR_INVALID_ARG, "%s: every pointer must be 16-byte aligned", fn);
    }
    const size_t D = (size_t)H * 128, wb = D * cv.W * 4, sb = (size_t)B * (cv.W - 1) * D * 4;
    const char *names_w[3] = {"conv_weight[0]", "conv_weight[1]", "conv_weight[2]"};
    const char *names_i[3] = {"conv_state_in[0]", "conv_state_in[1]", "conv_state_in[2]"};
    const char *names_o[3] = {"conv_state_out[0]", "conv_state_out[1]", "conv_state_out[2]"};
    for (int f = 0; f < 3; ++f) {
        const Span so{cv.s_out[f], sb, names_o[f]};
        for (int j = 0; j < n_in; ++j)
            KDA_REQUIRE(!overlaps(so, step_in[j]), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn, so.name,
                        step_in[j].name);
        for (int j = 0; j < n_out; ++j)
            KDA_REQUIRE(!overlaps(so, step_out[j]), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn, so.name,
                        step_out[j].name);
        for (int e = 0; e < 3; ++e) {
            const Span we{cv.w[e], wb, names_w[e]};
            KDA_REQUIRE(!overlaps(so, we), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn, so.name, we.name);
            if (hist) {
                const Span si{cv.s_in[e], sb, names_i[e]};
                KDA_REQUIRE(!overlaps(so, si) || (e == f && si.p == so.p), KDA_ERR_INVALID_ARG,
                            "%s: %s may be %s itself but must not overlap any other history", fn, so.name,
                            names_i[f]);
            }
            if (e > f) {
                const Span so2{cv.s_out[e], sb, names_o[e]};
                KDA_REQUIRE(!overlaps(so, so2), KDA_ERR_INVALID_ARG, "%s: %s must not overlap %s", fn, so.name,
                            so2.name);
            }
        }
        // the weights and old histories are inputs: no output of the step may overlap them
        const Span we{cv.w[f], wb, names_w[f]}, si{hist ? cv.s_in[f] : nullptr, sb, names_i[f]};
        for (int j = 0; j < n_out; ++j)
            KDA_REQUIRE(!overlaps(we, step_out[j]) && !overlaps(si, step_out[j]), KDA_ERR_INVALID_ARG,
                        "%s: %s must not overlap %s or %s", fn, step_out[j].name, we.name, si.name);
    }
    return KDA_OK;
}

kda_status step_impl(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                     const float *g, const float *beta, const GateLogits *gl, const float *state_in,
                     float *state_out, void *o, kda_dtype o_dtype, int B, int H, int K, int V, float scale,
                     int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w, float eps,
                     void *y, void *stream, const ConvArgs *cv = nullptr) {
    kda::g_err[0] = 0;
    int N = 0;
    KDA_REQUIRE(state_out, KDA_ERR_INVALID_ARG, "%s: state_out must not be NULL", fn);
    const float *gchk = gl ? reinterpret_cast<const float *>(gl->z) : g;
    const float *bchk = gl ? reinterpret_cast<const float *>(gl->b) : beta;
    kda_status s = check_seq_args(fn, q, k, v, qkv_dtype, gchk, bchk, state_in, state_out, o, o_dtype, nullptr,
                                  nullptr, 0, B, 1, H, K, V, scale, gate, gate_dtype, norm_w, eps, y, N);
    if (s != KDA_OK) return s;
    if (gl && (s = check_logits(fn, *gl, false)) != KDA_OK) return s;
    s = check_call_overlaps(fn, q, k, v, qkv_dtype, gchk, gl ? esize(gl->z_dtype) : 4, bchk,
                            gl ? esize(gl->b_dtype) : 4, state_in, state_out, o, o_dtype, nullptr, gate, gate_dtype,
                            norm_w, y, B, N, H, K, V);
    if (s != KDA_OK) return s;
    if (cv) {
        const size_t hk = (size_t)B * H * K, hv = (size_t)B * H * V, st = (size_t)B * H * K * V * 4;
        const Span in[] = {{q, hk * esize(qkv_dtype), "q"},
                           {k, hk * esize(qkv_dtype), "k"},
                           {v, hv * esize(qkv_dtype), "v"},
                           {gchk, hk * (gl ? esize(gl->z_dtype) : 4), gl ? "g_logits" : "g"},
                           {bchk, (size_t)B * H * (gl ? esize(gl->b_dtype) : 4), gl ? "beta_logits" : "beta"},
                           {gate, gate ? hv * esize(gate_dtype) : 0, "gate"},
                           {norm_w, norm_w ? (size_t)V * 4 : 0, "norm_w"},
                           {state_in, state_in ? st : 0, "state_in"}};
        const Span out[] = {{o, o ? hv * esize(o_dtype) : 0, "o"},
                            {y, y ? hv * esize(o_dtype) : 0, "y"},
                            {state_out, st, "state_out"}};
        if ((s = check_conv(fn, *cv, B, H, K, V, in, 8, out, 3)) != KDA_OK) return s;
    }
    kda::SeqParams p = make_params(q, k, v, qkv_dtype, g, beta, state_in, state_out, o, o_dtype, nullptr, nullptr, N,
                                   1, H, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y);
    set_logits(p, gl, K);
    if (cv) {
        const bool hist = cv->s_in && cv->s_in[0];
        for (int f = 0; f < 3; ++f) {
            p.cw[f] = cv->w[f];
            p.cs_in[f] = hist ? cv->s_in[f] : nullptr;
            p.cs_out[f] = cv->s_out[f];
        }
        p.conv_w = cv->W;
    }
    return kda::launch_recurrent(p, K, V, (cudaStream_t)stream);
}

}  // namespace

namespace kda {

kda_status chunk_fwd_entry(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                           const float *g, const float *beta, const float *initial_state, float *final_state, void *o,
                           kda_dtype o_dtype, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                           int B, int T, int H, int K, int V, int chunk, float scale, int use_qk_l2norm,
                           const void *gate, kda_dtype gate_dtype, const float *norm_w, float eps, void *y,
                           void *workspace, size_t workspace_bytes, int mode, void *stream) {
    return chunk_impl(fn, q, k, v, qkv_dtype, g, beta, nullptr, initial_state, final_state, o, o_dtype, cu_seqlens,
                      cu_seqlens_host, n_seqs, B, T, H, K, V, chunk, scale, use_qk_l2norm, gate, gate_dtype, norm_w,
                      eps, y, workspace, workspace_bytes, mode, stream);
}

kda_status chunk_call(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                      const float *g, const float *beta, const GateLogits *gl, const float *initial_state,
                      float *final_state, void *o, kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk,
                      float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w,
                      float eps, void *y, int mode, void *stream) {
    return chunk_impl(fn, q, k, v, qkv_dtype, g, beta, gl, initial_state, final_state, o, o_dtype, nullptr, nullptr,
                      0, B, T, H, K, V, chunk, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, nullptr, 0,
                      mode, stream);
}

}  // namespace kda

extern "C" {

int kda_version(void) { return kda::kVersion; }

const char *kda_last_error(void) { return kda::g_err; }

const char *kda_status_string(int s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        default: return "KDA_ERR_UNKNOWN";
    }
}

uint64_t kda_launch_count(void) { return kda::g_launches.load(std::memory_order_relaxed); }

kda_status kda_device_status(void *stream) {
    kda::g_err[0] = 0;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        set_error("kda_device_status: the stream failed: %s", cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    const int n_tc0 = kda::take_chunk_tc_timeouts(st);
    const int n_prep = kda::take_chunk_prep_timeouts(st);
    const int n_chain = kda::take_chunk_chain_timeouts(st);
    const int n_dec = kda::take_decode_timeouts(st);
    const int n_conv = kda::take_short_conv_timeouts(st);
    const int n_proj = kda::take_oproj_timeouts(st);
    if (n_tc0 < 0 || n_prep < 0 || n_chain < 0 || n_dec < 0 || n_conv < 0 || n_proj < 0) return KDA_ERR_CUDA;
    const int n_tc = n_tc0 + n_prep + n_chain;
    if (n_tc + n_dec + n_conv + n_proj > 0) {
        set_error("kda_device_status: bounded waits gave up in %d prefill, %d decode, %d short-convolution and %d "
                  "output-projection CTAs; their outputs hold NaN",
                  n_tc, n_dec, n_conv, n_proj);
        return KDA_ERR_TIMEOUT;
    }
    return KDA_OK;
}

kda_status kda_chunk_prepass_hits(void *stream, uint64_t *chunks) {
    kda::g_err[0] = 0;
    KDA_REQUIRE(chunks, KDA_ERR_INVALID_ARG, "kda_chunk_prepass_hits: chunks must not be NULL");
    const long long n = kda::take_chunk_blob_chunks((cudaStream_t)stream);
    if (n < 0) return KDA_ERR_CUDA;
    *chunks = (uint64_t)n;
    return KDA_OK;
}

kda_status kda_set_wait_limit(int64_t polls) {
    kda::g_err[0] = 0;
    KDA_REQUIRE(polls <= (int64_t)UINT32_MAX, KDA_ERR_INVALID_ARG, "kda_set_wait_limit: at most %u polls",
                UINT32_MAX);
    kda::g_wait_polls.store(polls < 0 ? kda::kDefaultWaitPolls : (uint32_t)polls, std::memory_order_relaxed);
    return KDA_OK;
}

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                         const float *g, const float *beta, const float *initial_state,
                         float *final_state, void *o, kda_dtype o_dtype,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                         int B, int T, int H, int K, int V, int chunk, float scale,
                         int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                         const float *norm_w, float eps, void *y, void *workspace, size_t workspace_bytes, int mode,
                         void *stream) {
    return chunk_impl("kda_chunk_fwd", q, k, v, qkv_dtype, g, beta, nullptr, initial_state, final_state, o, o_dtype,
                      cu_seqlens, cu_seqlens_host, n_seqs, B, T, H, K, V, chunk, scale, use_qk_l2norm, gate,
                      gate_dtype, norm_w, eps, y, workspace, workspace_bytes, mode, stream);
}

size_t kda_chunk_workspace_size(int B, int T, int H, int n_seqs) {
    if (B <= 0 || T < 0 || H <= 0 || n_seqs < 0) return 0;
    const int N = n_seqs > 0 ? n_seqs : B;
    return kda::chunk_workspace_bytes((int64_t)B * T, N, H);
}

kda_status kda_chunk_fwd_logits(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                kda_dtype beta_logits_dtype, const float *initial_state, float *final_state,
                                void *o, kda_dtype o_dtype, const int32_t *cu_seqlens,
                                const int32_t *cu_seqlens_host, int n_seqs, int B, int T, int H, int K, int V,
                                int chunk, float scale, int use_qk_l2norm, const void *gate,
                                kda_dtype gate_dtype, const float *norm_w, float eps, void *y, void *workspace,
                                size_t workspace_bytes, int mode, void *stream) {
    const GateLogits gl{g_logits, g_logits_dtype, A_log, dt_bias, g_lower_bound, beta_logits, beta_logits_dtype};
    return chunk_impl("kda_chunk_fwd_logits", q, k, v, qkv_dtype, nullptr, nullptr, &gl, initial_state, final_state,
                      o, o_dtype, cu_seqlens, cu_seqlens_host, n_seqs, B, T, H, K, V, chunk, scale, use_qk_l2norm,
                      gate, gate_dtype, norm_w, eps, y, workspace, workspace_bytes, mode, stream);
}

kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                             const float *g, const float *beta, const float *initial_state,
                             float *final_state, void *o, kda_dtype o_dtype, float *states,
                             const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                             int n_seqs, int B, int T, int H, int K, int V, float scale,
                             int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                             const float *norm_w, float eps, void *y, void *stream) {
    kda::g_err[0] = 0;
    int N = 0;
    kda_status s = check_seq_args("kda_recurrent_fwd", q, k, v, qkv_dtype, g, beta, initial_state,
                                  final_state, o, o_dtype, cu_seqlens, cu_seqlens_host, n_seqs, B, T,
                                  H, K, V, scale, gate, gate_dtype, norm_w, eps, y, N);
    if (s != KDA_OK) return s;
    KDA_REQUIRE(!states || aligned16(states), KDA_ERR_INVALID_ARG, "kda_recurrent_fwd: states must be 16-byte aligned");
    s = check_call_overlaps("kda_recurrent_fwd", q, k, v, qkv_dtype, g, 4, beta, 4, initial_state, final_state, o,
                            o_dtype, states, gate, gate_dtype, norm_w, y, (int64_t)B * T, N, H, K, V);
    if (s != KDA_OK) return s;
    kda::SeqParams p = make_params(q, k, v, qkv_dtype, g, beta, initial_state, final_state, o, o_dtype,
                                   states, cu_seqlens, N, T, H, scale, use_qk_l2norm, gate, gate_dtype,
                                   norm_w, eps, y);
    set_logits(p, nullptr, K);
    return kda::launch_recurrent(p, K, V, (cudaStream_t)stream);
}

kda_status kda_recurrent_step(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                              const float *g, const float *beta, const float *state_in,
                              float *state_out, void *o, kda_dtype o_dtype, int B, int H, int K,
                              int V, float scale, int use_qk_l2norm, const void *gate,
                              kda_dtype gate_dtype, const float *norm_w, float eps, void *y,
                              void *stream) {
    return step_impl("kda_recurrent_step", q, k, v, qkv_dtype, g, beta, nullptr, state_in, state_out, o, o_dtype, B,
                     H, K, V, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, stream);
}

kda_status kda_recurrent_step_logits(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                     const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                     const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                     kda_dtype beta_logits_dtype, const float *state_in, float *state_out,
                                     void *o, kda_dtype o_dtype, int B, int H, int K, int V, float scale,
                                     int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                     const float *norm_w, float eps, void *y, void *stream) {
    const GateLogits gl{g_logits, g_logits_dtype, A_log, dt_bias, g_lower_bound, beta_logits, beta_logits_dtype};
    return step_impl("kda_recurrent_step_logits", q, k, v, qkv_dtype, nullptr, nullptr, &gl, state_in, state_out, o,
                     o_dtype, B, H, K, V, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, stream);
}

kda_status kda_recurrent_step_conv(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                   const float *const conv_weight[3], int W, const float *const conv_state_in[3],
                                   float *const conv_state_out[3], const float *g, const float *beta,
                                   const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                   const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                   kda_dtype beta_logits_dtype, const float *state_in, float *state_out, void *o,
                                   kda_dtype o_dtype, int B, int H, int K, int V, float scale, int use_qk_l2norm,
                                   const void *gate, kda_dtype gate_dtype, const float *norm_w, float eps, void *y,
                                   void *stream) {
    kda::g_err[0] = 0;
    const char *fn = "kda_recurrent_step_conv";
    const bool plain = g || beta, logits = g_logits || beta_logits || A_log;
    KDA_REQUIRE(plain != logits, KDA_ERR_INVALID_ARG,
                "%s: give either g and beta or g_logits, A_log and beta_logits, not both or neither", fn);
    const ConvArgs cv{conv_weight, W, conv_state_in, conv_state_out};
    if (logits) {
        const GateLogits gl{g_logits, g_logits_dtype, A_log, dt_bias, g_lower_bound, beta_logits, beta_logits_dtype};
        return step_impl(fn, q, k, v, qkv_dtype, nullptr, nullptr, &gl, state_in, state_out, o, o_dtype, B, H, K, V,
                         scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, stream, &cv);
    }
    return step_impl(fn, q, k, v, qkv_dtype, g, beta, nullptr, state_in, state_out, o, o_dtype, B, H, K, V, scale,
                     use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, stream, &cv);
}

kda_status kda_gated_rmsnorm(const void *o, kda_dtype o_dtype, const void *gate,
                             kda_dtype gate_dtype, const float *w, float eps, void *y,
                             kda_dtype y_dtype, int64_t rows, int H, int V, void *stream) {
    kda::g_err[0] = 0;
    KDA_REQUIRE((o && gate && y) || rows == 0, KDA_ERR_INVALID_ARG,
                "kda_gated_rmsnorm: o, gate and y must not be NULL");
    KDA_REQUIRE(w, KDA_ERR_INVALID_ARG, "kda_gated_rmsnorm: w must not be NULL");
    KDA_REQUIRE(dtype_ok(o_dtype) && dtype_ok(gate_dtype) && dtype_ok(y_dtype), KDA_ERR_UNSUPPORTED,
                "kda_gated_rmsnorm: unsupported dtype");
    KDA_REQUIRE(rows >= 0 && H > 0, KDA_ERR_INVALID_ARG, "kda_gated_rmsnorm: need rows >= 0 and H > 0");
    KDA_REQUIRE(dim_ok(V), KDA_ERR_UNSUPPORTED, "kda_gated_rmsnorm: V=%d (supported: 32, 64, 128)", V);
    KDA_REQUIRE(eps > 0.f && std::isfinite(eps), KDA_ERR_INVALID_ARG, "kda_gated_rmsnorm: eps must be > 0");
    KDA_REQUIRE(aligned16(o) && aligned16(gate) && aligned16(w) && aligned16(y), KDA_ERR_INVALID_ARG,
                "kda_gated_rmsnorm: every pointer must be 16-byte aligned");
    KDA_REQUIRE(o != y || o_dtype == y_dtype, KDA_ERR_INVALID_ARG,
                "kda_gated_rmsnorm: in place (o == y) needs o_dtype == y_dtype");
    return kda::launch_gated_rmsnorm(o, o_dtype == KDA_BF16, gate, gate_dtype == KDA_BF16, w, eps, y,
                                     y_dtype == KDA_BF16, rows, H, V, (cudaStream_t)stream);
}

kda_status kda_short_conv_fwd(const void *x, kda_dtype x_dtype, const float *weight, const float *bias,
                              const float *conv_state_in, float *conv_state_out, void *y,
                              kda_dtype y_dtype, const int32_t *cu_seqlens,
                              const int32_t *cu_seqlens_host, int n_seqs, int B, int T, int D, int W,
                              int activation, void *stream) {
    kda::g_err[0] = 0;
    const char *fn = "kda_short_conv_fwd";
    const int64_t rows = (int64_t)B * T;
    KDA_REQUIRE(B > 0 && T >= 0 && D > 0, KDA_ERR_INVALID_ARG, "%s: need B > 0, T >= 0, D > 0", fn);
    KDA_REQUIRE(rows == 0 || (x && y), KDA_ERR_INVALID_ARG, "%s: x and y must not be NULL", fn);
    KDA_REQUIRE(weight, KDA_ERR_INVALID_ARG, "%s: weight must not be NULL", fn);
    KDA_REQUIRE(dtype_ok(x_dtype) && dtype_ok(y_dtype), KDA_ERR_UNSUPPORTED, "%s: unsupported dtype", fn);
    KDA_REQUIRE(W >= 2 && W <= 4, KDA_ERR_UNSUPPORTED, "%s: W=%d (supported: 2, 3, 4)", fn, W);
    KDA_REQUIRE(D % 8 == 0, KDA_ERR_UNSUPPORTED, "%s: D=%d must be a multiple of 8", fn, D);
    KDA_REQUIRE(activation == 0 || activation == 1, KDA_ERR_INVALID_ARG, "%s: activation must be 0 or 1", fn);
    KDA_REQUIRE(rows <= (int64_t)INT32_MAX, KDA_ERR_INVALID_ARG, "%s: B*T=%lld too large", fn, (long long)rows);
    const void *ptrs[] = {x, weight, bias, conv_state_in, conv_state_out, y, cu_seqlens};
    for (const void *ptr : ptrs)
        KDA_REQUIRE(!ptr || aligned16(ptr), KDA_ERR_INVALID_ARG, "%s: every pointer must be 16-byte aligned", fn);
    const size_t xbytes = (size_t)rows * D * (x_dtype == KDA_BF16 ? 2 : 4);
    const size_t ybytes = (size_t)rows * D * (y_dtype == KDA_BF16 ? 2 : 4);
    KDA_REQUIRE(rows == 0 || (const char *)y + ybytes <= (const char *)x || (const char *)x + xbytes <= (const char *)y,
                KDA_ERR_INVALID_ARG, "%s: y must not overlap x", fn);
    int N = B;
    if (cu_seqlens) {
        KDA_REQUIRE(B == 1 && n_seqs > 0, KDA_ERR_INVALID_ARG, "%s: varlen needs B == 1 and n_seqs > 0", fn);
        if (cu_seqlens_host) {
            KDA_REQUIRE(cu_seqlens_host[0] == 0, KDA_ERR_INVALID_ARG, "%s: cu_seqlens[0] must be 0", fn);
            for (int i = 0; i < n_seqs; ++i)
                KDA_REQUIRE(cu_seqlens_host[i + 1] >= cu_seqlens_host[i], KDA_ERR_INVALID_ARG,
                            "%s: cu_seqlens must not decrease (entry %d)", fn, i + 1);
            KDA_REQUIRE(cu_seqlens_host[n_seqs] == T, KDA_ERR_INVALID_ARG, "%s: cu_seqlens[n_seqs] = %d but T = %d",
                        fn, cu_seqlens_host[n_seqs], T);
        }
        N = n_seqs;
    } else {
        KDA_REQUIRE(!cu_seqlens_host, KDA_ERR_INVALID_ARG, "%s: cu_seqlens_host given without cu_seqlens", fn);
    }
    if (conv_state_in && conv_state_out) {
        const size_t sbytes = (size_t)N * (W - 1) * D * sizeof(float);
        const char *a = (const char *)conv_state_in, *b = (const char *)conv_state_out;
        const bool overlap = a < b + sbytes && b < a + sbytes;
        KDA_REQUIRE(!overlap || (a == b && !cu_seqlens && T == 1), KDA_ERR_INVALID_ARG,
                    "%s: conv_state_out may alias conv_state_in only for a decode step (dense, T = 1)", fn);
    }
    return kda::launch_short_conv(x, x_dtype == KDA_BF16, weight, bias, conv_state_in, conv_state_out, y,
                                  y_dtype == KDA_BF16, cu_seqlens, N, rows, T, D, W, activation,
                                  (cudaStream_t)stream);
}

kda_status kda_o_proj(const void *y, const void *w_o, void *out, kda_dtype out_dtype, int64_t rows,
                      int in_features, int out_features, void *stream) {
    kda::g_err[0] = 0;
    const char *fn = "kda_o_proj";
    KDA_REQUIRE(rows >= 0 && in_features > 0 && out_features > 0, KDA_ERR_INVALID_ARG,
                "%s: need rows >= 0 and positive feature counts", fn);
    KDA_REQUIRE(rows == 0 || (y && w_o && out), KDA_ERR_INVALID_ARG, "%s: y, w_o and out must not be NULL", fn);
    KDA_REQUIRE(dtype_ok(out_dtype), KDA_ERR_UNSUPPORTED, "%s: unsupported out dtype", fn);
    KDA_REQUIRE(kda::o_proj_supported(in_features, out_features), KDA_ERR_UNSUPPORTED,
                "%s: in_features must be a multiple of 64 and out_features a multiple of 128", fn);
    KDA_REQUIRE(rows <= INT32_MAX, KDA_ERR_INVALID_ARG, "%s: too many rows", fn);
    const void *ptrs[] = {y, w_o, out};
    for (const void *ptr : ptrs)
        KDA_REQUIRE(!ptr || aligned16(ptr), KDA_ERR_INVALID_ARG, "%s: every pointer must be 16-byte aligned", fn);
    if (rows == 0) return KDA_OK;
    {
        const size_t r = (size_t)rows, ob = out_dtype == KDA_BF16 ? 2 : 4;
        const Span o{out, r * out_features * ob, "out"};
        KDA_REQUIRE(!overlaps(o, Span{y, r * in_features * 2, "y"}) &&
                        !overlaps(o, Span{w_o, (size_t)out_features * in_features * 2, "w_o"}),
                    KDA_ERR_INVALID_ARG, "%s: out must not overlap y or w_o", fn);
    }
    return kda::launch_o_proj(y, w_o, out, out_dtype == KDA_BF16, rows, in_features, out_features,
                              (cudaStream_t)stream);
}

}  // extern "C"
