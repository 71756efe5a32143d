// kda_host_stream.cu -- kda_chunk_fwd on host buffers: a dense prompt streamed through the
// device in segments of whole chunks.
//
// Pages: nnterp encyclopedia "Kimi-Linear", section 03 "Loading" (the chunked kernel
// carries the recurrent state from one 64-token chunk to the next).  Because the state
// crosses a call boundary in fp32 exactly as it crosses a chunk boundary, a prompt cut
// into segments of whole chunks gives the result of one call.
//
// Three streams: while the caller's stream runs segment i (state updated in place in the
// workspace), an internal stream copies segment i+1's inputs in and another copies
// segment i-1's outputs out, so for a long prompt the host link rather than the kernel
// sets the pace.  Each tensor of a segment moves as one 2-D copy over the B sequences
// (row pitch T tokens on the host, n tokens on the device).  Two device buffers per
// tensor; events in rings of two order a buffer's reuse after the kernel that read it
// (inputs) or the copy that drained it (outputs).  This host code issues copies and
// kernel calls only: every step of the arithmetic runs in the chunked kernels.
#include <string.h>

#include <cuda_runtime.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDefaultSegment = 1024;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Byte layout of the workspace for one call.  Element sizes of 0 leave a tensor out.
struct HostLayout {
    size_t state, norm_w, a_log, dt_bias;  // offsets of the state and the small parameters
    size_t in[6];                          // q, k, v, g (or its logits), beta (or its logit), gate: buffer 0
    size_t out[2];                         // o, y: buffer 0
    size_t in_row[6], out_row[2];          // bytes per token (all heads) of each tensor
    size_t buf_stride;                     // buffer 1 = buffer 0 + buf_stride
    size_t bytes;

    HostLayout(int B, int H, int K, int V, int seg, size_t e_qkv, size_t e_g, size_t e_b, size_t e_gate,
               size_t e_o, size_t e_y) {
        size_t off = 0;
        auto take = [&](size_t n) {
            const size_t at = off;
            off += round256(n);
            return at;
        };
        state = take((size_t)B * H * K * V * 4);
        norm_w = take((size_t)V * 4);
        a_log = take((size_t)H * 4);
        dt_bias = take((size_t)H * K * 4);
        const size_t rows[6] = {(size_t)H * K * e_qkv, (size_t)H * K * e_qkv, (size_t)H * V * e_qkv,
                                (size_t)H * K * e_g,   (size_t)H * e_b,       (size_t)H * V * e_gate};
        const size_t orow[2] = {(size_t)H * V * e_o, (size_t)H * V * e_y};
        const size_t base = off;
        for (int i = 0; i < 6; ++i) {
            in_row[i] = rows[i];
            in[i] = take((size_t)B * seg * rows[i]);
        }
        for (int i = 0; i < 2; ++i) {
            out_row[i] = orow[i];
            out[i] = take((size_t)B * seg * orow[i]);
        }
        buf_stride = off - base;
        bytes = off + buf_stride;
    }
};

// The streams and events of one call; destroyed on every return path.  Destroying a
// stream or an event with work still queued is allowed: CUDA releases it afterwards.
struct CallStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[8] = {};  // in_ready[2], done[2], out_done[2], start, end
    ~CallStreams() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
    }
};

#define KDA_CUDA_OK(call, what)                                                            \
    do {                                                                                   \
        const cudaError_t e_ = (call);                                                     \
        if (e_ != cudaSuccess) {                                                           \
            set_error("%s: %s failed: %s", fn, what, cudaGetErrorString(e_));             \
            return KDA_ERR_CUDA;                                                           \
        }                                                                                  \
    } while (0)

#define KDA_HOST_REQUIRE(cond, code, ...) \
    do {                                  \
        if (!(cond)) {                    \
            set_error(__VA_ARGS__);       \
            return code;                  \
        }                                 \
    } while (0)

size_t esz(int dtype) { return dtype == KDA_BF16 ? 2 : 4; }

bool host_overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
    return x < y + nb && y < x + na;
}

// One H2D (or D2H) 2-D copy of tokens [t0, t0 + n) of every sequence of a [B, T, row]
// host tensor from (or into) a dense [B, n, row] device buffer.
cudaError_t copy_seg(void *dev, const void *host_base, size_t row, int B, int T, int t0, int n, bool to_device,
                     cudaStream_t st) {
    if (!row || n == 0) return cudaSuccess;
    char *h = const_cast<char *>(static_cast<const char *>(host_base)) + (size_t)t0 * row;
    if (to_device)
        return cudaMemcpy2DAsync(dev, (size_t)n * row, h, (size_t)T * row, (size_t)n * row, B,
                                 cudaMemcpyHostToDevice, st);
    return cudaMemcpy2DAsync(h, (size_t)T * row, dev, (size_t)n * row, (size_t)n * row, B, cudaMemcpyDeviceToHost,
                             st);
}

kda_status host_impl(const char *fn, const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                     const float *g, const float *beta, const GateLogits *gl, const float *initial_state,
                     float *final_state, void *o, kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk,
                     float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w,
                     float eps, void *y, int segment, void *workspace, size_t workspace_bytes, int mode,
                     void *stream) {
    KDA_HOST_REQUIRE(B > 0 && T >= 0 && H > 0 && K > 0 && V > 0, KDA_ERR_INVALID_ARG,
                     "%s: need B > 0, T >= 0 and H, K, V > 0", fn);
    KDA_HOST_REQUIRE(chunk == 16 || chunk == 32 || chunk == 64, KDA_ERR_UNSUPPORTED,
                     "%s: chunk=%d (supported: 16, 32, 64)", fn, chunk);
    const int seg = segment > 0 ? segment : kDefaultSegment;
    KDA_HOST_REQUIRE(seg % 64 == 0, KDA_ERR_INVALID_ARG,
                     "%s: segment=%d must be a multiple of 64 tokens (whole chunks)", fn, seg);
    KDA_HOST_REQUIRE(q || T == 0, KDA_ERR_INVALID_ARG, "%s: q must not be NULL", fn);
    KDA_HOST_REQUIRE(!gate || norm_w, KDA_ERR_INVALID_ARG, "%s: the gated norm needs norm_w", fn);
    KDA_HOST_REQUIRE(!gl || gl->A_log, KDA_ERR_INVALID_ARG, "%s: A_log must not be NULL", fn);
    KDA_HOST_REQUIRE(workspace && ((uintptr_t)workspace & 255u) == 0, KDA_ERR_INVALID_ARG,
                     "%s: the device workspace must be given, 256-byte aligned", fn);
    const bool want_o = o != nullptr, want_y = gate && y;
    KDA_HOST_REQUIRE(want_o || want_y || T == 0, KDA_ERR_INVALID_ARG,
                     "%s: o may be NULL only when the gated norm writes y", fn);
    // the fp32 path writes o into y's buffer and normalises there when o is not wanted
    const size_t e_g = gl ? esz(gl->z_dtype) : 4, e_b = gl ? esz(gl->b_dtype) : 4;
    const HostLayout L(B, H, K, V, seg, esz(qkv_dtype), e_g, e_b, gate ? esz(gate_dtype) : 0,
                       want_o ? esz(o_dtype) : 0, want_y ? esz(o_dtype) : 0);
    KDA_HOST_REQUIRE(workspace_bytes >= L.bytes, KDA_ERR_INVALID_ARG,
                     "%s: the workspace holds %zu bytes, this call needs %zu (kda_chunk_fwd_host_workspace_size)", fn,
                     workspace_bytes, L.bytes);
    const void *src[6] = {q, k, v, gl ? gl->z : g, gl ? gl->b : beta, gate};
    void *dst[2] = {o, want_y ? y : nullptr};
    // copies out of one segment run while the next segment's inputs are read: no host
    // output may share bytes with a host input
    {
        const size_t rows = (size_t)B * T, st = (size_t)B * H * K * V * 4;
        for (int j = 0; j < 2; ++j) {
            for (int i = 0; i < 6; ++i)
                KDA_HOST_REQUIRE(!host_overlap(dst[j], rows * L.out_row[j], src[i], rows * L.in_row[i]),
                                 KDA_ERR_INVALID_ARG, "%s: the outputs must not overlap the inputs", fn);
            KDA_HOST_REQUIRE(!host_overlap(dst[j], rows * L.out_row[j], final_state, final_state ? st : 0),
                             KDA_ERR_INVALID_ARG, "%s: the outputs must not overlap final_state", fn);
        }
        KDA_HOST_REQUIRE(!host_overlap(o, rows * L.out_row[0], dst[1], rows * L.out_row[1]), KDA_ERR_INVALID_ARG,
                         "%s: o must not overlap y", fn);
        for (int i = 0; i < 6; ++i)
            KDA_HOST_REQUIRE(!host_overlap(final_state, final_state ? st : 0, src[i], rows * L.in_row[i]),
                             KDA_ERR_INVALID_ARG, "%s: final_state must not overlap the inputs", fn);
    }

    char *ws = static_cast<char *>(workspace);
    cudaStream_t main = (cudaStream_t)stream;
    CallStreams cs;
    KDA_CUDA_OK(cudaStreamCreateWithFlags(&cs.in, cudaStreamNonBlocking), "creating a copy stream");
    KDA_CUDA_OK(cudaStreamCreateWithFlags(&cs.out, cudaStreamNonBlocking), "creating a copy stream");
    for (cudaEvent_t &e : cs.ev) KDA_CUDA_OK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "creating an event");
    cudaEvent_t *in_ready = cs.ev, *done = cs.ev + 2, *out_done = cs.ev + 4, start = cs.ev[6], end = cs.ev[7];
    // the copy streams start after the caller's earlier work (which may still use the workspace)
    KDA_CUDA_OK(cudaEventRecord(start, main), "recording an event");
    KDA_CUDA_OK(cudaStreamWaitEvent(cs.in, start, 0), "ordering the copy stream");
    KDA_CUDA_OK(cudaStreamWaitEvent(cs.out, start, 0), "ordering the copy stream");

    // the call's own parameters and the initial state, on the caller's stream
    float *state = reinterpret_cast<float *>(ws + L.state);
    const size_t st_bytes = (size_t)B * H * K * V * 4;
    if (initial_state)
        KDA_CUDA_OK(cudaMemcpyAsync(state, initial_state, st_bytes, cudaMemcpyHostToDevice, main), "copying the state in");
    else
        KDA_CUDA_OK(cudaMemsetAsync(state, 0, st_bytes, main), "clearing the state");
    float *d_norm_w = nullptr, *d_alog = nullptr, *d_dtb = nullptr;
    if (gate) {
        d_norm_w = reinterpret_cast<float *>(ws + L.norm_w);
        KDA_CUDA_OK(cudaMemcpyAsync(d_norm_w, norm_w, (size_t)V * 4, cudaMemcpyHostToDevice, main), "copying norm_w");
    }
    GateLogits dgl{};
    if (gl) {
        dgl = *gl;
        d_alog = reinterpret_cast<float *>(ws + L.a_log);
        KDA_CUDA_OK(cudaMemcpyAsync(d_alog, gl->A_log, (size_t)H * 4, cudaMemcpyHostToDevice, main), "copying A_log");
        dgl.A_log = d_alog;
        if (gl->dt_bias) {
            d_dtb = reinterpret_cast<float *>(ws + L.dt_bias);
            KDA_CUDA_OK(cudaMemcpyAsync(d_dtb, gl->dt_bias, (size_t)H * K * 4, cudaMemcpyHostToDevice, main),
                        "copying dt_bias");
            dgl.dt_bias = d_dtb;
        }
    }

    const int n_seg = (T + seg - 1) / seg;
    auto in_buf = [&](int i, int b) { return ws + L.in[i] + (size_t)b * L.buf_stride; };
    auto out_buf = [&](int j, int b) { return ws + L.out[j] + (size_t)b * L.buf_stride; };
    auto copy_in = [&](int s) -> kda_status {
        const int t0 = s * seg, n = T - t0 < seg ? T - t0 : seg, b = s & 1;
        if (s >= 2) KDA_CUDA_OK(cudaStreamWaitEvent(cs.in, done[b], 0), "ordering a copy");  // segment s-2 read it
        for (int i = 0; i < 6; ++i)
            if (src[i]) KDA_CUDA_OK(copy_seg(in_buf(i, b), src[i], L.in_row[i], B, T, t0, n, true, cs.in), "a copy in");
        KDA_CUDA_OK(cudaEventRecord(in_ready[b], cs.in), "recording an event");
        return KDA_OK;
    };
    kda_status s = KDA_OK;
    if (n_seg > 0 && (s = copy_in(0)) != KDA_OK) return s;
    for (int i = 0; i < n_seg; ++i) {
        if (i + 1 < n_seg && (s = copy_in(i + 1)) != KDA_OK) return s;
        const int t0 = i * seg, n = T - t0 < seg ? T - t0 : seg, b = i & 1;
        KDA_CUDA_OK(cudaStreamWaitEvent(main, in_ready[b], 0), "ordering the kernel");
        if (i >= 2) KDA_CUDA_OK(cudaStreamWaitEvent(main, out_done[b], 0), "ordering the kernel");  // i-2 drained
        void *od = want_o ? out_buf(0, b) : nullptr, *yd = want_y ? out_buf(1, b) : nullptr;
        GateLogits sgl = dgl;  // with logits, they travel in the g and beta buffers
        sgl.z = in_buf(3, b);
        sgl.b = in_buf(4, b);
        s = chunk_call(fn, in_buf(0, b), in_buf(1, b), in_buf(2, b), qkv_dtype,
                       gl ? nullptr : reinterpret_cast<const float *>(in_buf(3, b)),
                       gl ? nullptr : reinterpret_cast<const float *>(in_buf(4, b)), gl ? &sgl : nullptr, state, state,
                       od, o_dtype, B, n, H, K, V, chunk, scale, use_qk_l2norm, gate ? in_buf(5, b) : nullptr,
                       gate_dtype, d_norm_w, eps, yd, mode, main);
        if (s != KDA_OK) return s;
        KDA_CUDA_OK(cudaEventRecord(done[b], main), "recording an event");
        KDA_CUDA_OK(cudaStreamWaitEvent(cs.out, done[b], 0), "ordering a copy");
        for (int j = 0; j < 2; ++j)
            if (dst[j]) KDA_CUDA_OK(copy_seg(out_buf(j, b), dst[j], L.out_row[j], B, T, t0, n, false, cs.out), "a copy out");
        KDA_CUDA_OK(cudaEventRecord(out_done[b], cs.out), "recording an event");
    }
    if (final_state) {
        KDA_CUDA_OK(cudaEventRecord(end, main), "recording an event");
        KDA_CUDA_OK(cudaStreamWaitEvent(cs.out, end, 0), "ordering a copy");
        KDA_CUDA_OK(cudaMemcpyAsync(final_state, state, st_bytes, cudaMemcpyDeviceToHost, cs.out), "copying the state out");
    }
    // the caller's stream covers the whole call: it waits for the last copies out
    KDA_CUDA_OK(cudaEventRecord(end, cs.out), "recording an event");
    KDA_CUDA_OK(cudaStreamWaitEvent(main, end, 0), "joining the copy stream");
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" {

size_t kda_chunk_fwd_host_workspace_size(int B, int H, int K, int V, int segment) {
    if (B <= 0 || H <= 0 || K <= 0 || V <= 0 || segment < 0) return 0;
    const kda::HostLayout L(B, H, K, V, segment > 0 ? segment : kda::kDefaultSegment, 4, 4, 4, 4, 4, 4);
    return L.bytes;
}

kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v, kda_dtype qkv_dtype, const float *g,
                              const float *beta, const float *initial_state, float *final_state, void *o,
                              kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk, float scale,
                              int use_qk_l2norm, const void *gate, kda_dtype gate_dtype, const float *norm_w,
                              float eps, void *y, int segment, void *workspace, size_t workspace_bytes, int mode,
                              void *stream) {
    kda::set_error("%s", "");
    const char *fn = "kda_chunk_fwd_host";
    if (!g || !beta) {
        if ((int64_t)B * T != 0) {
            kda::set_error("%s: g and beta must not be NULL", fn);
            return KDA_ERR_INVALID_ARG;
        }
    }
    return kda::host_impl(fn, q, k, v, qkv_dtype, g, beta, nullptr, initial_state, final_state, o, o_dtype, B, T, H,
                          K, V, chunk, scale, use_qk_l2norm, gate, gate_dtype, norm_w, eps, y, segment, workspace,
                          workspace_bytes, mode, stream);
}

kda_status kda_chunk_fwd_logits_host(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                     const void *g_logits, kda_dtype g_logits_dtype, const float *A_log,
                                     const float *dt_bias, float g_lower_bound, const void *beta_logits,
                                     kda_dtype beta_logits_dtype, const float *initial_state, float *final_state,
                                     void *o, kda_dtype o_dtype, int B, int T, int H, int K, int V, int chunk,
                                     float scale, int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                     const float *norm_w, float eps, void *y, int segment, void *workspace,
                                     size_t workspace_bytes, int mode, void *stream) {
    kda::set_error("%s", "");
    const kda::GateLogits gl{g_logits, g_logits_dtype, A_log, dt_bias, g_lower_bound, beta_logits, beta_logits_dtype};
    return kda::host_impl("kda_chunk_fwd_logits_host", q, k, v, qkv_dtype, nullptr, nullptr, &gl, initial_state,
                          final_state, o, o_dtype, B, T, H, K, V, chunk, scale, use_qk_l2norm, gate, gate_dtype,
                          norm_w, eps, y, segment, workspace, workspace_bytes, mode, stream);
}

}  // extern "C"
