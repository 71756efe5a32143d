// kda_oproj.cu -- the layer's output projection of the gated-norm output.
//
// Page: Kimi-K3 atlas "gate-project (decode, P = 1000)", sections "Parameters"
// (output projection 88,080,384 weights = 12288 inputs x 7168 outputs) and "Code"
// (o = o_proj(o) after o_norm and the heads flattened to heads * head_dim).
//
//   out[r][n] = sum_c y[r][c] * w_o[n][c]      (nn.Linear, no bias)
//
// A plain dense GEMM: it runs in cuBLASLt (bf16 operands, fp32 accumulation) on the
// caller's workspace.  In column-major terms out^T [N, M] = (W [K, N])^T y^T [K, M],
// i.e. A = w_o read transposed, B = y, with M = rows, N = out_features, K = in_features.
// The cuBLASLt handle is created once per process (host state); the plan for the
// last shape is cached.
#include <cublasLt.h>

#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

std::mutex g_lt_mutex;
cublasLtHandle_t g_lt = nullptr;

struct Plan {
    int64_t M = -1;
    int N = 0, K = 0, out_bf16 = -1;
    size_t ws = 0;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
    cublasLtMatmulAlgo_t algo;
    void release() {
        if (op) cublasLtMatmulDescDestroy(op);
        if (a) cublasLtMatrixLayoutDestroy(a);
        if (b) cublasLtMatrixLayoutDestroy(b);
        if (c) cublasLtMatrixLayoutDestroy(c);
        op = nullptr;
        a = b = c = nullptr;
        M = -1;
    }
};
Plan g_plan;

kda_status lt_fail(const char *what, cublasStatus_t s) {
    set_error("o_proj: %s failed (cublas status %d)", what, (int)s);
    return KDA_ERR_CUDA;
}

}  // namespace

kda_status launch_o_proj(const void *y, const void *w, void *out, int out_bf16, int64_t M, int K, int N, void *ws,
                         size_t ws_bytes, cudaStream_t st) {
    std::lock_guard<std::mutex> lock(g_lt_mutex);
    cublasStatus_t s;
    if (!g_lt && (s = cublasLtCreate(&g_lt)) != CUBLAS_STATUS_SUCCESS) return lt_fail("cublasLtCreate", s);
    Plan &pl = g_plan;
    if (pl.M != M || pl.N != N || pl.K != K || pl.out_bf16 != out_bf16 || pl.ws != ws_bytes) {
        pl.release();
        if ((s = cublasLtMatmulDescCreate(&pl.op, CUBLAS_COMPUTE_32F, CUDA_R_32F)) != CUBLAS_STATUS_SUCCESS)
            return lt_fail("cublasLtMatmulDescCreate", s);
        const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
        cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta));
        cublasLtMatmulDescSetAttribute(pl.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb));
        if ((s = cublasLtMatrixLayoutCreate(&pl.a, CUDA_R_16BF, K, N, K)) != CUBLAS_STATUS_SUCCESS ||
            (s = cublasLtMatrixLayoutCreate(&pl.b, CUDA_R_16BF, K, M, K)) != CUBLAS_STATUS_SUCCESS ||
            (s = cublasLtMatrixLayoutCreate(&pl.c, out_bf16 ? CUDA_R_16BF : CUDA_R_32F, N, M, N)) !=
                CUBLAS_STATUS_SUCCESS) {
            pl.release();
            return lt_fail("cublasLtMatrixLayoutCreate", s);
        }
        cublasLtMatmulPreference_t pref = nullptr;
        cublasLtMatmulPreferenceCreate(&pref);
        cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes, sizeof(ws_bytes));
        cublasLtMatmulHeuristicResult_t res;
        int found = 0;
        s = cublasLtMatmulAlgoGetHeuristic(g_lt, pl.op, pl.a, pl.b, pl.c, pl.c, pref, 1, &res, &found);
        cublasLtMatmulPreferenceDestroy(pref);
        if (s != CUBLAS_STATUS_SUCCESS || found == 0) {
            pl.release();
            set_error("o_proj: no cuBLASLt algorithm for M=%lld N=%d K=%d", (long long)M, N, K);
            return KDA_ERR_UNSUPPORTED;
        }
        pl.algo = res.algo;
        pl.M = M;
        pl.N = N;
        pl.K = K;
        pl.out_bf16 = out_bf16;
        pl.ws = ws_bytes;
    }
    const float alpha = 1.f, beta = 0.f;
    s = cublasLtMatmul(g_lt, pl.op, &alpha, w, pl.a, y, pl.b, &beta, out, pl.c, out, pl.c, &pl.algo, ws, ws_bytes, st);
    if (s != CUBLAS_STATUS_SUCCESS) return lt_fail("cublasLtMatmul", s);
    note_launch();
    return check_launch("o_proj (cuBLASLt)");
}

}  // namespace kda
