// kda_chunk_noalloc.cu -- kda_chunk_fwd_noalloc: the split tensor-core prefill with its
// scratch in a fixed array that belongs to the library, for callers that cannot hand
// it a workspace.
//
// The split prefill keeps every chunk's state-independent operands between its two
// kernels (32 KiB per chunk slot and head, kda_chunk_workspace_size).  kda_chunk_fwd
// takes that memory from the caller.  Some callers cannot provide it: code behind a
// fixed operator or plugin interface whose calls carry only the input and output
// tensors, and code running where device allocation is not allowed or not available
// (a memory pool owned by someone else, a real-time path that must not allocate).
// For them this entry point uses a file-scope device array of kNoallocWorkspaceBytes
// instead, so a call allocates nothing: no cudaMalloc, no cudaFree, no allocating
// library routine.  The array is part of the library's device image: every GPU that
// loads the library holds it until the process exits.
#include <mutex>

#include "kda_chunk_common.cuh"
#include "kda_internal.cuh"

namespace kda {
namespace {

// 64 MiB: 2048 (chunk slot, head) blobs, e.g. one prompt of up to 1280 tokens at 96 heads.
constexpr size_t kNoallocWorkspaceBytes = size_t(64) << 20;

static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoallocWorkspaceBytes];

// The array's device address on each device (devices 0-63), looked up on the first call
// made with that device current.  In host code the array's name is only a stand-in for
// the symbol, never an address a kernel may be given.
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {nullptr};

void *noalloc_workspace() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (dev >= 0 && dev < 64 && g_noalloc_ptr[dev]) return g_noalloc_ptr[dev];
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_workspace);
    if (e != cudaSuccess || !ptr) {
        set_error("kda_chunk_fwd_noalloc: cannot find the device address of the fixed workspace: %s",
                  cudaGetErrorString(e));
        cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0 && dev < 64) g_noalloc_ptr[dev] = ptr;
    return ptr;
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, kda_dtype qkv_dtype,
                                            const float *g, const float *beta, const float *initial_state,
                                            float *final_state, void *o, kda_dtype o_dtype,
                                            const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int n_seqs,
                                            int B, int T, int H, int K, int V, int chunk, float scale,
                                            int use_qk_l2norm, const void *gate, kda_dtype gate_dtype,
                                            const float *norm_w, float eps, void *y, int mode, void *stream) {
    const char *fn = "kda_chunk_fwd_noalloc";
    const int N = n_seqs > 0 ? n_seqs : B;
    if (B > 0 && T > 0 && H > 0 && N > 0) {
        const size_t need = kda::chunk_workspace_bytes((int64_t)B * T, N, H);
        if (need > kda::kNoallocWorkspaceBytes) {
            kda::set_error("%s: this call needs %zu bytes of scratch and the fixed workspace holds %zu "
                           "(%d (chunk slot, head) blobs); use kda_chunk_fwd with a workspace",
                           fn, need, kda::kNoallocWorkspaceBytes, (int)(kda::kNoallocWorkspaceBytes / kda::chunk::kBlobBytes));
            return KDA_ERR_UNSUPPORTED;
        }
    }
    void *ws = kda::noalloc_workspace();
    if (!ws) return KDA_ERR_CUDA;
    return kda::chunk_fwd_entry(fn, q, k, v, qkv_dtype, g, beta, initial_state, final_state, o, o_dtype, cu_seqlens,
                                cu_seqlens_host, n_seqs, B, T, H, K, V, chunk, scale, use_qk_l2norm, gate, gate_dtype,
                                norm_w, eps, y, ws, kda::kNoallocWorkspaceBytes, mode, stream);
}
