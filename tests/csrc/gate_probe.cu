// gate_probe.cu -- GPU unit test of the device functions that turn the layer's logits
// into the decay g and the write strength beta (kda_internal.cuh): one thread per
// element evaluates gate_of_logit and beta_of_logit exactly as the kernels do, for
// comparison with the fp64 formulas on the host.
#include <cuda_runtime.h>

#include "kda_internal.cuh"

namespace {

__global__ void gate_probe_kernel(const float *x, int n, float a_h, float lower, float *g, float *beta) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    g[i] = kda::gate_of_logit(x[i], a_h, lower);
    beta[i] = kda::beta_of_logit(x[i]);
}

}  // namespace

extern "C" int gate_probe(const float *x, int n, float a_h, float lower, float *g, float *beta, void *stream) {
    if (n <= 0) return 0;
    gate_probe_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(x, n, a_h, lower, g, beta);
    return (int)cudaGetLastError();
}
