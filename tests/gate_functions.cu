// Test harness (compiled by tests/test_gpu_gate_functions.py): evaluates on
// the GPU every form of the gate that the library's kernels use, and CUDA's
// own log2f(1 / (1 + expf(-x))) for comparison.
#include "../hybrid_gated_linear_attn_b300/csrc/prefill_ws.cuh"

__global__ void eval_kernel(const float *x, float *out, int n, int which)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float g = x[i];
    float r = 0.f;
    switch (which) {
    case 0: r = lizard::ws::log2_sigmoid(g); break;                          // polynomial (tensor-core backward)
    case 1: r = lizard::ws::log2_sigmoid2(make_float2(g, g)).x; break;       // ex2 + lg2 (exact intra-chunk path)
    case 3: r = lizard::log_sigmoid(g); break;                               // natural log (CUDA-core kernels)
    case 4: r = lizard::ws::rcp(1.f + lizard::ws::ex2(g * -lizard::ws::LOG2E)); break;  // sigmoid as 1 / (1 + 2^{-g log2 e})
    case 5: r = log2f(1.f / (1.f + expf(-g))); break;                         // CUDA's own, for comparison
    default: break;
    }
    out[i] = r;
}

extern "C" int lizard_test_eval_gate(const float *x, float *out, int n, int which)
{
    eval_kernel<<<(n + 255) / 256, 256>>>(x, out, n, which);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 1;
}
