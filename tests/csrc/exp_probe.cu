// exp_probe.cu - test-only wrappers that run the library's device helpers
// exp_shifted (common.cuh) and merge2 (pipeline.cuh) elementwise, and CUDA's
// expf on the same fp32 differences, so a test can bound the helpers' error.
// Built by tests/test_gpu_exp_helper.py; not part of librowops.
#include <cuda_runtime.h>

#include "../../row_wise_softmax_warp_gb300/csrc/common.cuh"
#include "../../row_wise_softmax_warp_gb300/csrc/pipeline.cuh"

namespace {

__global__ void k_exp_shifted(const float* x, const float* m, float* out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = rowops::exp_shifted(x[i], m[i]);
}

__global__ void k_expf_diff(const float* x, const float* m, float* out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = expf(x[i] - m[i]);
}

__global__ void k_merge2(const float* m1, const float* s1, const float* m2, const float* s2, float* m_out,
                         float* s_out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        float m = m1[i], s = s1[i];
        rowops::merge2(m, s, m2[i], s2[i]);
        m_out[i] = m;
        s_out[i] = s;
    }
}

unsigned blocks(int n) { return unsigned((n + 255) / 256); }

}  // namespace

extern "C" int probe_exp_shifted(const float* x, const float* m, float* out, int n) {
    if (n <= 0) return 0;
    k_exp_shifted<<<blocks(n), 256>>>(x, m, out, n);
    return int(cudaDeviceSynchronize());
}

extern "C" int probe_expf_diff(const float* x, const float* m, float* out, int n) {
    if (n <= 0) return 0;
    k_expf_diff<<<blocks(n), 256>>>(x, m, out, n);
    return int(cudaDeviceSynchronize());
}

extern "C" int probe_merge2(const float* m1, const float* s1, const float* m2, const float* s2, float* m_out,
                            float* s_out, int n) {
    if (n <= 0) return 0;
    k_merge2<<<blocks(n), 256>>>(m1, s1, m2, s2, m_out, s_out, n);
    return int(cudaDeviceSynchronize());
}
