// combine.cuh -- the routing-weighted gather-combine of the k expert outputs
// of every token (each token needs 10 of the model's experts, upstream Strata
// README, "How does it work?").
#pragma once

#include "common.cuh"

namespace moeq {

// One CTA per token; y[t] = (res ? res[t] : 0) + sum_j w[t,j] D[inv[t,j]], j ascending.
// A sorted position outside [0, P) (a pair the permutation rejected) adds
// nothing and raises MOEQ_STATUS_BAD_INDEX.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ D, const int32_t *__restrict__ inv,
                                                      const float *__restrict__ w, int k, int H, long long P,
                                                      const float *__restrict__ res, float *__restrict__ y) {
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int pos = inv[(size_t)t * k + threadIdx.x];
        if (pos < 0 || pos >= P) set_status(MOEQ_STATUS_BAD_INDEX);
    }
    for (int h = 4 * threadIdx.x; h < H; h += 4 * blockDim.x) {
        float4 acc = res ? *reinterpret_cast<const float4 *>(res + (size_t)t * H + h) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int pos = inv[(size_t)t * k + j];
            if (pos < 0 || pos >= P) continue;
            const float wj = w[(size_t)t * k + j];
            const float4 d = __ldg(reinterpret_cast<const float4 *>(D + (size_t)pos * H + h));
            acc.x = fmaf(wj, d.x, acc.x);
            acc.y = fmaf(wj, d.y, acc.y);
            acc.z = fmaf(wj, d.z, acc.z);
            acc.w = fmaf(wj, d.w, acc.w);
        }
        *reinterpret_cast<float4 *>(y + (size_t)t * H + h) = acc;
    }
}

// y = residual ? x : 0 (the starting value the expert kernels add into).
__global__ void init_y_kernel(const float *__restrict__ x, float *__restrict__ y, size_t n, int residual) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 4; i += (size_t)gridDim.x * blockDim.x) {
        float4 v = residual ? reinterpret_cast<const float4 *>(x)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(y)[i] = v;
    }
}

}  // namespace moeq
