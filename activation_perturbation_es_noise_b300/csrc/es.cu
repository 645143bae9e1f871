// es.cu -- weight-space ES for the few parameters the activation method does
// not cover.
//
// The pages estimate every weight by perturbing activations except the 2L
// residual-mixing scalars of the network (Dust translation, §2.1), which stay
// with weight-space evolution strategies: a population of perturbed copies of
// those scalars, one forward each, and the noise weighted by the centred loss
// change.  The library supplies the population side:
//   theta_i = theta + sigma eps_i,                       i = 0 .. K-1
//   g = (1/(K sigma)) sum_i (L_i - mean_j L_j) eps_i      (an estimate of +dL/dtheta)
// with eps_i[j] the normal of the same counter scheme as the activation noise,
// (j/4, token0, draw0 + i, layer) -- one "token", the parameters as channels.
// The K losses come from the caller's forwards.
#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {
namespace {

// One thread per (draw, block of 4 parameters).
__global__ void es_perturb_kernel(const float* __restrict__ theta, int64_t n, int K,
                                  uint32_t draw0, uint32_t token, uint32_t layer, float sigma,
                                  PhiloxKeys keys, float* __restrict__ out) {
    const int64_t nblk = (n + 3) / 4;
    const int64_t total = nblk * K;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(idx / nblk);
        const int64_t j = idx - static_cast<int64_t>(i) * nblk;
        const float4 e = words_to_normals(philox4x32_10(static_cast<uint32_t>(j), token,
                                                        draw0 + static_cast<uint32_t>(i), layer,
                                                        keys));
        const float ev[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = 4 * j + k;
            if (c < n && DUST_IB(static_cast<int64_t>(i) * n + c, static_cast<int64_t>(K) * n)) out[static_cast<int64_t>(i) * n + c] = fmaf(sigma, ev[k], theta[c]);
        }
    }
}

// One thread per block of 4 parameters, the draws in order; every thread
// forms the losses' mean in the same order (no reduction needed), as an
// offset from the first loss so that the small differences L_i - L_0 are
// exact and the centring keeps their precision.
__global__ void es_estimate_kernel(const float* __restrict__ losses, int64_t n, int K,
                                   uint32_t draw0, uint32_t token, uint32_t layer, float scale,
                                   PhiloxKeys keys, float* __restrict__ g) {
    const int64_t nblk = (n + 3) / 4;
    const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (j >= nblk) return;
    const float pilot = losses[0];
    float mean = 0.f;
    for (int i = 0; i < K; ++i) mean += losses[i] - pilot;
    mean /= static_cast<float>(K);
    const BlockHalf bh = philox_block_half(static_cast<uint32_t>(j), layer, keys);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < K; ++i) {
        const float c = (losses[i] - pilot) - mean;
        const float4 e = words_to_normals(
            philox_rest(philox_draw_half(draw0 + static_cast<uint32_t>(i), token, keys), bh, keys));
        acc[0] = fmaf(c, e.x, acc[0]);
        acc[1] = fmaf(c, e.y, acc[1]);
        acc[2] = fmaf(c, e.z, acc[2]);
        acc[3] = fmaf(c, e.w, acc[3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (4 * j + k < n && DUST_IB(4 * j + k, n)) g[4 * j + k] = acc[k] * scale;
}

bool es_args_ok(int64_t n, const dust_noise& nz) {
    return n >= 1 && n <= (1LL << 26) && nz.num_draws >= 2 && nz.num_draws <= (1u << 20) &&
           nz.sigma > 0.0f && nz.sigma < INFINITY &&
           static_cast<uint64_t>(nz.draw0) + nz.num_draws <= (1ULL << 32);
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" dust_status dust_es_perturb(const float* theta, int64_t n, dust_noise nz,
                                       float* theta_out, void* stream) {
    if (!theta || !theta_out || !es_args_ok(n, nz)) return DUST_ERR_INVALID_ARG;
    const int64_t work = ((n + 3) / 4) * nz.num_draws;
    int64_t blocks = ceil_div(work, 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    es_perturb_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        theta, n, static_cast<int>(nz.num_draws), nz.draw0, nz.token0, nz.layer, nz.sigma,
        philox_round_keys(nz.seed), theta_out);
    return launch_status();
}

extern "C" dust_status dust_es_estimate(const float* losses, int64_t n, dust_noise nz, float* g,
                                        void* stream) {
    if (!losses || !g || !es_args_ok(n, nz)) return DUST_ERR_INVALID_ARG;
    const float scale =
        static_cast<float>(1.0 / (static_cast<double>(nz.num_draws) * nz.sigma));
    es_estimate_kernel<<<static_cast<unsigned>(ceil_div((n + 3) / 4, 128)), 128, 0,
                         static_cast<cudaStream_t>(stream)>>>(
        losses, n, static_cast<int>(nz.num_draws), nz.draw0, nz.token0, nz.layer, scale,
        philox_round_keys(nz.seed), g);
    return launch_status();
}

namespace dust {
DUST_DEBUG_READER(9)
}  // namespace dust
