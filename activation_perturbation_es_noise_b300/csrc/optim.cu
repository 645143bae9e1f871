// optim.cu -- the optimiser step that consumes an estimated weight gradient.
//
// The pages train with SGD and momentum and report that Adam works on the
// estimates unchanged (Dust translation, experiment set-up and §3.3 "Dust
// under Adam"; laoyaoba.com, section on Adam compatibility).  Neither page
// fixes the form of the update, so both follow their textbook definitions:
//
//   SGD with momentum (heavy ball, no dampening):
//       b <- mu b + (G + wd W),   W <- W - lr b
//   Adam (Kingma & Ba, 2015) with the weight decay decoupled as in AdamW
//   (Loshchilov & Hutter, 2019), step t >= 1:
//       m <- b1 m + (1 - b1) G,   v <- b2 v + (1 - b2) G^2
//       W <- W - lr ( (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps) + wd W )
//
// Both are one pass over HBM: W, G and the moments are read once and written
// once (G only read), four elements per thread and load, and the same pass can
// write the bf16 copy of W that the next forward feeds to the tensor cores.
#include <cmath>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {
namespace {

struct OptArgs {
    float* W;
    const float* G;
    float* m;  // momentum buffer (SGD) or first moment (Adam)
    float* v;  // second moment (Adam)
    __nv_bfloat16* wbf;  // optional bf16 copy of the updated W
    int64_t n;
    int64_t n4;  // elements handled four at a time (0 when a pointer is unaligned)
    float lr, wd;
    float mu;                  // SGD
    float b1, b2, eps;         // Adam
    float inv_bc1, inv_bc2;    // 1 / (1 - b1^t), 1 / (1 - b2^t)
};

template <bool ADAM>
__device__ __forceinline__ void update(const OptArgs& a, float& w, float g, float& m, float& v) {
    if (ADAM) {
        m = a.b1 * m + (1.0f - a.b1) * g;
        v = a.b2 * v + (1.0f - a.b2) * (g * g);
        const float mhat = m * a.inv_bc1;
        const float den = sqrtf(v * a.inv_bc2) + a.eps;
        w = w - a.lr * (mhat / den + a.wd * w);
    } else {
        m = a.mu * m + (g + a.wd * w);
        w = w - a.lr * m;
    }
}

template <bool ADAM>
__global__ void __launch_bounds__(256) optim_kernel(const OptArgs a) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (int64_t i = t0; i < a.n4; i += stride) {
        if (!DUST_IB(4 * i + 3, a.n)) break;
        float4 w = reinterpret_cast<const float4*>(a.W)[i];
        const float4 g = __ldcs(reinterpret_cast<const float4*>(a.G) + i);
        float4 m = reinterpret_cast<const float4*>(a.m)[i];
        float4 v = ADAM ? reinterpret_cast<const float4*>(a.v)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        update<ADAM>(a, w.x, g.x, m.x, v.x);
        update<ADAM>(a, w.y, g.y, m.y, v.y);
        update<ADAM>(a, w.z, g.z, m.z, v.z);
        update<ADAM>(a, w.w, g.w, m.w, v.w);
        reinterpret_cast<float4*>(a.W)[i] = w;
        reinterpret_cast<float4*>(a.m)[i] = m;
        if (ADAM) reinterpret_cast<float4*>(a.v)[i] = v;
        if (a.wbf) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(w.x, w.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(w.z, w.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(a.wbf)[i] = pk;
        }
    }
    for (int64_t i = 4 * a.n4 + t0; i < a.n; i += stride) {
        float w = a.W[i], m = a.m[i], v = ADAM ? a.v[i] : 0.f;
        update<ADAM>(a, w, a.G[i], m, v);
        a.W[i] = w;
        a.m[i] = m;
        if (ADAM) a.v[i] = v;
        if (a.wbf) a.wbf[i] = __float2bfloat16_rn(w);
    }
}

bool finite(float x) { return x == x && x < INFINITY && x > -INFINITY; }

// 1 / (1 - beta^t) in double on the host, as -1 / expm1(t ln beta) so that it
// keeps its accuracy when beta^t is close to 1 (beta near 1, t small).
float inv_bias_correction(float beta, int64_t t) {
    if (beta == 0.0f) return 1.0f;
    return static_cast<float>(-1.0 / std::expm1(static_cast<double>(t) *
                                                 std::log(static_cast<double>(beta))));
}

dust_status launch_optim(OptArgs& a, bool adam, cudaStream_t s) {
    if (a.n == 0) return DUST_OK;
    const bool vec = aligned(a.W, 16) && aligned(a.G, 16) && aligned(a.m, 16) &&
                     (!adam || aligned(a.v, 16)) && (!a.wbf || aligned(a.wbf, 8));
    a.n4 = vec ? a.n / 4 : 0;
    const int64_t work = a.n4 > 0 ? a.n4 : a.n;
    int64_t blocks = ceil_div(work, 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    timer_begin(s);
    if (adam)
        optim_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    else
        optim_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    timer_end(s);
    return launch_status();
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" dust_status dust_sgd_step(float* W, const float* G, float* momentum_buf, int64_t n,
                                     float lr, float momentum, float weight_decay,
                                     void* W_bf16, void* stream) {
    if (n == 0) return DUST_OK;
    if (!W || !G || !momentum_buf || n < 0) return DUST_ERR_INVALID_ARG;
    if (!aligned(W, 4) || !aligned(G, 4) || !aligned(momentum_buf, 4) ||
        (W_bf16 && !aligned(W_bf16, 2)))
        return DUST_ERR_INVALID_ARG;
    if (!finite(lr) || !(momentum >= 0.0f && momentum <= 1.0f) || !finite(weight_decay) ||
        weight_decay < 0.0f)
        return DUST_ERR_INVALID_ARG;
    OptArgs a{};
    a.W = W;
    a.G = G;
    a.m = momentum_buf;
    a.wbf = static_cast<__nv_bfloat16*>(W_bf16);
    a.n = n;
    a.lr = lr;
    a.wd = weight_decay;
    a.mu = momentum;
    return launch_optim(a, false, static_cast<cudaStream_t>(stream));
}

extern "C" dust_status dust_adam_step(float* W, const float* G, float* m, float* v, int64_t n,
                                      float lr, float beta1, float beta2, float eps,
                                      float weight_decay, int64_t step, void* W_bf16,
                                      void* stream) {
    if (n == 0) return DUST_OK;
    if (!W || !G || !m || !v || n < 0 || step < 1) return DUST_ERR_INVALID_ARG;
    if (!aligned(W, 4) || !aligned(G, 4) || !aligned(m, 4) || !aligned(v, 4) ||
        (W_bf16 && !aligned(W_bf16, 2)))
        return DUST_ERR_INVALID_ARG;
    if (!finite(lr) || !(beta1 >= 0.0f && beta1 < 1.0f) || !(beta2 >= 0.0f && beta2 < 1.0f) ||
        !(eps > 0.0f) || !finite(eps) || !finite(weight_decay) || weight_decay < 0.0f)
        return DUST_ERR_INVALID_ARG;
    OptArgs a{};
    a.W = W;
    a.G = G;
    a.m = m;
    a.v = v;
    a.wbf = static_cast<__nv_bfloat16*>(W_bf16);
    a.n = n;
    a.lr = lr;
    a.wd = weight_decay;
    a.b1 = beta1;
    a.b2 = beta2;
    a.eps = eps;
    a.inv_bc1 = inv_bias_correction(beta1, step);
    a.inv_bc2 = inv_bias_correction(beta2, step);
    return launch_optim(a, true, static_cast<cudaStream_t>(stream));
}

namespace dust {
DUST_DEBUG_READER(8)
}  // namespace dust
