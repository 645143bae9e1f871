// head.cu -- the LM-head estimator, perturbed on the cached logits.
//
// The pages perturb the head's output (the logits) directly and recompute
// only the cross-entropy, which is cheap enough to give the head a much larger
// population (laoyaoba.com article, section 机制拆解; Dust translation,
// hn.213312.xyz, §2.3 干扰与调优).  With gamma = 0 the reward of a token is
// its own centred loss decrease (§2.2 信用分配), so for draw i and token t
//
//   dl_{i,t} = CE(z_t + sigma a_{i,t}) - CE(z_t)
//            = log sum_v p_{t,v} exp(sigma a_{i,t,v}) - sigma a_{i,t,y_t},
//
// with p_t = softmax(z_t) (the lse of the clean logits cancels exactly), and
//
//   g_t = -(1/(K sigma)) sum_i c_{i,t} a_{i,t},  c_{i,t} = -(dl_{i,t} - m_t),
//       = (S1_t - m_t S0_t) / (K sigma),
//   S1_t = sum_i dl_{i,t} a_{i,t},  S0_t = sum_i a_{i,t},  m_t = mean_i dl_{i,t}.
//
// One CTA owns one token (and one chunk of draws when there are too few
// tokens to fill the GPU).  Its threads hold the token's probabilities and the
// S1/S0 accumulators of their channels in registers; every draw regenerates
// the noise of those channels from its counter, reduces sum p e^{sigma a}
// across the CTA, and folds dl a into the accumulators.  Nothing per draw ever
// leaves the chip.
#include <cmath>

#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {
namespace {

struct HeadArgs {
    const float* logits;
    const int32_t* targets;
    int T, V, nblk, K, Q, chunk;
    uint32_t draw0, token0, layer;
    float sig_l2e;  // s = sigma * log2(e): the kernel works with b = s a
    float clog;     // -2 ln(2) s^2: the fast Box-Muller's log constant for b = s a
    float g_scale;  // 1 / (K sigma s): turns the b-scaled sums into g
    float qscale;   // 2^E > 0: the pair kernel's fixed-point scale of sum p 2^b
    float qinv;     // 2^-E (qscale = 0: float sums instead)
    float* g_hat;   // T x V fp32, may be null
    __nv_bfloat16* gbf;
    int64_t ldg;    // row stride of gbf (elements)
    float* part_s1;  // Q x T x V
    float* part_s0;
    float* part_dl;  // Q x T
    uint32_t* status;
    // Vocabulary-chunk mode (the kernel's CH flag): this launch covers columns
    // col0 .. col0 + V - 1 of rows ldz apart, p is normalised by the full
    // row's log-sum-exp lse[t], the rest of the row's probability mass stays
    // unperturbed, and draw i uses the counter draw0 + i * draw_stride.
    int64_t ldz;       // row stride of the logits, g_hat and the partials
    int col0, Vfull;
    uint32_t draw_stride;
    const float* lse;
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ln S for S > 0 (S is a probability-weighted mean of exp(sigma a), near 1):
// the same exponent split and atanh series as the noise generator's log.
__device__ __forceinline__ float log_pos(float S) {
    return -0.5f * neg2_log_unit(S);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Block-wide reductions for the once-per-token softmax (all threads get the
// same value; the summation order is fixed).
template <bool ONE_WARP>
__device__ __forceinline__ float block_sum(float v, float* scratch) {
    v = warp_sum(v);
    if (ONE_WARP) return v;
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[warp] = v;
    __syncthreads();
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += scratch[w];
    return s;
}
template <bool ONE_WARP>
__device__ __forceinline__ float block_max(float v, float* scratch) {
    v = warp_max(v);
    if (ONE_WARP) return v;
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) scratch[warp] = v;
    __syncthreads();
    float s = -INFINITY;
    for (int w = 0; w < nw; ++w) s = fmaxf(s, scratch[w]);
    return s;
}

// NB channel blocks of 4 per thread; ONE_WARP: the CTA is a single warp and
// all reductions are shuffles.  Otherwise blockDim.x <= 256.
// ANTI: antithetic pairs.  Every draw's noise a is used twice, as +a and -a;
// the pair's centred decrease is c = -(dl(+a) - dl(-a)) / 2, so
//   g_t = (1/(2 K sigma)) sum_i (dl_i(+a) - dl_i(-a)) a_i
// needs neither the mean over draws nor the sum of the noise (S0).
// CH: one vocabulary chunk per launch (see HeadArgs).
template <int NB, bool ONE_WARP, bool ANTI, bool CH = false>
__global__ void __launch_bounds__(ONE_WARP ? 32 : 256)
    head_draws_kernel(const HeadArgs A, const PhiloxKeys keys) {
    __shared__ float red[2][8];
    __shared__ float red_m[2][8];
    __shared__ float red_y[2];
    __shared__ float scratch[8];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int NT = ONE_WARP ? 32 : static_cast<int>(blockDim.x);
    if (!ONE_WARP && tid < 16) {  // slots of absent warps
        red[tid >> 3][tid & 7] = 0.f;
        red_m[tid >> 3][tid & 7] = 0.f;
    }
    const int t = blockIdx.x / A.Q;
    const int q = blockIdx.x - t * A.Q;
    const int i_begin = q * A.chunk;
    const int i_end = min(A.K, i_begin + A.chunk);
    const int V = A.V;
    const bool vec = (V & 3) == 0;
    const int64_t zbase = static_cast<int64_t>(t) * (CH ? A.ldz : V) + (CH ? A.col0 : 0);
    const int64_t zext = static_cast<int64_t>(A.T) * (CH ? A.ldz : V);  // logits, g_hat extent
    const float* zrow = A.logits + zbase;

    // Cached logits of this token -> registers; softmax.
    float p[NB][4];
    float zmax = -INFINITY;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int j = b * NT + tid;
        if (vec && j < A.nblk && DUST_IB(zbase + 4 * j + 3, zext)) {
            const float4 z4 = __ldg(reinterpret_cast<const float4*>(zrow) + j);
            p[b][0] = z4.x; p[b][1] = z4.y; p[b][2] = z4.z; p[b][3] = z4.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = 4 * j + k;
                p[b][k] = (j < A.nblk && c < V && DUST_IB(zbase + c, zext)) ? __ldg(zrow + c)
                                                                            : -INFINITY;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) zmax = fmaxf(zmax, p[b][k]);
    }
    float unpert = 0.f;  // CH: the probability mass outside the chunk
    if (CH) {
        const float lse = DUST_IB(t, A.T) ? __ldg(A.lse + t) : 0.f;
        float pc = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                p[b][k] = (p[b][k] == -INFINITY) ? 0.f : expf(p[b][k] - lse);
                pc += p[b][k];
            }
        unpert = 1.0f - block_sum<ONE_WARP>(pc, scratch);
    } else {
        zmax = block_max<ONE_WARP>(zmax, scratch);
        float zsum = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                p[b][k] = (p[b][k] == -INFINITY) ? 0.f : expf(p[b][k] - zmax);
                zsum += p[b][k];
            }
        zsum = block_sum<ONE_WARP>(zsum, scratch);
        const float zinv = 1.0f / zsum;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k) p[b][k] *= zinv;
    }

    // Target channel: the thread that owns it supplies sigma a_y every draw
    // (in chunk mode only when the target lies in the chunk).
    int y = DUST_IB(t, A.T) ? __ldg(A.targets + t) : -1;
    if (y < 0 || y >= (CH ? A.Vfull : V)) {
        if (tid == 0 && q == 0) record_status(A.status, DUST_ERR_DEVICE_RANGE);
        y = -1;
    } else if (CH) {
        y -= A.col0;
        if (y < 0 || y >= V) y = -1;
    }
    const int yblk = y >> 2;
    const bool owner = (y >= 0) && (yblk % NT == tid);
    const int yb = (y >= 0) ? yblk / NT : 0;
    const int yc = y & 3;
    const int ylane = (y >= 0) ? (yblk % NT) & 31 : 0;
    const bool ywarp = (y >= 0) && (((yblk % NT) >> 5) == warp);

    BlockHalf bh[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)  // global channel blocks (the chunk's offset in chunk mode)
        bh[b] = philox_block_half((CH ? A.col0 / 4 : 0) + b * NT + tid, A.layer, keys);

    float s1[NB][4], s0[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) s1[b][k] = s0[b][k] = 0.f;
    float sdl = 0.f;
    const uint32_t token = A.token0 + static_cast<uint32_t>(t);

#pragma unroll 1
    for (int i = i_begin; i < i_end; ++i) {
        const DrawHalf dh = philox_draw_half(
            A.draw0 + static_cast<uint32_t>(i) * (CH ? A.draw_stride : 1u), token, keys);
        // All NB blocks advance in lockstep (words, then normals, then the
        // loss terms) so that their independent chains interleave.
        uint4 w[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) w[b] = philox_rest(dh, bh[b], keys);
        // Blocks past the vocabulary (only in the last block row) carry real
        // noise of unused counters; their probabilities are zero and their
        // accumulators are never written, so they change nothing.  a holds
        // b = s a: exp(sigma a) = 2^b, and the accumulators are rescaled once
        // at the end.
        float a[NB][4];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float4 n = words_to_normals_fast(w[b], A.clog);
            a[b][0] = n.x;
            a[b][1] = n.y;
            a[b][2] = n.z;
            a[b][3] = n.w;
        }
        float pb[NB], pm[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float q = p[b][0] * ex2_approx(a[b][0]);
            q = fmaf(p[b][1], ex2_approx(a[b][1]), q);
            q = fmaf(p[b][2], ex2_approx(a[b][2]), q);
            pb[b] = fmaf(p[b][3], ex2_approx(a[b][3]), q);
            if (ANTI) {
                float r = p[b][0] * ex2_approx(-a[b][0]);
                r = fmaf(p[b][1], ex2_approx(-a[b][1]), r);
                r = fmaf(p[b][2], ex2_approx(-a[b][2]), r);
                pm[b] = fmaf(p[b][3], ex2_approx(-a[b][3]), r);
            }
        }
        float part = pb[0], partm = ANTI ? pm[0] : 0.f;
#pragma unroll
        for (int b = 1; b < NB; ++b) {
            part += pb[b];
            if (ANTI) partm += pm[b];
        }
        float ay = 0.f;
        if (ywarp) {  // warp-uniform: only the warp that holds the target's block
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (b == yb) ay = yc == 0 ? a[b][0] : yc == 1 ? a[b][1] : yc == 2 ? a[b][2] : a[b][3];
        }
        part = warp_sum(part);
        if (ANTI) partm = warp_sum(partm);
        float S, Sm = 1.f;
        if (ONE_WARP) {
            S = CH ? part + unpert : part;
            Sm = partm;
            ay = __shfl_sync(0xFFFFFFFFu, ay, ylane);
        } else {
            const int buf = i & 1;
            if (lane == 0) {
                red[buf][warp] = part;
                if (ANTI) red_m[buf][warp] = partm;
            }
            if (owner) red_y[buf] = ay;
            __syncthreads();
            // Eight warp partials (absent warps read zero), summed by a
            // butterfly over lanes 0..7: every lane forms the same sum.
            S = red[buf][lane & 7];
            S += __shfl_xor_sync(0xFFFFFFFFu, S, 1);
            S += __shfl_xor_sync(0xFFFFFFFFu, S, 2);
            S += __shfl_xor_sync(0xFFFFFFFFu, S, 4);
            if (CH) S += unpert;
            if (ANTI) {
                Sm = red_m[buf][lane & 7];
                Sm += __shfl_xor_sync(0xFFFFFFFFu, Sm, 1);
                Sm += __shfl_xor_sync(0xFFFFFFFFu, Sm, 2);
                Sm += __shfl_xor_sync(0xFFFFFFFFu, Sm, 4);
            }
            ay = (y >= 0) ? red_y[buf] : 0.f;
        }
        if (ANTI) {
            // dl(+a) - dl(-a) = ln S+ - ln S- - 2 sigma a_y, sigma a_y = b_y ln 2.
            const float dd = fmaf(ay, -1.3862943611198906f, log_pos(S) - log_pos(Sm));
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k) s1[b][k] = fmaf(dd, a[b][k], s1[b][k]);
        } else {
            // sigma a_y = b_y ln 2.
            const float dl = fmaf(ay, -0.69314718055994531f, log_pos(S));
            sdl += dl;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    s1[b][k] = fmaf(dl, a[b][k], s1[b][k]);
                    s0[b][k] += a[b][k];
                }
        }
    }

    if (A.Q == 1) {
        const float mean = sdl / static_cast<float>(A.K);
        float* grow = A.g_hat ? A.g_hat + static_cast<int64_t>(t) * (CH ? A.ldz : V) +
                                    (CH ? A.col0 : 0)
                              : nullptr;
        __nv_bfloat16* brow = A.gbf + static_cast<int64_t>(t) * A.ldg + (CH ? A.col0 : 0);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int j = b * NT + tid;
            if (j >= A.nblk) continue;
            float g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) g[k] = (s1[b][k] - mean * s0[b][k]) * A.g_scale;
            if (vec) {
                if (grow && DUST_IB(zbase + 4 * j + 3, zext))
                    *reinterpret_cast<float4*>(grow + 4 * j) = make_float4(g[0], g[1], g[2], g[3]);
                __nv_bfloat162 lo = __floats2bfloat162_rn(g[0], g[1]);
                __nv_bfloat162 hi = __floats2bfloat162_rn(g[2], g[3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&lo);
                pk.y = *reinterpret_cast<uint32_t*>(&hi);
                if (DUST_IB((brow - A.gbf) + 4 * j + 3, static_cast<int64_t>(A.T) * A.ldg))
                    *reinterpret_cast<uint2*>(brow + 4 * j) = pk;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = 4 * j + k;
                    if (c < V) {
                        if (grow && DUST_IB(zbase + c, zext)) grow[c] = g[k];
                        if (DUST_IB((brow - A.gbf) + c, static_cast<int64_t>(A.T) * A.ldg))
                            brow[c] = __float2bfloat16_rn(g[k]);
                    }
                }
            }
        }
    } else {
        const int64_t off = (static_cast<int64_t>(q) * A.T + t) * (CH ? A.ldz : V) + (CH ? A.col0 : 0);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int j = b * NT + tid;
            if (j >= A.nblk) continue;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = 4 * j + k;
                if (c < V && DUST_IB(off + c, static_cast<int64_t>(A.Q) * zext)) {
                    A.part_s1[off + c] = s1[b][k];
                    A.part_s0[off + c] = s0[b][k];
                }
            }
        }
        if (tid == 0 && DUST_IB(static_cast<int64_t>(q) * A.T + t, static_cast<int64_t>(A.Q) * A.T))
            A.part_dl[static_cast<int64_t>(q) * A.T + t] = sdl;
    }
}

// Sums the draw-chunk partials in chunk order and forms g (fp32 + bf16 copy).
// (Columns col0 .. col0 + V - 1 of rows ldz apart, as the draws kernel.)
__global__ void head_finalize_kernel(const HeadArgs A) {
    const int t = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= A.V) return;
    float sdl = 0.f, s1 = 0.f, s0 = 0.f;
    for (int q = 0; q < A.Q; ++q) {
        const int64_t off = (static_cast<int64_t>(q) * A.T + t) * A.ldz + A.col0 + c;
        if (!DUST_IB(off, static_cast<int64_t>(A.Q) * A.T * A.ldz) ||
            !DUST_IB(static_cast<int64_t>(q) * A.T + t, static_cast<int64_t>(A.Q) * A.T))
            continue;
        sdl += A.part_dl[static_cast<int64_t>(q) * A.T + t];
        s1 += A.part_s1[off];
        s0 += A.part_s0[off];
    }
    const float mean = sdl / static_cast<float>(A.K);
    const float g = (s1 - mean * s0) * A.g_scale;
    const int64_t gi = static_cast<int64_t>(t) * A.ldz + A.col0 + c;
    if (A.g_hat && DUST_IB(gi, static_cast<int64_t>(A.T) * A.ldz)) A.g_hat[gi] = g;
    const int64_t bi = static_cast<int64_t>(t) * A.ldg + A.col0 + c;
    if (DUST_IB(bi, static_cast<int64_t>(A.T) * A.ldg)) A.gbf[bi] = __float2bfloat16_rn(g);
}

// The mean-baseline draws, two per pass (leave-one-out is the same kernel
// with another final scale).
//
// The token's probabilities live in shared memory, not registers, and every
// pass over the thread's channel blocks generates two draws' noise block by
// block: the two Philox chains of a block interleave, and the block's two
// noise vectors (b = s a) go to shared memory, where the accumulation after
// the reduction reads them back.  That leaves the S1/S0 accumulators and the
// working set in 128 registers, so four 128-thread CTAs share an SM, and
// halves the CTA reductions and barriers per draw.  The two sums
// sum_v p_v 2^b_v are reduced across the CTA in fixed point, as exact 32-bit
// integer sums (redux.sync per warp, one shared-memory add per warp), so
// their value does not depend on the order of the adds: qscale = 2^E with
// E chosen on the host so that the largest possible sum, 2^(5.8 s), stays
// below 2^32.  When sigma is too large for 24 fractional bits the sums are
// floats added in warp order instead.  The loss change is
// ln S - b_y ln 2, with the hardware log2 for ln S (absolute error about
// 1.7e-7, against loss changes of order sigma).
//
// Dynamic shared memory: NB x NT float4 of probabilities, then 2 x NB x NT
// float4 of noise.
// NTC: the CTA's thread count when it is fixed at compile time (32 for
// one-warp CTAs, 256 for vocabularies of 3073 to 4096 entries), else 0
// (blockDim.x, up to 256): constant strides keep the shared-memory
// addressing off the integer multiplier that Philox saturates.  With 256
// threads four CTAs fit an SM (64 registers, 48 KB of shared memory each),
// 32 warps.
// FIXED: the sums are reduced in fixed point (qscale > 0), else as floats.
template <int NB, bool ONE_WARP, int NTC, bool FIXED>
__global__ void __launch_bounds__(NTC == 0 ? 256 : NTC, NTC == 32 ? 16 : (NTC == 256 ? 4 : 2))
    head_pair_kernel(const HeadArgs A, const PhiloxKeys keys) {
    extern __shared__ float4 pair_smem[];
    __shared__ uint32_t qsum[3][2];   // fixed-point sums, three rotating slots
    __shared__ float fsum[2][2][8];   // float sums per warp, two slots
    __shared__ float red_y[2][2];     // b of the target channel, per draw
    __shared__ float scratch[8];

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int NT = ONE_WARP ? 32 : (NTC > 0 ? NTC : static_cast<int>(blockDim.x));
    const int NW = NT >> 5;
    float4* psm = pair_smem;
    float4* nsm = pair_smem + NB * NT;  // [draw of the pair][block][thread]
    if (tid < 6) qsum[tid >> 1][tid & 1] = 0u;
    const int t = blockIdx.x / A.Q;
    const int q = blockIdx.x - t * A.Q;
    const int i_begin = q * A.chunk;
    const int i_end = min(A.K, i_begin + A.chunk);
    const int V = A.V;
    const bool vec = (V & 3) == 0;
    const int64_t zbase = static_cast<int64_t>(t) * V;
    const int64_t zext = static_cast<int64_t>(A.T) * V;  // logits, g_hat extent
    const float* zrow = A.logits + zbase;

    // Cached logits of this token -> softmax -> shared memory.
    float p[NB][4];
    float zmax = -INFINITY;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int j = b * NT + tid;
        if (vec && j < A.nblk && DUST_IB(zbase + 4 * j + 3, zext)) {
            const float4 z4 = __ldg(reinterpret_cast<const float4*>(zrow) + j);
            p[b][0] = z4.x; p[b][1] = z4.y; p[b][2] = z4.z; p[b][3] = z4.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = 4 * j + k;
                p[b][k] = (j < A.nblk && c < V && DUST_IB(zbase + c, zext)) ? __ldg(zrow + c)
                                                                            : -INFINITY;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) zmax = fmaxf(zmax, p[b][k]);
    }
    zmax = block_max<ONE_WARP>(zmax, scratch);
    float zsum = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            p[b][k] = (p[b][k] == -INFINITY) ? 0.f : expf(p[b][k] - zmax);
            zsum += p[b][k];
        }
    zsum = block_sum<ONE_WARP>(zsum, scratch);
    const float zinv = 1.0f / zsum;
#pragma unroll
    for (int b = 0; b < NB; ++b)
        psm[b * NT + tid] = make_float4(p[b][0] * zinv, p[b][1] * zinv, p[b][2] * zinv,
                                        p[b][3] * zinv);

    int y = DUST_IB(t, A.T) ? __ldg(A.targets + t) : -1;
    if (y < 0 || y >= V) {
        if (tid == 0 && q == 0) record_status(A.status, DUST_ERR_DEVICE_RANGE);
        y = -1;
    }
    const int yblk = y >> 2;
    const bool owner = (y >= 0) && (yblk % NT == tid);
    const int yb = (y >= 0) ? yblk / NT : -1;
    const int yc = y & 3;
    const int ylane = (y >= 0) ? (yblk % NT) & 31 : 0;
    const bool ywarp = (y >= 0) && (((yblk % NT) >> 5) == warp);

    float s1[NB][4], s0[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) s1[b][k] = s0[b][k] = 0.f;
    float sdl = 0.f;
    const uint32_t token = A.token0 + static_cast<uint32_t>(t);
    constexpr bool fixed = FIXED;
    if (!ONE_WARP) __syncthreads();  // qsum zeroed before the first pass adds to it

    int pass = 0;
#pragma unroll 1
    for (int i = i_begin; i < i_end; i += 2, ++pass) {
        // The second draw of an odd count's last pass is generated but not
        // counted (w1 = 0).
        const float w1 = (i + 1 < i_end) ? 1.f : 0.f;
        const DrawHalf2 dh0 =
            philox_draw_half2(philox_draw_half(A.draw0 + static_cast<uint32_t>(i), token, keys));
        const DrawHalf2 dh1 =
            philox_draw_half2(philox_draw_half(A.draw0 + static_cast<uint32_t>(i + 1), token, keys));
        float ay0 = 0.f, ay1 = 0.f;
        // sum_v p_v 2^b_v of each draw as two interleaved partial sums (even
        // and odd channels of the thread's blocks), on packed pairs
        float2 pe0 = make_float2(0.f, 0.f), pe1 = pe0;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            // Blocks past the vocabulary (only in the last block row) carry
            // real noise of unused counters; their probabilities are zero and
            // their accumulators are never written.
            const BlockHalf2 hb = philox_block_half2(philox_block_half(b * NT + tid, A.layer, keys), keys);
            const uint4 wd0 = philox_rest2(dh0, hb, keys);
            const uint4 wd1 = philox_rest2(dh1, hb, keys);
            const float4 n0 = words_to_normals_fast(wd0, A.clog);
            const float4 n1 = words_to_normals_fast(wd1, A.clog);
            const float4 pb = psm[b * NT + tid];
            const float2 plo = make_float2(pb.x, pb.y), phi = make_float2(pb.z, pb.w);
            pe0 = fma2(plo, make_float2(ex2_approx(n0.x), ex2_approx(n0.y)), pe0);
            pe0 = fma2(phi, make_float2(ex2_approx(n0.z), ex2_approx(n0.w)), pe0);
            pe1 = fma2(plo, make_float2(ex2_approx(n1.x), ex2_approx(n1.y)), pe1);
            pe1 = fma2(phi, make_float2(ex2_approx(n1.z), ex2_approx(n1.w)), pe1);
            nsm[b * NT + tid] = n0;
            nsm[(NB + b) * NT + tid] = n1;
            if (ywarp && b == yb) {  // warp-uniform
                ay0 = yc == 0 ? n0.x : yc == 1 ? n0.y : yc == 2 ? n0.z : n0.w;
                ay1 = yc == 0 ? n1.x : yc == 1 ? n1.y : yc == 2 ? n1.z : n1.w;
            }
        }
        const float pt0 = pe0.x + pe0.y, pt1 = pe1.x + pe1.y;
        const int slot = pass % 3, buf = pass & 1;
        float S0, S1;
        if (fixed) {
            const uint32_t q0 = __float2uint_rn(pt0 * A.qscale);
            const uint32_t q1 = __float2uint_rn(pt1 * A.qscale);
            uint32_t r0, r1;
            asm volatile("redux.sync.add.u32 %0, %1, 0xffffffff;" : "=r"(r0) : "r"(q0));
            asm volatile("redux.sync.add.u32 %0, %1, 0xffffffff;" : "=r"(r1) : "r"(q1));
            if (ONE_WARP) {
                S0 = static_cast<float>(r0) * A.qinv;
                S1 = static_cast<float>(r1) * A.qinv;
            } else if (lane == 0) {
                atomicAdd(&qsum[slot][0], r0);
                atomicAdd(&qsum[slot][1], r1);
            }
        } else {
            const float f0 = warp_sum(pt0), f1 = warp_sum(pt1);
            if (ONE_WARP) {
                S0 = f0;
                S1 = f1;
            } else if (lane == 0) {
                fsum[buf][0][warp] = f0;
                fsum[buf][1][warp] = f1;
            }
        }
        if (ONE_WARP) {
            ay0 = __shfl_sync(0xFFFFFFFFu, ay0, ylane);
            ay1 = __shfl_sync(0xFFFFFFFFu, ay1, ylane);
        } else {
            if (owner) {
                red_y[buf][0] = ay0;
                red_y[buf][1] = ay1;
            }
            __syncthreads();
            if (fixed) {
                S0 = static_cast<float>(qsum[slot][0]) * A.qinv;
                S1 = static_cast<float>(qsum[slot][1]) * A.qinv;
                // the slot read two passes ago is free again (every thread
                // has passed this pass's barrier since reading it)
                if (tid < 2) qsum[(pass + 2) % 3][tid] = 0u;
            } else {
                S0 = fsum[buf][0][0];
                S1 = fsum[buf][1][0];
                for (int w2 = 1; w2 < NW; ++w2) {
                    S0 += fsum[buf][0][w2];
                    S1 += fsum[buf][1][w2];
                }
            }
            ay0 = y >= 0 ? red_y[buf][0] : 0.f;
            ay1 = y >= 0 ? red_y[buf][1] : 0.f;
        }
        // dl = ln S - sigma a_y, with sigma a_y = b_y ln 2.
        const float dl0 = (lg2_approx(S0) - ay0) * 0.69314718055994531f;
        const float dl1 = (lg2_approx(S1) - ay1) * 0.69314718055994531f * w1;
        sdl += dl0 + dl1;
        const float2 d0 = make_float2(dl0, dl0), d1 = make_float2(dl1, dl1);
        const float2 ww = make_float2(w1, w1);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float4 n0 = nsm[b * NT + tid];
            const float4 n1 = nsm[(NB + b) * NT + tid];
            // s1 += dl0 n0 + dl1 n1; s0 += n0 + w1 n1, channel pairs (0, 1), (2, 3)
            float2 u = fma2(d1, make_float2(n1.x, n1.y),
                            fma2(d0, make_float2(n0.x, n0.y), make_float2(s1[b][0], s1[b][1])));
            float2 v = fma2(d1, make_float2(n1.z, n1.w),
                            fma2(d0, make_float2(n0.z, n0.w), make_float2(s1[b][2], s1[b][3])));
            s1[b][0] = u.x; s1[b][1] = u.y; s1[b][2] = v.x; s1[b][3] = v.y;
            u = fma2(make_float2(n1.x, n1.y), ww,
                     add2(make_float2(s0[b][0], s0[b][1]), make_float2(n0.x, n0.y)));
            v = fma2(make_float2(n1.z, n1.w), ww,
                     add2(make_float2(s0[b][2], s0[b][3]), make_float2(n0.z, n0.w)));
            s0[b][0] = u.x; s0[b][1] = u.y; s0[b][2] = v.x; s0[b][3] = v.y;
        }
    }

    if (A.Q == 1) {
        const float mean = sdl / static_cast<float>(A.K);
        float* grow = A.g_hat ? A.g_hat + static_cast<int64_t>(t) * V : nullptr;
        __nv_bfloat16* brow = A.gbf + static_cast<int64_t>(t) * A.ldg;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int j = b * NT + tid;
            if (j >= A.nblk) continue;
            float g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) g[k] = (s1[b][k] - mean * s0[b][k]) * A.g_scale;
            if (vec) {
                if (grow && DUST_IB(zbase + 4 * j + 3, zext))
                    *reinterpret_cast<float4*>(grow + 4 * j) = make_float4(g[0], g[1], g[2], g[3]);
                __nv_bfloat162 lo = __floats2bfloat162_rn(g[0], g[1]);
                __nv_bfloat162 hi = __floats2bfloat162_rn(g[2], g[3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&lo);
                pk.y = *reinterpret_cast<uint32_t*>(&hi);
                if (DUST_IB((brow - A.gbf) + 4 * j + 3, static_cast<int64_t>(A.T) * A.ldg))
                    *reinterpret_cast<uint2*>(brow + 4 * j) = pk;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = 4 * j + k;
                    if (c < V) {
                        if (grow && DUST_IB(zbase + c, zext)) grow[c] = g[k];
                        if (DUST_IB((brow - A.gbf) + c, static_cast<int64_t>(A.T) * A.ldg))
                            brow[c] = __float2bfloat16_rn(g[k]);
                    }
                }
            }
        }
    } else {
        const int64_t off = (static_cast<int64_t>(q) * A.T + t) * V;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int j = b * NT + tid;
            if (j >= A.nblk) continue;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = 4 * j + k;
                if (c < V && DUST_IB(off + c, static_cast<int64_t>(A.Q) * zext)) {
                    A.part_s1[off + c] = s1[b][k];
                    A.part_s0[off + c] = s0[b][k];
                }
            }
        }
        if (tid == 0 && DUST_IB(static_cast<int64_t>(q) * A.T + t, static_cast<int64_t>(A.Q) * A.T))
            A.part_dl[static_cast<int64_t>(q) * A.T + t] = sdl;
    }
}

struct HeadPlan {
    int nblk, nb, nt, Q, chunk;
    bool one_warp;
    int64_t ldg, ldx;
    size_t ws_bytes;
    size_t off_gbf, off_xbf, off_s1, off_s0, off_dl;
};

constexpr int64_t kMaxV = 8192;

HeadPlan head_plan(int64_t T, int64_t V, int64_t d, uint32_t K) {
    HeadPlan P{};
    P.nblk = static_cast<int>(ceil_div(V, 4));
    if (P.nblk <= 32 * 8) {
        P.one_warp = true;
        P.nt = 32;
        const int need = static_cast<int>(ceil_div(P.nblk, 32));
        P.nb = need <= 1 ? 1 : need <= 2 ? 2 : need <= 4 ? 4 : 8;
    } else {
        P.one_warp = false;
        // 8 channel blocks per thread: half the per-element share of each
        // draw's CTA reduction and log, at 12 resident warps per SM
        // (4.79 against 4.84 ms with 4 blocks at 16384 x 4096, K 64)
        P.nb = 8;
        P.nt = static_cast<int>(round_up(ceil_div(P.nblk, P.nb), 32));
    }
    // Split the draws when there are too few tokens to fill 148 SMs.
    const int64_t target = P.one_warp ? 148 * 48 : 148 * 8;
    int64_t Q = 1;
    if (T < target) {
        Q = ceil_div(target, T);
        const int64_t qmax = K / 16 > 1 ? K / 16 : 1;
        if (Q > qmax) Q = qmax;
    }
    P.chunk = static_cast<int>(ceil_div(K, Q));
    P.Q = static_cast<int>(ceil_div(K, P.chunk));
    P.ldg = round_up(V, 8);
    P.ldx = round_up(d, 8);
    WsLayout w;
    w.take(kCtlBytes);
    P.off_gbf = w.take(static_cast<size_t>(T * P.ldg) * 2);
    P.off_xbf = w.take(static_cast<size_t>(T * P.ldx) * 2);
    if (P.Q > 1) {
        const size_t n = static_cast<size_t>(P.Q) * T * V;
        P.off_s1 = w.take(n * 4);
        P.off_s0 = w.take(n * 4);
        P.off_dl = w.take(static_cast<size_t>(P.Q) * T * 4);
    }
    P.ws_bytes = w.used;
    return P;
}

// The fast Box-Muller's log constant for b = s a, and the pair kernel's
// fixed-point scale: |a| < 5.8 by construction (u >= 2^-24), so every sum
// sum_v p_v 2^b_v (the p sum to 1) is below 2^(5.8 s); 2^E keeps it, and the
// lanes' rounding, below 2^32.  Below 24 fractional bits the kernel adds
// floats instead (qscale = 0).
void set_noise_scales(HeadArgs& A, double s) {
    A.clog = static_cast<float>(-2.0 * 0.69314718055994531 * s * s);
    const int E = static_cast<int>(std::floor(31.9 - 5.8 * s));
    if (E >= 24) {
        A.qscale = std::ldexp(1.0f, E);
        A.qinv = std::ldexp(1.0f, -E);
    } else {
        A.qscale = 0.f;
        A.qinv = 0.f;
    }
}

size_t pair_smem_bytes(int nb, int nt) { return static_cast<size_t>(3) * nb * nt * 16; }

template <int NB, bool OW, int NTC, bool FIXED>
dust_status launch_pairs_as(const HeadPlan& P, const HeadArgs& A, const PhiloxKeys& keys,
                            int64_t T, cudaStream_t s) {
    static std::atomic<uint64_t> smem_set{0};
    // the kernel's largest dynamic shared memory (up to 256 threads when NTC = 0)
    const size_t smem_max = pair_smem_bytes(NB, NTC == 0 ? 256 : NTC);
    const size_t smem = pair_smem_bytes(NB, P.nt);
    DUST_CUDA_TRY(set_smem_once(head_pair_kernel<NB, OW, NTC, FIXED>, static_cast<int>(smem_max),
                                smem_set));
    timer_begin(s);
    head_pair_kernel<NB, OW, NTC, FIXED><<<static_cast<unsigned>(T * P.Q), P.nt, smem, s>>>(A,
                                                                                           keys);
    timer_end(s);
    return launch_status();
}

template <int NB, bool OW, int NTC>
dust_status launch_pairs(const HeadPlan& P, const HeadArgs& A, const PhiloxKeys& keys, int64_t T,
                         cudaStream_t s) {
    return A.qscale > 0.f ? launch_pairs_as<NB, OW, NTC, true>(P, A, keys, T, s)
                          : launch_pairs_as<NB, OW, NTC, false>(P, A, keys, T, s);
}

template <int NB, bool OW>
dust_status launch_draws(const HeadPlan& P, const HeadArgs& A, const PhiloxKeys& keys,
                         int64_t T, bool anti, cudaStream_t s, bool chunk = false) {
    timer_begin(s);
    const unsigned grid = static_cast<unsigned>(T * P.Q);
    if (chunk)
        head_draws_kernel<NB, OW, false, true><<<grid, P.nt, 0, s>>>(A, keys);
    else if (anti)
        head_draws_kernel<NB, OW, true><<<grid, P.nt, 0, s>>>(A, keys);
    else
        head_draws_kernel<NB, OW, false><<<grid, P.nt, 0, s>>>(A, keys);
    timer_end(s);
    return launch_status();
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" size_t dust_head_workspace(int64_t T, int64_t V, int64_t d, uint32_t K) {
    if (T < 1 || V < 1 || d < 1 || K < 2) return 0;
    return head_plan(T, V, d, K).ws_bytes;
}

namespace dust {

dust_status head_estimate_check(const float* logits, const int32_t* targets, const void* x,
                                dust_dtype x_dtype, int64_t T, int64_t V, int64_t d,
                                const dust_noise& nz, dust_baseline baseline, const float* g_hat,
                                const float* G_W, const void* ws, size_t ws_bytes) {
    if (!logits || !targets || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (baseline != DUST_BASELINE_MEAN && baseline != DUST_BASELINE_LEAVE_ONE_OUT &&
        baseline != DUST_BASELINE_ANTITHETIC)
        return DUST_ERR_INVALID_ARG;
    if (T < 1 || V < 1 || d < 1 || nz.num_draws < 2) return DUST_ERR_INVALID_ARG;
    if (!(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (V > kMaxV || T > (1LL << 30) || d > (1LL << 30) || nz.num_draws > (1u << 30))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32)) return DUST_ERR_INVALID_ARG;
    if ((V % 4 == 0) && (!aligned(logits, 16) || (g_hat && !aligned(g_hat, 16))))
        return DUST_ERR_INVALID_ARG;
    const HeadPlan P = head_plan(T, V, d, nz.num_draws);
    if (!ws || ws_bytes < P.ws_bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

}  // namespace dust

namespace {

dust_status head_estimate(const float* logits, const int32_t* targets, const void* x,
                          dust_dtype x_dtype, int64_t T, int64_t V, int64_t d, dust_noise nz,
                          dust_baseline baseline, float* g_hat, float* G_W, void* ws,
                          size_t ws_bytes, void* stream) {
    const dust_status chk = head_estimate_check(logits, targets, x, x_dtype, T, V, d, nz,
                                                baseline, g_hat, G_W, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const HeadPlan P = head_plan(T, V, d, nz.num_draws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));

    HeadArgs A{};
    A.logits = logits;
    A.targets = targets;
    A.T = static_cast<int>(T);
    A.V = static_cast<int>(V);
    A.nblk = P.nblk;
    A.K = static_cast<int>(nz.num_draws);
    A.Q = P.Q;
    A.chunk = P.chunk;
    A.draw0 = nz.draw0;
    A.token0 = nz.token0;
    A.layer = nz.layer;
    const double s_l2e = static_cast<double>(nz.sigma) * 1.4426950408889634;
    A.sig_l2e = static_cast<float>(s_l2e);
    set_noise_scales(A, s_l2e);
    // g = (S1 - m S0) / (K sigma s) for the mean over draws; leave-one-out
    // means scale it by K / (K - 1); antithetic pairs give S1 / (2 K sigma s).
    const double ks = static_cast<double>(nz.sigma) * static_cast<double>(A.sig_l2e);
    const double K = static_cast<double>(nz.num_draws);
    A.g_scale = static_cast<float>(baseline == DUST_BASELINE_LEAVE_ONE_OUT ? 1.0 / ((K - 1.0) * ks)
                                   : baseline == DUST_BASELINE_ANTITHETIC  ? 1.0 / (2.0 * K * ks)
                                                                           : 1.0 / (K * ks));
    const bool anti = baseline == DUST_BASELINE_ANTITHETIC;
    A.g_hat = g_hat;
    A.gbf = reinterpret_cast<__nv_bfloat16*>(w + P.off_gbf);
    A.ldg = P.ldg;
    A.status = static_cast<uint32_t*>(ws);
    A.ldz = V;
    A.col0 = 0;
    A.Vfull = static_cast<int>(V);
    A.draw_stride = 1;
    if (P.Q > 1) {
        A.part_s1 = reinterpret_cast<float*>(w + P.off_s1);
        A.part_s0 = reinterpret_cast<float*>(w + P.off_s0);
        A.part_dl = reinterpret_cast<float*>(w + P.off_dl);
    }
    const PhiloxKeys keys = philox_round_keys(nz.seed);

    dust_status st;
    if (anti) {
        if (P.one_warp) {
            switch (P.nb) {
                case 1: st = launch_draws<1, true>(P, A, keys, T, true, s); break;
                case 2: st = launch_draws<2, true>(P, A, keys, T, true, s); break;
                case 4: st = launch_draws<4, true>(P, A, keys, T, true, s); break;
                default: st = launch_draws<8, true>(P, A, keys, T, true, s); break;
            }
        } else {
            st = launch_draws<8, false>(P, A, keys, T, true, s);  // head_plan: 8 blocks per thread
        }
    } else if (P.one_warp) {
        switch (P.nb) {
            case 1: st = launch_pairs<1, true, 32>(P, A, keys, T, s); break;
            case 2: st = launch_pairs<2, true, 32>(P, A, keys, T, s); break;
            case 4: st = launch_pairs<4, true, 32>(P, A, keys, T, s); break;
            default: st = launch_pairs<8, true, 32>(P, A, keys, T, s); break;
        }
    } else if (P.nt == 128) {
        // 4 blocks per thread at 256 threads instead of 8 at 128: the same
        // columns per CTA at twice the resident warps (3.96 against 3.98 ms
        // per call at 16384 x 4096, K 64)
        HeadPlan P4 = P;
        P4.nb = 4;
        P4.nt = 256;
        st = launch_pairs<4, false, 256>(P4, A, keys, T, s);
    } else {
        st = launch_pairs<8, false, 0>(P, A, keys, T, s);
    }
    if (st != DUST_OK) return st;
    if (P.Q > 1) {
        dim3 grid(static_cast<unsigned>(ceil_div(V, 128)), static_cast<unsigned>(T));
        head_finalize_kernel<<<grid, 128, 0, s>>>(A);
        if ((st = launch_status()) != DUST_OK) return st;
    }

    // x -> bf16 in a padded layout when needed, then G_W = g^T x.
    const void* xb = x;
    int64_t ldx = d;
    if (x_dtype == DUST_F32 || (d % 8) != 0 || !aligned(x, 16)) {
        void* xbf = w + P.off_xbf;
        st = x_dtype == DUST_F32
                 ? f32_to_bf16_launch(static_cast<const float*>(x), T, d, d, xbf, P.ldx, s)
                 : bf16_pad_launch(x, T, d, d, xbf, P.ldx, s);
        if (st != DUST_OK) return st;
        xb = xbf;
        ldx = P.ldx;
    }
    return gemm_bf16_launch(A.gbf, true, P.ldg, xb, true, ldx, V, d, T, 0, 1, G_W, d,
                            static_cast<uint32_t*>(ws), s);
}

}  // namespace

extern "C" dust_status dust_head_estimate(const float* logits, const int32_t* targets,
                                          const void* x, dust_dtype x_dtype, int64_t T,
                                          int64_t V, int64_t d, dust_noise nz, float* g_hat,
                                          float* G_W, void* ws, size_t ws_bytes, void* stream) {
    return head_estimate(logits, targets, x, x_dtype, T, V, d, nz, DUST_BASELINE_MEAN, g_hat,
                         G_W, ws, ws_bytes, stream);
}

extern "C" dust_status dust_head_estimate_baseline(const float* logits, const int32_t* targets,
                                                   const void* x, dust_dtype x_dtype, int64_t T,
                                                   int64_t V, int64_t d, dust_noise nz,
                                                   dust_baseline baseline, float* g_hat,
                                                   float* G_W, void* ws, size_t ws_bytes,
                                                   void* stream) {
    return head_estimate(logits, targets, x, x_dtype, T, V, d, nz, baseline, g_hat, G_W, ws,
                         ws_bytes, stream);
}

// ------------------------------------------------------------------------
// The exact head gradient, the backprop reference that the pages compare the
// estimate with (single-batch cosine with backprop as a tuning objective,
// Dust translation §2.3; cosine against backprop, §4.2):
//   g_t = softmax(z_t) - e_{y_t},   G = sum_t g_t x_t^T.
// ------------------------------------------------------------------------
namespace dust {
namespace {

// One CTA per token: the row's max and exp-sum by block reductions, then
// p - onehot written as fp32 (optional) and as the bf16 GEMM operand.
__global__ void __launch_bounds__(256)
    head_grad_rows_kernel(const float* __restrict__ logits, const int32_t* __restrict__ targets,
                          int V, float* __restrict__ g_out, __nv_bfloat16* __restrict__ gbf,
                          int64_t ldg, uint32_t* status) {
    __shared__ float scratch[8];
    const int64_t t = blockIdx.x;
    const float* zr = logits + t * V;
    float m = -INFINITY;
    for (int v = threadIdx.x; v < V; v += blockDim.x) m = fmaxf(m, zr[v]);
    m = block_max<false>(m, scratch);
    float s = 0.f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(zr[v] - m);
    s = block_sum<false>(s, scratch);
    const float inv = 1.0f / s;
    int y = targets[t];
    if (y < 0 || y >= V) {
        if (threadIdx.x == 0) record_status(status, DUST_ERR_DEVICE_RANGE);
        y = -1;
    }
    for (int v = threadIdx.x; v < V; v += blockDim.x) {
        const float g = expf(zr[v] - m) * inv - (v == y ? 1.0f : 0.0f);
        if (g_out && DUST_IB(t * V + v, static_cast<int64_t>(gridDim.x) * V)) g_out[t * V + v] = g;
        if (DUST_IB(t * ldg + v, static_cast<int64_t>(gridDim.x) * ldg))
            gbf[t * ldg + v] = __float2bfloat16_rn(g);
    }
}

struct GradPlan {
    int64_t ldg, ldx;
    size_t off_gbf, off_xbf, bytes;
};

GradPlan grad_plan(int64_t T, int64_t V, int64_t d) {
    GradPlan P{};
    P.ldg = round_up(V, 8);
    P.ldx = round_up(d, 8);
    WsLayout w;
    w.take(kCtlBytes);
    P.off_gbf = w.take(static_cast<size_t>(T * P.ldg) * 2);
    P.off_xbf = w.take(static_cast<size_t>(T * P.ldx) * 2);
    P.bytes = w.used;
    return P;
}

}  // namespace
}  // namespace dust

extern "C" size_t dust_head_backprop_workspace(int64_t T, int64_t V, int64_t d) {
    if (T < 1 || V < 1 || d < 1) return 0;
    return grad_plan(T, V, d).bytes;
}

extern "C" dust_status dust_head_backprop(const float* logits, const int32_t* targets,
                                          const void* x, dust_dtype x_dtype, int64_t T,
                                          int64_t V, int64_t d, float* g_out, float* G_W,
                                          void* ws, size_t ws_bytes, void* stream) {
    if (!logits || !targets || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || V < 1 || d < 1) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (T > (1LL << 30) || V > (1LL << 30) || d > (1LL << 30)) return DUST_ERR_UNSUPPORTED;
    const GradPlan P = grad_plan(T, V, d);
    if (!ws || ws_bytes < P.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    __nv_bfloat16* gbf = reinterpret_cast<__nv_bfloat16*>(w + P.off_gbf);
    head_grad_rows_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(
        logits, targets, static_cast<int>(V), g_out, gbf, P.ldg, static_cast<uint32_t*>(ws));
    dust_status st = launch_status();
    if (st != DUST_OK) return st;
    const void* xb = x;
    int64_t ldx = d;
    if (x_dtype == DUST_F32 || (d % 8) != 0 || !aligned(x, 16)) {
        void* xbf = w + P.off_xbf;
        st = x_dtype == DUST_F32
                 ? f32_to_bf16_launch(static_cast<const float*>(x), T, d, d, xbf, P.ldx, s)
                 : bf16_pad_launch(x, T, d, d, xbf, P.ldx, s);
        if (st != DUST_OK) return st;
        xb = xbf;
        ldx = P.ldx;
    }
    return gemm_bf16_launch(gbf, true, P.ldg, xb, true, ldx, V, d, T, 0, 1, G_W, d,
                            static_cast<uint32_t*>(ws), s);
}

// ------------------------------------------------------------------------
// The head with a vocabulary chunk perturbed per draw.  The pages' head
// perturbs the cached logits and each round recomputes the cross-entropy of
// only a small chunk of the vocabulary (laoyaoba.com, section 机制拆解).  Read
// plainly: with chunks of width w tiling the vocabulary, draw j perturbs chunk
// j mod (V/w) only, so
//   dl = log(1 + sum_{v in chunk} p_v (e^{sigma a_v} - 1)) - sigma a_y [y in chunk],
// each chunk's draws are centred by their own mean, and each chunk's columns
// of g average over that chunk's K w / V draws.  One launch per chunk.
// ------------------------------------------------------------------------
namespace dust {
namespace {

// Full-row log-sum-exp of the cached logits, one CTA per token.
__global__ void __launch_bounds__(256) row_lse_kernel(const float* __restrict__ z, int V,
                                                      float* __restrict__ lse) {
    __shared__ float scratch[8];
    const float* zr = z + static_cast<int64_t>(blockIdx.x) * V;
    float m = -INFINITY;
    for (int v = threadIdx.x; v < V; v += blockDim.x) m = fmaxf(m, zr[v]);
    m = block_max<false>(m, scratch);
    float s = 0.f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(zr[v] - m);
    s = block_sum<false>(s, scratch);
    if (threadIdx.x == 0) lse[blockIdx.x] = m + logf(s);
}

struct ChunkPlan {
    HeadPlan k;  // kernel configuration for one chunk (width w, K w / V draws)
    int64_t ldg, ldx;
    size_t off_gbf, off_xbf, off_lse, off_s1, off_s0, off_dl, bytes;
};

ChunkPlan chunk_plan(int64_t T, int64_t V, int64_t d, uint32_t K, int64_t w) {
    ChunkPlan P{};
    P.k = head_plan(T, w, d, static_cast<uint32_t>(K / (V / w)));
    P.ldg = round_up(V, 8);
    P.ldx = round_up(d, 8);
    WsLayout ws;
    ws.take(kCtlBytes);
    P.off_gbf = ws.take(static_cast<size_t>(T * P.ldg) * 2);
    P.off_xbf = ws.take(static_cast<size_t>(T * P.ldx) * 2);
    P.off_lse = ws.take(static_cast<size_t>(T) * 4);
    if (P.k.Q > 1) {
        P.off_s1 = ws.take(static_cast<size_t>(P.k.Q) * T * V * 4);
        P.off_s0 = ws.take(static_cast<size_t>(P.k.Q) * T * V * 4);
        P.off_dl = ws.take(static_cast<size_t>(P.k.Q) * T * 4);
    }
    P.bytes = ws.used;
    return P;
}

bool chunk_shape_ok(int64_t V, uint32_t K, int64_t w) {
    return w >= 4 && w % 4 == 0 && w <= kMaxV && V % w == 0 && K % (V / w) == 0 &&
           K / (V / w) >= 2;
}

}  // namespace
}  // namespace dust

extern "C" size_t dust_head_chunked_workspace(int64_t T, int64_t V, int64_t d, uint32_t K,
                                              int64_t chunk) {
    if (T < 1 || V < 1 || d < 1 || V > (1LL << 20) || !chunk_shape_ok(V, K, chunk)) return 0;
    return chunk_plan(T, V, d, K, chunk).bytes;
}

extern "C" dust_status dust_head_estimate_chunked(const float* logits, const int32_t* targets,
                                                  const void* x, dust_dtype x_dtype, int64_t T,
                                                  int64_t V, int64_t d, dust_noise nz,
                                                  int64_t chunk, float* g_hat, float* G_W,
                                                  void* ws, size_t ws_bytes, void* stream) {
    if (!logits || !targets || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || V < 1 || d < 1 || nz.num_draws < 2) return DUST_ERR_INVALID_ARG;
    if (!(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (!chunk_shape_ok(V, nz.num_draws, chunk)) return DUST_ERR_INVALID_ARG;
    if (V > (1LL << 20) || T > (1LL << 30) || d > (1LL << 30) || nz.num_draws > (1u << 30))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32)) return DUST_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || (g_hat && !aligned(g_hat, 16))) return DUST_ERR_INVALID_ARG;
    const ChunkPlan P = chunk_plan(T, V, d, nz.num_draws, chunk);
    if (!ws || ws_bytes < P.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    float* lse = reinterpret_cast<float*>(w + P.off_lse);
    row_lse_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(logits, static_cast<int>(V), lse);
    dust_status st = launch_status();
    if (st != DUST_OK) return st;

    const int nchunks = static_cast<int>(V / chunk);
    const uint32_t Kc = nz.num_draws / static_cast<uint32_t>(nchunks);
    HeadArgs A{};
    A.logits = logits;
    A.targets = targets;
    A.T = static_cast<int>(T);
    A.V = static_cast<int>(chunk);
    A.nblk = P.k.nblk;
    A.K = static_cast<int>(Kc);
    A.Q = P.k.Q;
    A.chunk = P.k.chunk;
    A.token0 = nz.token0;
    A.layer = nz.layer;
    const double s_l2e = static_cast<double>(nz.sigma) * 1.4426950408889634;
    A.sig_l2e = static_cast<float>(s_l2e);
    set_noise_scales(A, s_l2e);
    A.g_scale = static_cast<float>(
        1.0 / (static_cast<double>(Kc) * nz.sigma * static_cast<double>(A.sig_l2e)));
    A.g_hat = g_hat;
    A.gbf = reinterpret_cast<__nv_bfloat16*>(w + P.off_gbf);
    A.ldg = P.ldg;
    A.status = static_cast<uint32_t*>(ws);
    A.ldz = V;
    A.Vfull = static_cast<int>(V);
    A.draw_stride = static_cast<uint32_t>(nchunks);
    A.lse = lse;
    if (P.k.Q > 1) {
        A.part_s1 = reinterpret_cast<float*>(w + P.off_s1);
        A.part_s0 = reinterpret_cast<float*>(w + P.off_s0);
        A.part_dl = reinterpret_cast<float*>(w + P.off_dl);
    }
    const PhiloxKeys keys = philox_round_keys(nz.seed);
    for (int c = 0; c < nchunks; ++c) {
        A.col0 = static_cast<int>(c * chunk);
        A.draw0 = nz.draw0 + static_cast<uint32_t>(c);
        if (P.k.one_warp) {
            switch (P.k.nb) {
                case 1: st = launch_draws<1, true>(P.k, A, keys, T, false, s, true); break;
                case 2: st = launch_draws<2, true>(P.k, A, keys, T, false, s, true); break;
                case 4: st = launch_draws<4, true>(P.k, A, keys, T, false, s, true); break;
                default: st = launch_draws<8, true>(P.k, A, keys, T, false, s, true); break;
            }
        } else {
            st = launch_draws<8, false>(P.k, A, keys, T, false, s, true);
        }
        if (st != DUST_OK) return st;
        if (P.k.Q > 1) {
            dim3 grid(static_cast<unsigned>(ceil_div(chunk, 128)), static_cast<unsigned>(T));
            head_finalize_kernel<<<grid, 128, 0, s>>>(A);
            if ((st = launch_status()) != DUST_OK) return st;
        }
    }

    const void* xb = x;
    int64_t ldx = d;
    if (x_dtype == DUST_F32 || (d % 8) != 0 || !aligned(x, 16)) {
        void* xbf = w + P.off_xbf;
        st = x_dtype == DUST_F32
                 ? f32_to_bf16_launch(static_cast<const float*>(x), T, d, d, xbf, P.ldx, s)
                 : bf16_pad_launch(x, T, d, d, xbf, P.ldx, s);
        if (st != DUST_OK) return st;
        xb = xbf;
        ldx = P.ldx;
    }
    return gemm_bf16_launch(A.gbf, true, P.ldg, xb, true, ldx, V, d, T, 0, 1, G_W, d,
                            static_cast<uint32_t*>(ws), s);
}

namespace dust {
DUST_DEBUG_READER(1)
}  // namespace dust
