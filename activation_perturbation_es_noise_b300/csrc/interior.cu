// interior.cu -- the estimator for an interior linear layer with causal
// credit.
//
// The layer's output y1 = W1 x is perturbed per token, y1 + sigma a, and only
// the part after it is re-run from cached clean activations (laoyaoba.com
// article, section 机制拆解; Dust translation, hn.213312.xyz, §2.3).  The fixed
// downstream is GELU -> W2 -> causal per-sequence EMA -> W_head -> CE.  It is
// linear after the GELU, so a draw's logits are z_clean + dz with
//   dh = GELU(y1 + sigma a) - GELU(y1),  du = dh W2^T,
//   de_t = lam de_{t-1} + (1 - lam) du_t (per sequence),  dz = de W_head^T,
// and the loss change is dl = CE(z_clean + dz) - CE(z_clean)
//                           = log(1 + sum_v p_v expm1(dz_v)) - dz_y.
// Later tokens see earlier perturbations through the EMA, so the reward is
// the gamma-discounted suffix sum r_t = sum_{s>=t} gamma^(s-t) c_s of the
// centred loss decrease (Dust translation §2.2 信用分配), and
// g_t = -(1/(K sigma)) sum_i r_{i,t} a_{i,t}.
//
// Pipeline per chunk of nd draws (rows ordered token block of 128, draw,
// token in block, so that the draws of one token block sit next to each other
// and share its softmax rows in L2):
//   dh kernel      noise + GELU difference, split into bf16 hi and lo halves
//                  A1 = [hi | lo]  (rows x 2C)
//   GEMM 1         du = A1 [W2 | W2]^T on the tensor cores (fp32)
//   EMA kernel     de, split into A2 = [hi | lo]  (rows x 2 d_model)
//   GEMM 2 + CE    dz = A2 [W_head | W_head]^T, reduced in the epilogue to dl
// For d_model <= 512 the first three are one kernel (reforward.cu): GEMM 1
// generates A1 in shared memory and, when every sequence is whole 128-token
// blocks, runs the EMA in its epilogue and writes A2 directly.
// then once: centring, the segmented suffix scan, the noise-weighted sum for
// g (noise regenerated), and G_W1 = g^T x.
//
// The split-bf16 operands keep the re-forward within the fp32-level
// tolerance: a single bf16 rounding of dh or de perturbs the loss changes at
// the 1e-3 relative level, the hi + lo pair at about 1e-5.
#include <algorithm>

#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"
#include "gelu.cuh"

namespace dust {
namespace {

constexpr int kRowBlock = 128;


__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__device__ __forceinline__ uint2 pack4(__nv_bfloat16 a, __nv_bfloat16 b, __nv_bfloat16 c,
                                       __nv_bfloat16 d) {
    __nv_bfloat162 lo = __halves2bfloat162(a, b), hi = __halves2bfloat162(c, d);
    uint2 r;
    r.x = *reinterpret_cast<uint32_t*>(&lo);
    r.y = *reinterpret_cast<uint32_t*>(&hi);
    return r;
}

__device__ __forceinline__ int64_t chunk_row(int t, int i, int nd) {
    return (static_cast<int64_t>(t >> 7) * nd + i) * kRowBlock + (t & 127);
}

// p = softmax(z) per row, fp32, rows ldp apart (padding columns zero).
__global__ void softmax_rows_kernel(const float* __restrict__ z, int V, int ldp,
                                    float* __restrict__ p) {
    __shared__ float red[32];
    const int64_t t = blockIdx.x;
    const float* zr = z + t * V;
    float* pr = p + t * ldp;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float m = -INFINITY;
    const int64_t zext = static_cast<int64_t>(gridDim.x) * V;  // rows of z and p: gridDim.x
    for (int v = threadIdx.x; v < V; v += blockDim.x)
        if (DUST_IB(t * V + v, zext)) m = fmaxf(m, zr[v]);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = -INFINITY;
    for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    float s = 0.f;
    for (int v = threadIdx.x; v < V; v += blockDim.x)
        if (DUST_IB(t * V + v, zext)) s += expf(zr[v] - m);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w];
    const float inv = 1.0f / s;
    for (int v = threadIdx.x; v < ldp; v += blockDim.x)
        if (DUST_IB(t * ldp + v, static_cast<int64_t>(gridDim.x) * ldp))
            pr[v] = (v < V && DUST_IB(t * V + v, zext)) ? expf(zr[v] - m) * inv : 0.f;
}

struct DhArgs {
    const float* y1;
    const float* h0;      // GELU(y1), same function as below
    const void* coef;     // Taylor coefficients of the GELU difference (GeluCoefs layout)
    int taylor;
    int T, Tp, C, nd;
    uint32_t draw_first, token0, layer;  // draw_first = draw0 + i0
    float sigma;
    __nv_bfloat16* A1;  // rows x 2C
};

// One thread per (token, channel block of 4), looping over the chunk's draws:
// the clean activations (or the Taylor coefficients of the GELU difference)
// are read once and reused for every draw; the A1 rows of one draw are written
// by consecutive threads.
__global__ void interior_dh_kernel(const DhArgs a, const PhiloxKeys keys) {
    const int nblk = a.C >> 2;
    const int64_t n = static_cast<int64_t>(a.Tp) * nblk;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int j = static_cast<int>(idx % nblk);
        const int t = static_cast<int>(idx / nblk);
        const bool valid = t < a.T;
        const int64_t e4 = static_cast<int64_t>(valid ? t : 0) * (a.C / 4) + j;
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f), g = y, c1 = y;
        uint4 c23 = make_uint4(0u, 0u, 0u, 0u);
        if (valid && DUST_IB(e4, static_cast<int64_t>(a.T) * (a.C / 4))) {
            if (a.taylor) {
                const GeluCoefs cf = gelu_coefs(a.coef, static_cast<int64_t>(a.T) * (a.C / 4));
                c1 = __ldg(cf.c1 + e4);
                c23 = __ldg(cf.c23 + e4);
            } else {
                y = __ldg(reinterpret_cast<const float4*>(a.y1) + e4);
                g = __ldg(reinterpret_cast<const float4*>(a.h0) + e4);
            }
        }
        const BlockHalf2 bh = philox_block_half2(philox_block_half(j, a.layer, keys), keys);
        for (int i = 0; i < a.nd; ++i) {
            __nv_bfloat16* row = a.A1 + chunk_row(t, i, a.nd) * (2 * static_cast<int64_t>(a.C));
            __nv_bfloat16 h[4], l[4];
            if (valid) {
                const float4 nrm = words_to_normals_fast(
                    philox_rest2(philox_draw_half2(philox_draw_half(a.draw_first + i, a.token0 + t, keys)),
                                 bh, keys));
                float d[4];
                if (a.taylor) {
                    const float2 sg = make_float2(a.sigma, a.sigma);
                    const float2 e01 = mul2(sg, make_float2(nrm.x, nrm.y));
                    const float2 e23 = mul2(sg, make_float2(nrm.z, nrm.w));
                    float2 d01, d23;
                    gelu_taylor_pairs(c1, c23, make_float4(e01.x, e01.y, e23.x, e23.y), d01, d23);
                    d[0] = d01.x; d[1] = d01.y; d[2] = d23.x; d[3] = d23.y;
                } else {
                    // the GEMM 1 producers' arithmetic, on packed pairs (same bits)
                    const float2 sg = make_float2(a.sigma, a.sigma);
                    const float2 d01 = sub2(
                        gelu_as2(fma2(sg, make_float2(nrm.x, nrm.y), make_float2(y.x, y.y))),
                        make_float2(g.x, g.y));
                    const float2 d23 = sub2(
                        gelu_as2(fma2(sg, make_float2(nrm.z, nrm.w), make_float2(y.z, y.w))),
                        make_float2(g.z, g.w));
                    d[0] = d01.x; d[1] = d01.y; d[2] = d23.x; d[3] = d23.y;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) split_bf16(d[k], h[k], l[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) h[k] = l[k] = __float2bfloat16_rn(0.f);
            }
            const int64_t ri = chunk_row(t, i, a.nd) * (2 * static_cast<int64_t>(a.C));
            const int64_t rext = static_cast<int64_t>(a.nd) * a.Tp * 2 * a.C;
            if (DUST_IB(ri + 4 * j + 3, rext))
                *reinterpret_cast<uint2*>(row + 4 * j) = pack4(h[0], h[1], h[2], h[3]);
            if (DUST_IB(ri + a.C + 4 * j + 3, rext))
                *reinterpret_cast<uint2*>(row + a.C + 4 * j) = pack4(l[0], l[1], l[2], l[3]);
        }
    }
}

// Causal EMA down each sequence, written as the split pair [hi | lo].
// One CTA per (draw in chunk, sequence, 32 channels): lane = channel, warp w =
// the w-th of 16 consecutive token chunks of the sequence.  Each warp runs
// the recurrence over its chunk from zero and keeps its end state and
// lam^length; one warp then chains the chunk ends into every chunk's true
// starting state; each warp reruns its chunk from that state and writes the
// result.  The recurrence is the sequential one, started at the chained
// carry.
constexpr int kEmaWarps = 16;

__global__ void __launch_bounds__(32 * kEmaWarps)
    interior_ema_kernel(const float* __restrict__ du, int nd, int nseq, int seq_len, int dm,
                        float lam, __nv_bfloat16* __restrict__ A2) {
    __shared__ float s_end[kEmaWarps][32];
    __shared__ float s_pow[kEmaWarps][32];
    __shared__ float s_carry[kEmaWarps][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int ncb = (dm + 31) / 32;
    const int cb = blockIdx.x % ncb;
    const int rest = blockIdx.x / ncb;
    const int s = rest % nseq;
    const int i = rest / nseq;
    const int k = cb * 32 + lane;
    const bool ok = k < dm;
    const int clen = (seq_len + kEmaWarps - 1) / kEmaWarps;
    const int t0 = s * seq_len + min(seq_len, w * clen);
    const int t1 = s * seq_len + min(seq_len, (w + 1) * clen);
    const float one_m = 1.0f - lam;
    // du and A2 hold nd x round_up(T, 128) rows
    const int64_t rows_ext = static_cast<int64_t>(nd) * (((nseq * seq_len) + 127) / 128 * 128);
    const int64_t du_ext = rows_ext * dm, a2_ext = rows_ext * 2 * dm;

    float e = 0.f, pw = 1.f;
    if (ok) {
        // loads of 8 tokens issued together, then the 8 dependent steps
        int t = t0;
        for (; t + 8 <= t1; t += 8) {
            float u[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t di = chunk_row(t + q, i, nd) * dm + k;
                u[q] = DUST_IB(di, du_ext) ? __ldg(du + di) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                e = fmaf(lam, e, one_m * u[q]);
                pw *= lam;
            }
        }
        for (; t < t1; ++t) {
            const int64_t di = chunk_row(t, i, nd) * dm + k;
            e = fmaf(lam, e, one_m * (DUST_IB(di, du_ext) ? __ldg(du + di) : 0.f));
            pw *= lam;
        }
    }
    s_end[w][lane] = e;
    s_pow[w][lane] = pw;
    __syncthreads();
    if (w == 0) {
        float c = 0.f;
        for (int q = 0; q < kEmaWarps; ++q) {
            s_carry[q][lane] = c;
            c = fmaf(s_pow[q][lane], c, s_end[q][lane]);
        }
    }
    __syncthreads();
    if (ok) {
        e = s_carry[w][lane];
        int t = t0;
        for (; t + 8 <= t1; t += 8) {
            float u[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t di = chunk_row(t + q, i, nd) * dm + k;
                u[q] = DUST_IB(di, du_ext) ? __ldg(du + di) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int64_t r = chunk_row(t + q, i, nd);
                e = fmaf(lam, e, one_m * u[q]);
                __nv_bfloat16 h, l;
                split_bf16(e, h, l);
                if (DUST_IB(r * 2 * dm + dm + k, a2_ext)) {
                    A2[r * 2 * dm + k] = h;
                    A2[r * 2 * dm + dm + k] = l;
                }
            }
        }
        for (; t < t1; ++t) {
            const int64_t r = chunk_row(t, i, nd);
            e = fmaf(lam, e, one_m * (DUST_IB(r * dm + k, du_ext) ? __ldg(du + r * dm + k) : 0.f));
            __nv_bfloat16 h, l;
            split_bf16(e, h, l);
            if (DUST_IB(r * 2 * dm + dm + k, a2_ext)) {
                A2[r * 2 * dm + k] = h;
                A2[r * 2 * dm + dm + k] = l;
            }
        }
    }
}

__global__ void draw_mean_kernel(const float* __restrict__ dl, int K, int T, float* __restrict__ m) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float s = 0.f;
    for (int i = 0; i < K; ++i)
        if (DUST_IB(static_cast<int64_t>(i) * T + t, static_cast<int64_t>(K) * T))
            s += dl[static_cast<int64_t>(i) * T + t];
    if (DUST_IB(t, T)) m[t] = s / static_cast<float>(K);
}

// r_{i,t} = c_{i,t} + gamma r_{i,t+1} inside each sequence, c = -(dl - m).
// r_t = sum_{s >= t, same sequence} gamma^(s-t) c_s with c = -(dl - m), one
// warp per (draw, sequence): lane l owns a contiguous chunk of the sequence,
// runs it once from zero (its chunk's value at the chunk start, A_l, and
// gamma^len, P_l), the warp combines the chunks from the end by a shuffle
// scan of (A, P) pairs, and each lane reruns its chunk from its true carry.
__global__ void reward_scan_kernel(const float* __restrict__ dl, const float* __restrict__ m,
                                   int K, int T, int seq_len, float gamma, float* __restrict__ r) {
    const int nseq = T / seq_len;
    const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (wid >= K * nseq) return;
    const int i = wid / nseq, s = wid - i * nseq;
    const int64_t rowoff = static_cast<int64_t>(i) * T;
    const int chunk = (seq_len + 31) / 32;
    const int t0 = s * seq_len + min(seq_len, lane * chunk);
    const int t1 = s * seq_len + min(seq_len, (lane + 1) * chunk);
    float A = 0.f, P = 1.f;
    const int64_t kt = static_cast<int64_t>(K) * T;
    for (int t = t1 - 1; t >= t0; --t) {
        if (!DUST_IB(rowoff + t, kt) || !DUST_IB(t, T)) continue;
        A = fmaf(gamma, A, -(dl[rowoff + t] - m[t]));
        P *= gamma;
    }
    // Suffix combine over lanes: (A, P)_l <- (A_l + P_l A_{l+1}, P_l P_{l+1}),
    // doubling the reach each step; afterwards A_l is r at the chunk's start.
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float An = __shfl_down_sync(0xFFFFFFFFu, A, o);
        const float Pn = __shfl_down_sync(0xFFFFFFFFu, P, o);
        if (lane + o < 32) {
            A = fmaf(P, An, A);
            P *= Pn;
        }
    }
    // carry into this chunk's last token: r at the next chunk's start
    float acc = __shfl_down_sync(0xFFFFFFFFu, A, 1);
    if (lane == 31) acc = 0.f;
    for (int t = t1 - 1; t >= t0; --t) {
        if (!DUST_IB(rowoff + t, kt) || !DUST_IB(t, T)) continue;
        acc = fmaf(gamma, acc, -(dl[rowoff + t] - m[t]));
        r[rowoff + t] = acc;
    }
}

struct GhatArgs {
    const float* r;  // K x T
    int T, C, K;
    uint32_t draw0, token0, layer;
    float neg_inv_ks;  // -1 / (K sigma)
    float* g_hat;      // T x C or null
    __nv_bfloat16* gbf;  // T x C
};

// One thread per (token, two channel blocks j and j + C/8): g =
// -(1/(K sigma)) sum_i r a, with the noise regenerated from its counters.  The
// two blocks advance in lockstep so that their Philox chains interleave.
__global__ void interior_ghat_kernel(const GhatArgs a, const PhiloxKeys keys) {
    const int half = a.C >> 3;  // channel blocks per half row
    const int64_t n = static_cast<int64_t>(a.T) * half;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int j0 = static_cast<int>(idx % half);
        const int t = static_cast<int>(idx / half);
        const int jb[2] = {j0, j0 + half};
        BlockHalf2 bh[2];
        float4 acc[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            bh[u] = philox_block_half2(philox_block_half(jb[u], a.layer, keys), keys);
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float* rcol = a.r + t;
#pragma unroll 2
        for (int i = 0; i < a.K; ++i) {
            const float ri = DUST_IB(t + static_cast<int64_t>(i) * a.T, static_cast<int64_t>(a.K) * a.T)
                                 ? __ldg(rcol + static_cast<int64_t>(i) * a.T)
                                 : 0.f;
            const DrawHalf2 dh = philox_draw_half2(philox_draw_half(a.draw0 + i, a.token0 + t, keys));
            uint4 w[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) w[u] = philox_rest2(dh, bh[u], keys);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float4 nrm = words_to_normals_fast(w[u]);
                const float2 r2 = make_float2(ri, ri);
                const float2 lo = fma2(r2, make_float2(nrm.x, nrm.y), make_float2(acc[u].x, acc[u].y));
                const float2 hi = fma2(r2, make_float2(nrm.z, nrm.w), make_float2(acc[u].z, acc[u].w));
                acc[u] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float4 g = make_float4(acc[u].x * a.neg_inv_ks, acc[u].y * a.neg_inv_ks,
                                         acc[u].z * a.neg_inv_ks, acc[u].w * a.neg_inv_ks);
            const int64_t off = static_cast<int64_t>(t) * a.C + 4 * jb[u];
            if (!DUST_IB(off + 3, static_cast<int64_t>(a.T) * a.C)) continue;
            if (a.g_hat) *reinterpret_cast<float4*>(a.g_hat + off) = g;
            *reinterpret_cast<uint2*>(a.gbf + off) =
                pack4(__float2bfloat16_rn(g.x), __float2bfloat16_rn(g.y),
                      __float2bfloat16_rn(g.z), __float2bfloat16_rn(g.w));
        }
    }
}

struct InteriorPlan {
    int64_t Tp, ldx;
    int nd;      // draws per chunk
    bool fused;  // GEMM 1 generates its A operand on chip
    size_t off_p, off_h0, off_coef, off_a1, off_du, off_a2, off_dl, off_m, off_r, off_gbf, off_xbf, bytes;
};

InteriorPlan interior_plan(int64_t T, int64_t d_in, int64_t C, int64_t dm, int64_t V, uint32_t K) {
    InteriorPlan P{};
    P.Tp = round_up(T, kRowBlock);
    P.ldx = round_up(d_in, 8);
    // Draws per chunk: at least eight 128-row tiles per SM, and where the
    // count allows, a chunk of nd x (token blocks) tiles that is a whole
    // number of waves over the 148 SMs.
    const int64_t ntb = P.Tp / kRowBlock;
    int64_t nd = ceil_div(148 * 8, ntb);
    for (int64_t c = nd; c <= std::min<int64_t>(64, 4 * nd); ++c)
        if ((c * ntb) % 148 == 0) {
            nd = c;
            break;
        }
    nd = std::max<int64_t>(1, std::min<int64_t>({nd, 64, static_cast<int64_t>(K)}));
    P.nd = static_cast<int>(nd);
    P.fused = reforward1_supported(C, dm);
    const size_t rows = static_cast<size_t>(nd * P.Tp);
    WsLayout w;
    w.take(kCtlBytes);
    P.off_p = w.take(static_cast<size_t>(T * round_up(V, 4)) * 4);
    P.off_h0 = w.take(static_cast<size_t>(T * C) * 4);
    P.off_coef = w.take(static_cast<size_t>(T * C) * 8);  // GeluCoefs
    P.off_a1 = w.take(P.fused ? 0 : rows * static_cast<size_t>(2 * C) * 2);
    P.off_du = w.take(rows * static_cast<size_t>(dm) * 4);
    P.off_a2 = w.take(rows * static_cast<size_t>(2 * dm) * 2);
    P.off_dl = w.take(static_cast<size_t>(K) * T * 4);
    P.off_m = w.take(static_cast<size_t>(T) * 4);
    P.off_r = w.take(static_cast<size_t>(K) * T * 4);
    P.off_gbf = w.take(static_cast<size_t>(T * C) * 2);
    P.off_xbf = w.take(static_cast<size_t>(T * P.ldx) * 2);
    P.bytes = w.used;
    return P;
}

unsigned grid_cap(int64_t n, int threads) {
    int64_t b = ceil_div(n, threads);
    b = std::min<int64_t>(b, 148 * 32);
    return static_cast<unsigned>(std::max<int64_t>(b, 1));
}

}  // namespace

dust_status credit_and_ghat_launch(const float* dl, float* mean, float* r, int T, int seq_len,
                                   int C, const dust_noise& nz, const PhiloxKeys& keys,
                                   float* g_hat, __nv_bfloat16* gbf, cudaStream_t s) {
    const int K = static_cast<int>(nz.num_draws);
    const int nseq = T / seq_len;
    draw_mean_kernel<<<static_cast<unsigned>(ceil_div(T, 256)), 256, 0, s>>>(dl, K, T, mean);
    reward_scan_kernel<<<static_cast<unsigned>(ceil_div(static_cast<int64_t>(K) * nseq, 4)), 128,
                         0, s>>>(dl, mean, K, T, seq_len, nz.gamma, r);
    dust_status st = launch_status();
    if (st != DUST_OK) return st;
    GhatArgs ga{r, T, C, K, nz.draw0, nz.token0, nz.layer,
                static_cast<float>(-1.0 / (static_cast<double>(K) * nz.sigma)), g_hat, gbf};
    interior_ghat_kernel<<<grid_cap(static_cast<int64_t>(T) * (C / 8), 256), 256, 0, s>>>(ga, keys);
    return launch_status();
}
}  // namespace dust

using namespace dust;

extern "C" size_t dust_linear_workspace(int64_t T, int64_t d_in, int64_t C, int64_t d_model,
                                        int64_t V, uint32_t K) {
    if (T < 1 || d_in < 1 || C < 1 || d_model < 1 || V < 1 || K < 2) return 0;
    return interior_plan(T, d_in, C, d_model, V, K).bytes;
}

dust_status dust::linear_estimate_check(const void* x, const float* y1, const void* W2,
                                        float ema_decay, const void* W_head,
                                        const float* z_clean, const int32_t* targets, int64_t T,
                                        int64_t seq_len, int64_t d_in, int64_t C,
                                        int64_t d_model, int64_t V, const dust_noise& nz,
                                        const float* g_hat, const float* G_W1, const void* ws,
                                        size_t ws_bytes) {
    if (!x || !y1 || !W2 || !W_head || !z_clean || !targets || !G_W1) return DUST_ERR_INVALID_ARG;
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || d_in < 1 || C < 1 || d_model < 1 || V < 1)
        return DUST_ERR_INVALID_ARG;
    if (nz.num_draws < 2 || !(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (!(nz.gamma >= 0.0f && nz.gamma <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (!(ema_decay >= 0.0f && ema_decay <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (C % 64 != 0 || d_model % 64 != 0) return DUST_ERR_UNSUPPORTED;
    if (T > (1LL << 28) || C > (1LL << 16) || d_model > (1LL << 16) || V > (1LL << 20) ||
        d_in > (1LL << 20) || nz.num_draws > (1u << 24))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32) ||
        static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (!aligned(y1, 16) || !aligned(W2, 16) || !aligned(W_head, 16) || !aligned(z_clean, 16) ||
        (g_hat && !aligned(g_hat, 16)))
        return DUST_ERR_INVALID_ARG;
    const InteriorPlan P = interior_plan(T, d_in, C, d_model, V, nz.num_draws);
    if (!ws || ws_bytes < P.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

extern "C" dust_status dust_linear_estimate(const void* x, const float* y1, const void* W2,
                                            float ema_decay, const void* W_head,
                                            const float* z_clean, const int32_t* targets,
                                            int64_t T, int64_t seq_len, int64_t d_in, int64_t C,
                                            int64_t d_model, int64_t V, dust_noise nz,
                                            float* g_hat, float* G_W1, void* ws, size_t ws_bytes,
                                            void* stream) {
    const dust_status chk = linear_estimate_check(x, y1, W2, ema_decay, W_head, z_clean, targets,
                                                  T, seq_len, d_in, C, d_model, V, nz, g_hat,
                                                  G_W1, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const InteriorPlan P = interior_plan(T, d_in, C, d_model, V, nz.num_draws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint32_t* status = static_cast<uint32_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));

    float* p = reinterpret_cast<float*>(w + P.off_p);
    __nv_bfloat16* A1 = reinterpret_cast<__nv_bfloat16*>(w + P.off_a1);
    float* du = reinterpret_cast<float*>(w + P.off_du);
    __nv_bfloat16* A2 = reinterpret_cast<__nv_bfloat16*>(w + P.off_a2);
    float* dl = reinterpret_cast<float*>(w + P.off_dl);
    float* mean = reinterpret_cast<float*>(w + P.off_m);
    float* r = reinterpret_cast<float*>(w + P.off_r);
    __nv_bfloat16* gbf = reinterpret_cast<__nv_bfloat16*>(w + P.off_gbf);
    const int K = static_cast<int>(nz.num_draws);
    const int Ti = static_cast<int>(T), Ci = static_cast<int>(C), dmi = static_cast<int>(d_model);
    const PhiloxKeys keys = philox_round_keys(nz.seed);
    dust_status st;

    const int64_t ldp = round_up(V, 4);
    softmax_rows_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(z_clean, static_cast<int>(V),
                                                                 static_cast<int>(ldp), p);
    if ((st = launch_status()) != DUST_OK) return st;
    float* h0 = reinterpret_cast<float*>(w + P.off_h0);
    if ((st = gelu_launch(y1, T * C, h0, s)) != DUST_OK) return st;
    // Small sigma: GELU(y1 + d) - GELU(y1) by its third-order Taylor
    // polynomial in d, coefficients once per call (8 bytes per channel),
    // read once per draw by GEMM 1's on-chip producers and once per chunk by
    // the staged path; a few packed fmas replace the GELU's erf, reciprocal
    // and exponential.
    const bool taylor = 5.77 * nz.sigma <= 0.15;
    void* coef = w + P.off_coef;
    if (taylor && (st = gelu_taylor_launch(y1, T * C, coef, s)) != DUST_OK) return st;

    const int nseq = static_cast<int>(T / seq_len);
    const bool fuse_ema = P.fused && seq_len % kRowBlock == 0 && P.Tp == T;
    for (int i0 = 0; i0 < K; i0 += P.nd) {
        const int nd = std::min(P.nd, K - i0);
        const int64_t rows = nd * P.Tp;
        // (the benchmark hook times GEMM 1 here, GEMM 2 inside gemm_ce_launch,
        // and the credit + g pass after the loop)
        if (P.fused) {
            // Whole token blocks per sequence: the EMA runs in GEMM 1's
            // epilogue, one CTA walking a sequence's blocks for one draw.
            timer_begin(s);
            st = reforward1_launch(y1, h0, coef, taylor, W2, T, P.Tp, C, d_model, nd,
                                   nz.draw0 + static_cast<uint32_t>(i0), nz.token0, nz.layer,
                                   nz.sigma, keys, du, fuse_ema ? A2 : nullptr, seq_len,
                                   ema_decay, status, s);
            timer_end(s);
            if (st != DUST_OK) return st;
        } else {
            DhArgs da{y1, h0, static_cast<const float4*>(coef), taylor ? 1 : 0, Ti,
                      static_cast<int>(P.Tp), Ci, nd, nz.draw0 + static_cast<uint32_t>(i0),
                      nz.token0, nz.layer, nz.sigma, A1};
            interior_dh_kernel<<<grid_cap(P.Tp * (C / 4), 256), 256, 0, s>>>(da, keys);
            if ((st = launch_status()) != DUST_OK) return st;
            timer_begin(s);
            st = gemm_bf16_launch(A1, false, 2 * C, W2, false, C, rows, d_model, 2 * C, C, 1, du,
                                  d_model, status, s);
            timer_end(s);
            if (st != DUST_OK) return st;
        }
        if (!fuse_ema) {
            if (P.Tp != T)
                DUST_CUDA_TRY(
                    cudaMemsetAsync(A2, 0, static_cast<size_t>(rows * 2 * d_model) * 2, s));
            interior_ema_kernel<<<static_cast<unsigned>(nd * nseq * ceil_div(d_model, 32)),
                                  32 * kEmaWarps, 0, s>>>(du, nd, nseq, static_cast<int>(seq_len),
                                                          dmi, ema_decay, A2);
            if ((st = launch_status()) != DUST_OK) return st;
        }
        st = gemm_ce_launch(A2, 2 * d_model, W_head, d_model, rows, V, 2 * d_model, d_model, p,
                            ldp, targets, T, nd, i0, dl, status, s);
        if (st != DUST_OK) return st;
    }

    timer_begin(s);
    st = credit_and_ghat_launch(dl, mean, r, Ti, static_cast<int>(seq_len), Ci, nz, keys, g_hat,
                                gbf, s);
    timer_end(s);
    if (st != DUST_OK) return st;

    const void* xb = x;
    int64_t ldx = d_in;
    if ((d_in % 8) != 0 || !aligned(x, 16)) {
        void* xbf = w + P.off_xbf;
        if ((st = bf16_pad_launch(x, T, d_in, d_in, xbf, P.ldx, s)) != DUST_OK) return st;
        xb = xbf;
        ldx = P.ldx;
    }
    return gemm_bf16_launch(gbf, true, C, xb, true, ldx, C, d_in, T, 0, 1, G_W1, d_in, status, s);
}

namespace dust {
DUST_DEBUG_READER(2)
}  // namespace dust
