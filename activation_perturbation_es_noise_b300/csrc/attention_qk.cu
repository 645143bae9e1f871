// attention_qk.cu -- the queries and keys inside attention, scored like the
// values by the error of the attention output.
//
// The pages score every perturbation inside attention by the attention-output
// error with a decay close to 1 for later tokens (Dust translation §2.3;
// laoyaoba.com, section 机制拆解).  Perturbing the query of every token by
// sigma a_s (or the key of every token by sigma a_t) shifts the causal scores
//   ds_{s,t} = sigma <a_s, k_t> / sqrt(64)     (queries)
//   ds_{s,t} = sigma <q_s, a_t> / sqrt(64)     (keys),
// and with the cached clean probabilities P and output o of the same forward
// the perturbed softmax row is P e^{ds} / sum_t P e^{ds}, so the output of
// token s changes by exactly
//   dO_s = (sum_{t<=s} w_{s,t} v_t - W_s o_s) / (1 + W_s),
//   w_{s,t} = P_{s,t} (e^{ds_{s,t}} - 1),   W_s = sum_{t<=s} w_{s,t}
// (P's causal row sums to 1 and o_s = sum_t P_{s,t} v_t).  The loss change is
// dl_s = sum_h <E_s[h], dO_s[h]>, then the usual centring, gamma-scan, g and
// G_W = g^T x (the interior layer's kernels and the outer-product GEMM).
//
// This version runs on the CUDA cores in fp32: one thread per query row keeps
// its 64 scaled noise values (queries) or its scaled query (keys) and its 64
// accumulators in registers; 32-key tiles of the clean keys (or the keys'
// noise) and of the values are staged in shared memory and read as
// broadcasts; the matching 128 x 32 tile of P is staged too (coalesced rows,
// padded against bank conflicts) so that no thread reads its own P row from
// global memory.  A CTA covers one tile of 128 queries of one sequence for one
// draw and walks the heads in order, so the per-token sum over heads needs no
// second pass.  The draws are the fastest grid index: the CTAs resident at one
// time share their sequence, query tile and head, and P, K and V come from L2
// after the first of them.  The per-pair work, 2 x 64 fused multiply-adds and
// one e^x - 1, is the kernel's roofline.
#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {
namespace {

constexpr int kHd = 64;       // channels per head
constexpr int kQKRows = 128;  // query rows per CTA, one per thread
constexpr int kQKKeys = 32;   // keys per staged tile

struct QKArgs {
    const float* Q;   // T x C clean queries (C = H 64)
    const float* Kk;  // T x C clean keys
    const float* V;   // T x C clean values
    const float* O;   // T x C clean attention output
    const float* P;   // nseq x H x L x L clean probabilities (causal rows)
    const float* E;   // T x C error of the attention output
    float* dl;        // K x T loss changes
    int T, L, H;
    uint32_t draw0, token0, layer;
    float scale;      // sigma / sqrt(64)
};

// e^x - 1 for the score shifts: the Taylor polynomial to x^6 for |x| < 1/4
// (truncation below 5e-8 relative there, and no cancellation), else expm1f.
__device__ __forceinline__ float expm1_shift(float x) {
    if (fabsf(x) < 0.25f) {
        float q = fmaf(x, 1.0f / 720.0f, 1.0f / 120.0f);
        q = fmaf(x, q, 1.0f / 24.0f);
        q = fmaf(x, q, 1.0f / 6.0f);
        q = fmaf(x, q, 0.5f);
        q = fmaf(x, q, 1.0f);
        return x * q;
    }
    return expm1f(x);
}

// grid: (draws, query tiles x sequences, heaviest tiles first); block: 128 threads.
// KEYS: the staged tiles carry the keys' noise and the thread holds its query;
// otherwise the thread holds its query's noise and the tiles the clean keys.
template <bool KEYS>
__global__ void __launch_bounds__(kQKRows) attn_qk_kernel(const QKArgs a, const PhiloxKeys keys) {
    __shared__ __align__(16) float kt[kQKKeys][kHd];
    __shared__ __align__(16) float vt[kQKKeys][kHd];
    __shared__ float pt[kQKRows][kQKKeys + 1];
    const int r = threadIdx.x;
    const int nseq = a.T / a.L;
    const int qb = a.L / kQKRows - 1 - static_cast<int>(blockIdx.y) / nseq;  // heavy first
    const int sq = static_cast<int>(blockIdx.y) % nseq;
    const int i = blockIdx.x;
    const uint32_t draw = a.draw0 + static_cast<uint32_t>(i);
    const int s = qb * kQKRows + r;                          // query position in its sequence
    const int64_t tg = static_cast<int64_t>(sq) * a.L + s;   // token
    const int C = a.H * kHd;
    const int kend = (qb + 1) * kQKRows;                     // keys up to the tile's last query
    const DrawHalf dh = philox_draw_half(draw, a.token0 + static_cast<uint32_t>(tg), keys);

    float dl = 0.f;
    for (int h = 0; h < a.H; ++h) {
        float qa[kHd];
        if (KEYS) {
#pragma unroll
            for (int c = 0; c < kHd; c += 4) {
                const float4 q4 = *reinterpret_cast<const float4*>(a.Q + tg * C + h * kHd + c);
                qa[c] = a.scale * q4.x;
                qa[c + 1] = a.scale * q4.y;
                qa[c + 2] = a.scale * q4.z;
                qa[c + 3] = a.scale * q4.w;
            }
        } else {
#pragma unroll
            for (int jb = 0; jb < kHd / 4; ++jb) {
                const float4 n = words_to_normals(philox_rest(
                    dh, philox_block_half(static_cast<uint32_t>(h * (kHd / 4) + jb), a.layer, keys),
                    keys));
                qa[4 * jb] = a.scale * n.x;
                qa[4 * jb + 1] = a.scale * n.y;
                qa[4 * jb + 2] = a.scale * n.z;
                qa[4 * jb + 3] = a.scale * n.w;
            }
        }
        float acc[kHd];
#pragma unroll
        for (int c = 0; c < kHd; ++c) acc[c] = 0.f;
        float wsum = 0.f;
        // row qb 128 of this (sequence, head)'s probabilities
        const float* ptile = a.P + ((static_cast<int64_t>(sq) * a.H + h) * a.L + qb * kQKRows) * a.L;

        for (int k0 = 0; k0 < kend; k0 += kQKKeys) {
            __syncthreads();  // the previous tile (or head) is no longer read
            for (int e = r; e < kQKKeys * (kHd / 4); e += kQKRows) {
                const int kk = e / (kHd / 4), jb = e % (kHd / 4);
                const int64_t tk = static_cast<int64_t>(sq) * a.L + k0 + kk;
                const float4 v4 = *reinterpret_cast<const float4*>(a.V + tk * C + h * kHd + 4 * jb);
                float4 k4;
                if (KEYS)
                    k4 = words_to_normals(philox4x32_10(static_cast<uint32_t>(h * (kHd / 4) + jb),
                                                        a.token0 + static_cast<uint32_t>(tk), draw,
                                                        a.layer, keys));
                else
                    k4 = *reinterpret_cast<const float4*>(a.Kk + tk * C + h * kHd + 4 * jb);
                *reinterpret_cast<float4*>(&vt[kk][4 * jb]) = v4;
                *reinterpret_cast<float4*>(&kt[kk][4 * jb]) = k4;
            }
            for (int e = r; e < kQKRows * (kQKKeys / 4); e += kQKRows) {
                const int row = e / (kQKKeys / 4), q4 = e % (kQKKeys / 4);
                const float4 p4 = __ldg(reinterpret_cast<const float4*>(
                    ptile + static_cast<int64_t>(row) * a.L + k0 + 4 * q4));
                pt[row][4 * q4] = p4.x;
                pt[row][4 * q4 + 1] = p4.y;
                pt[row][4 * q4 + 2] = p4.z;
                pt[row][4 * q4 + 3] = p4.w;
            }
            __syncthreads();
            const int tmax = min(kQKKeys, s - k0 + 1);  // causal: keys t <= s
            for (int kk = 0; kk < tmax; ++kk) {
                float d4[4] = {0.f, 0.f, 0.f, 0.f};  // four chains, not one of 64
#pragma unroll
                for (int c = 0; c < kHd; ++c) d4[c & 3] = fmaf(qa[c], kt[kk][c], d4[c & 3]);
                const float ds = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                const float w = pt[r][kk] * expm1_shift(ds);
                wsum += w;
#pragma unroll
                for (int c = 0; c < kHd; ++c) acc[c] = fmaf(w, vt[kk][c], acc[c]);
            }
        }
        const float* orow = a.O + tg * C + h * kHd;
        const float* erow = a.E + tg * C + h * kHd;
        float eo = 0.f;
#pragma unroll
        for (int c = 0; c < kHd; ++c) eo = fmaf(erow[c], fmaf(-wsum, orow[c], acc[c]), eo);
        dl += eo / (1.0f + wsum);
    }
    a.dl[static_cast<int64_t>(i) * a.T + tg] = dl;
}

struct QKPlan {
    int64_t ldx;
    size_t off_dl, off_m, off_r, off_gbf, off_xbf, bytes;
};

QKPlan qk_plan(int64_t T, int64_t H, int64_t d_in, uint32_t K) {
    QKPlan P{};
    const int64_t C = H * kHd;
    P.ldx = round_up(d_in, 8);
    WsLayout w;
    w.take(kCtlBytes);
    P.off_dl = w.take(static_cast<size_t>(K) * T * 4);
    P.off_m = w.take(static_cast<size_t>(T) * 4);
    P.off_r = w.take(static_cast<size_t>(K) * T * 4);
    P.off_gbf = w.take(static_cast<size_t>(T * C) * 2);
    P.off_xbf = w.take(static_cast<size_t>(T * P.ldx) * 2);
    P.bytes = w.used;
    return P;
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" size_t dust_attn_qk_workspace(int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                                         int64_t d_in, uint32_t K) {
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || H < 1 || dv != kHd || d_in < 1 || K < 2)
        return 0;
    return qk_plan(T, H, d_in, K).bytes;
}

extern "C" dust_status dust_attn_qk_estimate(int which, const float* Q, const float* Kk,
                                             const float* V, const float* O, const float* P,
                                             const float* E, const void* x, dust_dtype x_dtype,
                                             int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                                             int64_t d_in, dust_noise nz, float* g_hat,
                                             float* G_W, void* ws, size_t ws_bytes, void* stream) {
    if (which != 0 && which != 1) return DUST_ERR_INVALID_ARG;
    if (!Q || !Kk || !V || !O || !P || !E || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || H < 1 || d_in < 1) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (nz.num_draws < 2 || !(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (!(nz.gamma >= 0.0f && nz.gamma <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (dv != kHd || seq_len % kQKRows != 0 || seq_len > 8192 || H > 64 || T / kQKRows > 65535 ||
        nz.num_draws > 65535 || d_in > (1LL << 20))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32) ||
        static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(Kk, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(P, 16) || !aligned(E, 4) || (g_hat && !aligned(g_hat, 16)))
        return DUST_ERR_INVALID_ARG;
    const QKPlan Pl = qk_plan(T, H, d_in, nz.num_draws);
    if (!ws || ws_bytes < Pl.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint32_t* status = static_cast<uint32_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    const int64_t C = H * kHd;
    float* dl = reinterpret_cast<float*>(w + Pl.off_dl);
    float* mean = reinterpret_cast<float*>(w + Pl.off_m);
    float* r = reinterpret_cast<float*>(w + Pl.off_r);
    __nv_bfloat16* gbf = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_gbf);
    const PhiloxKeys keys = philox_round_keys(nz.seed);

    const QKArgs qa{Q, Kk, V, O, P, E, dl, static_cast<int>(T), static_cast<int>(seq_len),
                    static_cast<int>(H), nz.draw0, nz.token0, nz.layer, nz.sigma * 0.125f};
    const dim3 grid(nz.num_draws, static_cast<unsigned>(T / kQKRows));
    timer_begin(s);
    if (which == 1)
        attn_qk_kernel<true><<<grid, kQKRows, 0, s>>>(qa, keys);
    else
        attn_qk_kernel<false><<<grid, kQKRows, 0, s>>>(qa, keys);
    timer_end(s);
    dust_status st = launch_status();
    if (st != DUST_OK) return st;
    st = credit_and_ghat_launch(dl, mean, r, static_cast<int>(T), static_cast<int>(seq_len),
                                static_cast<int>(C), nz, keys, g_hat, gbf, s);
    if (st != DUST_OK) return st;
    const void* xb = x;
    int64_t ldx = d_in;
    if (x_dtype == DUST_F32 || (d_in % 8) != 0 || !aligned(x, 16)) {
        void* xbf = w + Pl.off_xbf;
        st = x_dtype == DUST_F32
                 ? f32_to_bf16_launch(static_cast<const float*>(x), T, d_in, d_in, xbf, Pl.ldx, s)
                 : bf16_pad_launch(x, T, d_in, d_in, xbf, Pl.ldx, s);
        if (st != DUST_OK) return st;
        xb = xbf;
        ldx = Pl.ldx;
    }
    return gemm_bf16_launch(gbf, true, C, xb, true, ldx, C, d_in, T, 0, 1, G_W, d_in, status, s);
}
