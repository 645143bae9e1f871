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
// This version runs on the CUDA cores in fp32, as two register-blocked
// products per 32-key tile (the flash-attention shape): the score shifts of a
// 128-query tile against the key tile, the weights w = P (e^ds - 1) formed in
// registers (P read straight from L2, the causal mask applied), and w times
// the value tile added to a 128 x 64 accumulator spread over the CTA's
// registers.  A CTA covers one tile of 128 queries of one sequence for one
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
constexpr int kQKRows = 128;  // query rows per CTA
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

// Shared memory of one CTA (floats): the thread side of the scores, transposed
// (channel-major, 64 x 128), a key tile transposed (64 x 32), a value tile
// (32 x 64), the weights w transposed (32 x 128), and per-row partial sums.
constexpr int kQKThreads = 128;
constexpr int kOffA = 0;
constexpr int kOffK = kOffA + kHd * kQKRows;
constexpr int kOffV = kOffK + kHd * kQKKeys;
constexpr int kOffW = kOffV + kQKKeys * kHd;
constexpr int kOffWs = kOffW + kQKKeys * kQKRows;  // 2 x 128 row sums of w
constexpr int kOffDl = kOffWs + 2 * kQKRows;       // 2 x 128 partial dl
constexpr int kQKSmemBytes = (kOffDl + 2 * kQKRows) * 4;

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Row of a thread's x-th query (x < 8) relative to its first row.
__device__ __forceinline__ constexpr int qk_row(int x) { return (x & 3) + 32 * (x >> 2); }

// grid: (draws, query tiles x sequences, heaviest tiles first); block: 256.
// Per 32-key tile two register-blocked products on the CUDA cores:
//   ds[128 x 32] = A[128 x 64] Kt^T   (A: scaled noise of the queries, or the
//                                     scaled queries when the keys carry it)
//   w = P (e^ds - 1), masked causally;  acc[128 x 64] += w[128 x 32] V[32 x 64].
// Warp w covers rows 64 (w mod 2) .. + 63 in both; lane (r8 = lane mod 8,
// q = lane / 8) owns rows 4 r8 .. + 3 and 32 + 4 r8 .. + 3 of them (eight lanes'
// 16-byte loads cover 128 contiguous bytes: no bank conflicts), keys 16 (w / 2) + 4 q .. + 3 of
// the first product and channels 32 (w / 2) + 8 q .. + 7 of the second, so
// that each 16-byte shared load feeds 32 / 3 (first) or 16 (second) fused
// multiply-adds.
template <bool KEYS>
__global__ void __launch_bounds__(kQKThreads, 3) attn_qk_kernel(const QKArgs a, const PhiloxKeys keys) {
    extern __shared__ __align__(16) float sm[];
    float* At = sm + kOffA;  // [c][row]
    float* Kt = sm + kOffK;  // [c][key]
    float* Vt = sm + kOffV;  // [key][c]
    float* Wt = sm + kOffW;  // [key][row]
    float* wsp = sm + kOffWs;
    float* dlp = sm + kOffDl;
    const int tid = threadIdx.x;
    const int lane = tid & 31, wi = tid >> 5;
    const int r8 = lane & 7, q = lane >> 3;
    const int rb = wi & 1, hb = wi >> 1;   // row block (64 rows), half (keys / channels)
    const int row0 = 64 * rb + 4 * r8;     // rows row0 + (x & 3) + 32 (x >> 2), x < 8
    const int key0 = 16 * hb + 4 * q;      // its 4 keys of a key tile (first product)
    const int ch0 = 32 * hb + 8 * q;       // its 8 channels (second product)
    const int nseq = a.T / a.L;
    const int qb = a.L / kQKRows - 1 - static_cast<int>(blockIdx.y) / nseq;  // heavy first
    const int sq = static_cast<int>(blockIdx.y) % nseq;
    const int i = blockIdx.x;
    const uint32_t draw = a.draw0 + static_cast<uint32_t>(i);
    const int C = a.H * kHd;
    const int64_t tok0 = static_cast<int64_t>(sq) * a.L + qb * kQKRows;  // the tile's first token
    const int s0 = qb * kQKRows + row0;                                   // position of row0
    const int kend = (qb + 1) * kQKRows;

    float dlr[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) dlr[x] = 0.f;
    for (int h = 0; h < a.H; ++h) {
        // the thread side of the scores, channel-major (lanes over rows: no conflicts)
        for (int e = tid; e < kQKRows * (kHd / 4); e += kQKThreads) {
            const int row = e % kQKRows, jb = e / kQKRows;
            float4 v;
            if (KEYS) {
                v = ld4(a.Q + (tok0 + row) * C + h * kHd + 4 * jb);
            } else {
                v = words_to_normals(philox4x32_10(static_cast<uint32_t>(h * (kHd / 4) + jb),
                                                   a.token0 + static_cast<uint32_t>(tok0 + row),
                                                   draw, a.layer, keys));
            }
            At[(4 * jb) * kQKRows + row] = a.scale * v.x;
            At[(4 * jb + 1) * kQKRows + row] = a.scale * v.y;
            At[(4 * jb + 2) * kQKRows + row] = a.scale * v.z;
            At[(4 * jb + 3) * kQKRows + row] = a.scale * v.w;
        }
        float acc[8][8];
        float wsacc[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            wsacc[x] = 0.f;
#pragma unroll
            for (int y = 0; y < 8; ++y) acc[x][y] = 0.f;
        }
        const float* prow = a.P + ((static_cast<int64_t>(sq) * a.H + h) * a.L + s0) * a.L;

        for (int k0 = 0; k0 < kend; k0 += kQKKeys) {
            __syncthreads();  // the previous tile's Kt, Vt, Wt (and At's writes) settled
            for (int e = tid; e < kQKKeys * (kHd / 4); e += kQKThreads) {
                const int key = e % kQKKeys, jb = e / kQKKeys;
                const int64_t tk = static_cast<int64_t>(sq) * a.L + k0 + key;
                float4 v;
                if (KEYS)
                    v = words_to_normals(philox4x32_10(static_cast<uint32_t>(h * (kHd / 4) + jb),
                                                       a.token0 + static_cast<uint32_t>(tk), draw,
                                                       a.layer, keys));
                else
                    v = ld4(a.Kk + tk * C + h * kHd + 4 * jb);
                Kt[(4 * jb) * kQKKeys + key] = v.x;
                Kt[(4 * jb + 1) * kQKKeys + key] = v.y;
                Kt[(4 * jb + 2) * kQKKeys + key] = v.z;
                Kt[(4 * jb + 3) * kQKKeys + key] = v.w;
            }
            for (int e = tid; e < kQKKeys * (kHd / 4); e += kQKThreads) {
                const int key = e / (kHd / 4), jb = e % (kHd / 4);
                const int64_t tk = static_cast<int64_t>(sq) * a.L + k0 + key;
                *reinterpret_cast<float4*>(Vt + key * kHd + 4 * jb) =
                    ld4(a.V + tk * C + h * kHd + 4 * jb);
            }
            __syncthreads();
            // ds = A Kt^T for 8 rows x 4 keys
            float w[8][4];
#pragma unroll
            for (int x = 0; x < 8; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) w[x][y] = 0.f;
#pragma unroll 8
            for (int c = 0; c < kHd; ++c) {
                const float4 a0 = ld4(At + c * kQKRows + row0);
                const float4 a1 = ld4(At + c * kQKRows + row0 + 32);
                const float4 kv = ld4(Kt + c * kQKKeys + key0);
                const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float kr[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int x = 0; x < 8; ++x)
#pragma unroll
                    for (int y = 0; y < 4; ++y) w[x][y] = fmaf(ar[x], kr[y], w[x][y]);
            }
            // w = P (e^ds - 1) on keys t <= s, in place
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float4 pv = __ldg(reinterpret_cast<const float4*>(
                    prow + static_cast<int64_t>(qk_row(x)) * a.L + k0 + key0));
                const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
                float part = 0.f;
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const bool live = k0 + key0 + y <= s0 + qk_row(x);
                    w[x][y] = live ? pr[y] * expm1_shift(w[x][y]) : 0.f;
                    part += w[x][y];
                }
                part += __shfl_xor_sync(0xffffffffu, part, 8);
                part += __shfl_xor_sync(0xffffffffu, part, 16);
                wsacc[x] += part;  // this half's 16 keys
            }
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                *reinterpret_cast<float4*>(Wt + (key0 + y) * kQKRows + row0) =
                    make_float4(w[0][y], w[1][y], w[2][y], w[3][y]);
                *reinterpret_cast<float4*>(Wt + (key0 + y) * kQKRows + row0 + 32) =
                    make_float4(w[4][y], w[5][y], w[6][y], w[7][y]);
            }
            __syncthreads();
            // acc += w V for 8 rows x 8 channels
#pragma unroll 4
            for (int t = 0; t < kQKKeys; ++t) {
                const float4 w0 = ld4(Wt + t * kQKRows + row0);
                const float4 w1 = ld4(Wt + t * kQKRows + row0 + 32);
                const float4 v0 = ld4(Vt + t * kHd + ch0);
                const float4 v1 = ld4(Vt + t * kHd + ch0 + 4);
                const float wr[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                const float vr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int x = 0; x < 8; ++x)
#pragma unroll
                    for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(wr[x], vr[y], acc[x][y]);
            }
        }
        // W_s from both halves' partial sums, then <E, dO> over this thread's channels
        if (q == 0) {
#pragma unroll
            for (int x = 0; x < 8; ++x) wsp[hb * kQKRows + row0 + qk_row(x)] = wsacc[x];
        }
        __syncthreads();
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            const float W = wsp[row0 + qk_row(x)] + wsp[kQKRows + row0 + qk_row(x)];
            const int64_t off = (tok0 + row0 + qk_row(x)) * C + h * kHd + ch0;
            const float4 o0 = ld4(a.O + off), o1 = ld4(a.O + off + 4);
            const float4 e0 = ld4(a.E + off), e1 = ld4(a.E + off + 4);
            const float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
            const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
            float eo = 0.f;
#pragma unroll
            for (int y = 0; y < 8; ++y) eo = fmaf(ev[y], fmaf(-W, ov[y], acc[x][y]), eo);
            eo += __shfl_xor_sync(0xffffffffu, eo, 8);
            eo += __shfl_xor_sync(0xffffffffu, eo, 16);
            dlr[x] += eo / (1.0f + W);  // this half's 32 channels
        }
        __syncthreads();  // wsp and At are rewritten by the next head
    }
    if (q == 0) {
#pragma unroll
        for (int x = 0; x < 8; ++x) dlp[hb * kQKRows + row0 + qk_row(x)] = dlr[x];
    }
    __syncthreads();
    if (tid < kQKRows)
        a.dl[static_cast<int64_t>(i) * a.T + tok0 + tid] = dlp[tid] + dlp[kQKRows + tid];
}

std::atomic<uint64_t> qk_smem_set[2];

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
        !aligned(P, 16) || !aligned(E, 16) || (g_hat && !aligned(g_hat, 16)))
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
    DUST_CUDA_TRY(which == 1 ? set_smem_once(attn_qk_kernel<true>, kQKSmemBytes, qk_smem_set[1])
                             : set_smem_once(attn_qk_kernel<false>, kQKSmemBytes, qk_smem_set[0]));
    timer_begin(s);
    if (which == 1)
        attn_qk_kernel<true><<<grid, kQKThreads, kQKSmemBytes, s>>>(qa, keys);
    else
        attn_qk_kernel<false><<<grid, kQKThreads, kQKSmemBytes, s>>>(qa, keys);
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
