// attention.cu -- perturbation inside attention: the values, scored by the
// attention-output error.
//
// The pages treat perturbations inside attention apart from the other linear
// layers: they barely move their own token's loss but are read by later
// tokens through attention, so they are scored by the error of the attention
// output, and later tokens' scores are discounted by a gamma close to 1 (Dust
// translation, §2.3; laoyaoba.com, section 机制拆解; yomxxx.com post).  For
// the values v_t = W_v x_t of one attention layer with cached clean
// probabilities P (per sequence and head, causal), perturbing every token's
// value by sigma a_t changes the outputs exactly linearly:
//   dO_s = sigma sum_{t <= s} P_{s,t} a_t          (per head),
// and with E the attention-output error estimate the loss change of token s is
// read to first order as dl_s = <E_s, dO_s> (over all heads).  From there the
// method is the usual one: c = -(dl - mean over draws), r_t = sum_{s >= t}
// gamma^(s-t) c_s per sequence, g_t = -(1/(K sigma)) sum_i r a, G = g^T x.
//
// Per group of four draws the noise of every (sequence, head) is written
// once as split bf16 [hi | lo] (keys along the row), and one tcgen05 kernel
// computes, for 128 queries x (4 draws x 64 channels), P A over the causal key
// range with P = [P_hi | P_lo] and A = [A_hi | A_lo] from TMA, every key
// slice bringing all four halves so that the three products hi.hi, hi.lo and
// lo.hi are issued back to back (the dropped lo.lo term is below 2^-16
// relative) and each byte is read once per tile, and
// reduces the accumulator rows against E in its epilogue, so dO never leaves
// the chip.  The credit and the error estimate reuse the interior layer's
// kernels.
#include <cudaTypedefs.h>

#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {

bool encode_bf16_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                    int64_t stride_elems, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int kDv = 64;           // channels per head
constexpr int kGroup = 4;         // draws per kernel launch (N = 4 x 64)
constexpr int kQM = 128;          // queries per tile
constexpr int kKB = 64;           // keys per stage
constexpr int kNB = kGroup * kDv; // 256
constexpr int kStages = 2;
constexpr uint32_t kABytes = kQM * kKB * 2;   // 16 KB
constexpr uint32_t kBBytes = kNB * kKB * 2;   // 32 KB
// one stage = a 64-key slice of P_hi, P_lo, A_hi and A_lo
constexpr uint32_t kStageBytes = 2 * kABytes + 2 * kBBytes;
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + 256;

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
    __nv_bfloat162 h = __halves2bfloat162(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// P (fp32, rows of L keys) -> [P_hi | P_lo] bf16 rows of 2L, zero above the
// diagonal (keys after the query).
__global__ void attn_split_p_kernel(const float* __restrict__ P, int64_t rows, int L,
                                    __nv_bfloat16* __restrict__ P2) {
    const int64_t n4 = rows * (L / 4);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / (L / 4);
        const int t0 = static_cast<int>(i - row * (L / 4)) * 4;
        const int s = static_cast<int>(row % L);
        if (!DUST_IB(row * L + t0 + 3, rows * L)) continue;
        const float4 v = __ldg(reinterpret_cast<const float4*>(P + row * L + t0));
        float x[4] = {v.x, v.y, v.z, v.w};
        __nv_bfloat16 hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = t0 + k <= s ? x[k] : 0.f;
            hi[k] = __float2bfloat16_rn(p);
            lo[k] = __float2bfloat16_rn(p - __bfloat162float(hi[k]));
        }
        __nv_bfloat16* out = P2 + row * (2 * static_cast<int64_t>(L));
        *reinterpret_cast<uint2*>(out + t0) =
            make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
        *reinterpret_cast<uint2*>(out + L + t0) =
            make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
    }
}

struct NoiseArgs {
    int nseq, H, L, nd;
    uint32_t draw_first, token0, layer;
    __nv_bfloat16* N2;  // rows ((sq H + h) 4 + d) 64 + ch, 2L columns [hi | lo]
};

// The group's value noise: grid.y = (sequence, head, draw), threads over
// (channel block of four, pair of keys) with keys fastest, so that each row's
// stores are contiguous across a warp and two keys' values go out as one
// 4-byte bf16 pair.  Draws past the group's count get zeros.
__global__ void __launch_bounds__(256) attn_noise_kernel(const NoiseArgs a, const PhiloxKeys keys) {
    const int y = blockIdx.y;  // (sq H + h) kGroup + d
    const int d = y % kGroup;
    const int sh = y / kGroup;
    const int h = sh % a.H;
    const int sq = sh / a.H;
    const int half_l = a.L / 2;
    const int per = (kDv / 4) * half_l;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < per; i += gridDim.x * blockDim.x) {
        const int jb = i / half_l;
        const int t = 2 * (i - jb * half_l);
        float4 n0 = make_float4(0.f, 0.f, 0.f, 0.f), n1 = n0;
        if (d < a.nd) {
            const uint32_t j = static_cast<uint32_t>(h * (kDv / 4) + jb);
            const uint32_t token = a.token0 + static_cast<uint32_t>(sq * a.L + t);
            const BlockHalf bh = philox_block_half(j, a.layer, keys);
            const uint32_t draw = a.draw_first + d;
            n0 = words_to_normals_fast(philox_rest(philox_draw_half(draw, token, keys), bh, keys));
            n1 = words_to_normals_fast(philox_rest(philox_draw_half(draw, token + 1, keys), bh, keys));
        }
        const float v0[4] = {n0.x, n0.y, n0.z, n0.w}, v1[4] = {n1.x, n1.y, n1.z, n1.w};
        const int64_t row0 = static_cast<int64_t>(y) * kDv + jb * 4;
        const int64_t n2_ext =
            static_cast<int64_t>(a.nseq) * a.H * kGroup * kDv * (2 * static_cast<int64_t>(a.L));
        if (!DUST_IB((row0 + 3) * (2 * static_cast<int64_t>(a.L)) + a.L + t + 1, n2_ext)) continue;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat16* out = a.N2 + (row0 + k) * (2 * static_cast<int64_t>(a.L));
            const __nv_bfloat16 h0 = __float2bfloat16_rn(v0[k]), h1 = __float2bfloat16_rn(v1[k]);
            *reinterpret_cast<uint32_t*>(out + t) = pack_bf16x2(h0, h1);
            *reinterpret_cast<uint32_t*>(out + a.L + t) =
                pack_bf16x2(__float2bfloat16_rn(v0[k] - __bfloat162float(h0)),
                            __float2bfloat16_rn(v1[k] - __bfloat162float(h1)));
        }
    }
}

struct AttnArgs {
    const float* E;  // T x C attention-output error, C = H 64
    float* dlh;      // K x H x T: sigma <E_s, dO_s> per head
    int T, L, H, nd, i0;
    float sigma;
    uint32_t* status;
};

// One CTA: query tile qb of sequence sq, head h (grid.x = tiles, heaviest
// first; grid.y = sq H + h).  Warp 0 streams the four halves of each 64-key
// slice by TMA, warp 1 issues the three split products of each slice into one
// 256-column accumulator, warps 2..5 reduce each query row against E.
__global__ void __launch_bounds__(192, 1)
    attn_v_kernel(const __grid_constant__ CUtensorMap tp, const __grid_constant__ CUtensorMap tn,
                  const AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t bars = base + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    const uint32_t acc_bar = bars + 16u * kStages;
    const uint32_t tmem_slot = acc_bar + 8u;
    volatile uint32_t* tmem_slot_gen =
        reinterpret_cast<volatile uint32_t*>(base_gen + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ntq = a.L / kQM;
    const int qb = ntq - 1 - static_cast<int>(blockIdx.x);
    const int sh = blockIdx.y;  // sq H + h
    const int h = sh % a.H;
    const int sq = sh / a.H;
    const int nit = 2 * (qb + 1);  // 64-key slices up to the tile's last query

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        mbar_fence_init();
        tma_prefetch_desc(&tp);
        tma_prefetch_desc(&tn);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot_gen;

    if (warp == 0) {
        if (lane == 0) {
            const int prow = sh * a.L + qb * kQM;
            const int nrow = sh * kNB;
            for (int it = 0; it < nit; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                if (it >= kStages && !mbar_wait(empty_bar(s), ph ^ 1u, a.status)) break;
                const int key0 = it * kKB;
                mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                const uint32_t dst = base + s * kStageBytes;
                tma_load_2d(dst, &tp, key0, prow, full_bar(s));                    // P_hi
                tma_load_2d(dst + kABytes, &tp, a.L + key0, prow, full_bar(s));    // P_lo
                tma_load_2d(dst + 2 * kABytes, &tn, key0, nrow, full_bar(s));      // A_hi
                tma_load_2d(dst + 2 * kABytes + kBBytes, &tn, a.L + key0, nrow,    // A_lo
                            full_bar(s));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kQM, kNB, false, false);
            bool ok = true;
            for (int it = 0; it < nit; ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                if (!mbar_wait(full_bar(s), ph, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pa = base + s * kStageBytes;  // P_hi, then P_lo
                const uint32_t na = pa + 2 * kABytes;        // A_hi, then A_lo
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk) {
                    const uint64_t ph_d = sdesc_sw128(pa + kk * 32u, 16u, 1024u);
                    const uint64_t pl_d = sdesc_sw128(pa + kABytes + kk * 32u, 16u, 1024u);
                    const uint64_t nh_d = sdesc_sw128(na + kk * 32u, 16u, 1024u);
                    const uint64_t nl_d = sdesc_sw128(na + kBBytes + kk * 32u, 16u, 1024u);
                    umma_bf16(tmem, ph_d, nh_d, idesc, (it | kk) != 0 ? 1u : 0u);
                    umma_bf16(tmem, ph_d, nl_d, idesc, 1u);
                    umma_bf16(tmem, pl_d, nh_d, idesc, 1u);
                }
                umma_commit(empty_bar(s));
            }
            (void)ok;
            umma_commit(acc_bar);  // also on failure, so the epilogue never waits forever
        }
    } else {
        // Epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = query rows.
        const int quarter = warp & 3;
        const int rit = quarter * 32 + lane;
        const int tg = sq * a.L + qb * kQM + rit;  // token
        bool ok = mbar_wait(acc_bar, 0, a.status);
        ok = __all_sync(0xFFFFFFFFu, ok);
        tc_fence_after();
        // (the TMEM loads below are warp-collective; the check skips the whole row set)
        if (ok && DUST_IB(static_cast<int64_t>(tg) * (a.H * kDv) + h * kDv + kDv - 1,
                          static_cast<int64_t>(a.T) * (a.H * kDv))) {
            const float* erow = a.E + static_cast<int64_t>(tg) * (a.H * kDv) + h * kDv;
            float acc[kGroup] = {0.f, 0.f, 0.f, 0.f};
            // accumulator columns: draw d, channels 32 half .. + 31
#pragma unroll
            for (int d = 0; d < kGroup; ++d) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                           (2 * d + half) * 32,
                                       r);
                    tmem_wait_ld();
                    const float4* e4 = reinterpret_cast<const float4*>(erow + half * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 e = __ldg(e4 + q);
                        acc[d] = fmaf(e.x, __uint_as_float(r[4 * q]), acc[d]);
                        acc[d] = fmaf(e.y, __uint_as_float(r[4 * q + 1]), acc[d]);
                        acc[d] = fmaf(e.z, __uint_as_float(r[4 * q + 2]), acc[d]);
                        acc[d] = fmaf(e.w, __uint_as_float(r[4 * q + 3]), acc[d]);
                    }
                }
            }
#pragma unroll
            for (int d = 0; d < kGroup; ++d)
                if (d < a.nd && DUST_IB((static_cast<int64_t>(a.i0 + d) * a.H + h) * a.T + tg,
                                        static_cast<int64_t>(a.i0 + a.nd) * a.H * a.T))
                    a.dlh[(static_cast<int64_t>(a.i0 + d) * a.H + h) * a.T + tg] = a.sigma * acc[d];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// dl[i][t] = sum over heads of dlh[i][h][t], heads in order.
__global__ void attn_head_sum_kernel(const float* __restrict__ dlh, int K, int H, int T,
                                     float* __restrict__ dl) {
    const int64_t n = static_cast<int64_t>(K) * T;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t k = i / T, t = i - k * T;
        float s = 0.f;
        for (int h = 0; h < H; ++h)
            if (DUST_IB((k * H + h) * T + t, n * H)) s += dlh[(k * H + h) * T + t];
        dl[i] = s;
    }
}

struct AttnPlan {
    int64_t ldx;
    size_t off_p2, off_n2, off_dlh, off_dl, off_m, off_r, off_gbf, off_xbf, bytes;
};

AttnPlan attn_plan(int64_t T, int64_t L, int64_t H, int64_t d_in, uint32_t K) {
    AttnPlan P{};
    const int64_t nseq = T / L, C = H * kDv;
    P.ldx = round_up(d_in, 8);
    WsLayout w;
    w.take(kCtlBytes);
    P.off_p2 = w.take(static_cast<size_t>(nseq * H * L) * static_cast<size_t>(2 * L) * 2);
    P.off_n2 = w.take(static_cast<size_t>(nseq * H * kNB) * static_cast<size_t>(2 * L) * 2);
    P.off_dlh = w.take(static_cast<size_t>(K) * H * T * 4);
    P.off_dl = w.take(static_cast<size_t>(K) * T * 4);
    P.off_m = w.take(static_cast<size_t>(T) * 4);
    P.off_r = w.take(static_cast<size_t>(K) * T * 4);
    P.off_gbf = w.take(static_cast<size_t>(T * C) * 2);
    P.off_xbf = w.take(static_cast<size_t>(T * P.ldx) * 2);
    P.bytes = w.used;
    return P;
}

unsigned blocks_for(int64_t n, int threads) {
    int64_t b = ceil_div(n, threads);
    if (b > 148 * 16) b = 148 * 16;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" size_t dust_attn_value_workspace(int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                                            int64_t d_in, uint32_t K) {
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || H < 1 || dv != kDv || d_in < 1 || K < 2)
        return 0;
    return attn_plan(T, seq_len, H, d_in, K).bytes;
}

dust_status dust::attn_value_check(const float* P, const float* E, const void* x,
                                   dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t H,
                                   int64_t dv, int64_t d_in, const dust_noise& nz,
                                   const float* g_hat, const float* G_W, const void* ws,
                                   size_t ws_bytes) {
    if (!P || !E || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || H < 1 || d_in < 1) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (nz.num_draws < 2 || !(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (!(nz.gamma >= 0.0f && nz.gamma <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (dv != kDv || seq_len % kQM != 0 || seq_len > 8192 || H > 64 || T / seq_len * H > 16383 ||
        T > (1LL << 26) ||
        d_in > (1LL << 20) || nz.num_draws > (1u << 20))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32) ||
        static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (!aligned(P, 16) || !aligned(E, 16) || (g_hat && !aligned(g_hat, 16)))
        return DUST_ERR_INVALID_ARG;
    const AttnPlan Pl = attn_plan(T, seq_len, H, d_in, nz.num_draws);
    if (!ws || ws_bytes < Pl.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

extern "C" dust_status dust_attn_value_estimate(const float* P, const float* E, const void* x,
                                                dust_dtype x_dtype, int64_t T, int64_t seq_len,
                                                int64_t H, int64_t dv, int64_t d_in,
                                                dust_noise nz, float* g_hat, float* G_W,
                                                void* ws, size_t ws_bytes, void* stream) {
    const dust_status chk = attn_value_check(P, E, x, x_dtype, T, seq_len, H, dv, d_in, nz, g_hat,
                                             G_W, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const AttnPlan Pl = attn_plan(T, seq_len, H, d_in, nz.num_draws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint32_t* status = static_cast<uint32_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));

    const int L = static_cast<int>(seq_len), Hi = static_cast<int>(H), Ti = static_cast<int>(T);
    const int64_t nseq = T / seq_len, C = H * kDv;
    const int K = static_cast<int>(nz.num_draws);
    __nv_bfloat16* P2 = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_p2);
    __nv_bfloat16* N2 = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_n2);
    float* dlh = reinterpret_cast<float*>(w + Pl.off_dlh);
    float* dl = reinterpret_cast<float*>(w + Pl.off_dl);
    float* mean = reinterpret_cast<float*>(w + Pl.off_m);
    float* r = reinterpret_cast<float*>(w + Pl.off_r);
    __nv_bfloat16* gbf = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_gbf);
    const PhiloxKeys keys = philox_round_keys(nz.seed);

    const int64_t prows = nseq * H * seq_len;
    attn_split_p_kernel<<<blocks_for(prows * (seq_len / 4), 256), 256, 0, s>>>(P, prows, L, P2);
    dust_status st = launch_status();
    if (st != DUST_OK) return st;

    CUtensorMap tp, tn;
    if (!encode_bf16_2d(&tp, P2, 2 * seq_len, prows, 2 * seq_len, kKB, kQM) ||
        !encode_bf16_2d(&tn, N2, 2 * seq_len, nseq * H * kNB, 2 * seq_len, kKB, kNB))
        return DUST_ERR_CUDA;
    static std::atomic<uint64_t> smem_set{0};
    DUST_CUDA_TRY(set_smem_once(attn_v_kernel, static_cast<int>(kSmemBytes), smem_set));
    const dim3 grid(static_cast<unsigned>(seq_len / kQM), static_cast<unsigned>(nseq * H));
    for (int i0 = 0; i0 < K; i0 += kGroup) {
        const int nd = K - i0 < kGroup ? K - i0 : kGroup;
        NoiseArgs na{static_cast<int>(nseq), Hi, L, nd, nz.draw0 + static_cast<uint32_t>(i0),
                     nz.token0, nz.layer, N2};
        const dim3 ng(static_cast<unsigned>(ceil_div((kDv / 4) * seq_len / 2, 256)),
                      static_cast<unsigned>(nseq * H * kGroup));
        attn_noise_kernel<<<ng, 256, 0, s>>>(na, keys);
        if ((st = launch_status()) != DUST_OK) return st;
        AttnArgs aa{E, dlh, Ti, L, Hi, nd, i0, nz.sigma, status};
        timer_begin(s);
        attn_v_kernel<<<grid, 192, kSmemBytes, s>>>(tp, tn, aa);
        timer_end(s);
        if ((st = launch_status()) != DUST_OK) return st;
    }
    attn_head_sum_kernel<<<blocks_for(static_cast<int64_t>(K) * T, 256), 256, 0, s>>>(dlh, K, Hi,
                                                                                     Ti, dl);
    if ((st = launch_status()) != DUST_OK) return st;
    st = credit_and_ghat_launch(dl, mean, r, Ti, L, static_cast<int>(C), nz, keys, g_hat, gbf, s);
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

// ------------------------------------------------------------------------
// Gates of the attention output, the other elementwise member of the
// attention internals the pages list (Dust translation §2.3): the gated
// output is sig(z_s) * o_s per channel with z_s = W_g x_s.  Perturbing every
// token's gate pre-activation changes only its own gated output,
//   d(o~)_s = (sig(z_s + sigma a_s) - sig(z_s)) * o_s,
// and it is scored, like the values, by the error E of the gated output:
// dl_s = <E_s, d(o~)_s>.  sig(z + d) - sig(z) = sig(z + d) (1 - sig(z))
// (1 - e^-d) has no cancellation for small d.
// ------------------------------------------------------------------------
namespace dust {
namespace {

struct GateArgs {
    const float* z;  // T x C gate pre-activations
    const float* o;  // T x C attention output before the gate
    const float* E;  // T x C error of the gated output
    float* dl;       // K x T
    int T, C, K;
    uint32_t draw0, token0, layer;
    float sigma;
};

// One warp per token; each lane owns channel blocks lane, lane + 32, ... and
// the warp sums its lanes by shuffles, draw after draw.
__global__ void __launch_bounds__(256) attn_gate_dl_kernel(const GateArgs a, const PhiloxKeys keys) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= a.T) return;
    const int nblk = a.C / 4;
    const int64_t row = static_cast<int64_t>(t) * a.C;
    const uint32_t token = a.token0 + static_cast<uint32_t>(t);
    for (int i = 0; i < a.K; ++i) {
        const DrawHalf dh = philox_draw_half(a.draw0 + static_cast<uint32_t>(i), token, keys);
        float part = 0.f;
        for (int j = lane; j < nblk; j += 32) {
            if (!DUST_IB(row + 4 * j + 3, static_cast<int64_t>(a.T) * a.C)) break;
            const float4 n = words_to_normals_fast(philox_rest(dh, philox_block_half(j, a.layer, keys), keys));
            const float4 z = __ldg(reinterpret_cast<const float4*>(a.z + row) + j);
            const float4 o = __ldg(reinterpret_cast<const float4*>(a.o + row) + j);
            const float4 e = __ldg(reinterpret_cast<const float4*>(a.E + row) + j);
            const float zz[4] = {z.x, z.y, z.z, z.w}, oo[4] = {o.x, o.y, o.z, o.w};
            const float ee[4] = {e.x, e.y, e.z, e.w}, nn[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float d = a.sigma * nn[k];
                const float s1 = 1.0f / (1.0f + expf(-(zz[k] + d)));
                const float s0c = 1.0f / (1.0f + expf(zz[k]));  // 1 - sig(z)
                part = fmaf(ee[k] * oo[k], s1 * s0c * -expm1f(-d), part);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
        if (lane == 0 && DUST_IB(static_cast<int64_t>(i) * a.T + t, static_cast<int64_t>(a.K) * a.T))
            a.dl[static_cast<int64_t>(i) * a.T + t] = part;
    }
}

struct GatePlan {
    int64_t ldx;
    size_t off_dl, off_m, off_r, off_gbf, off_xbf, bytes;
};

GatePlan gate_plan(int64_t T, int64_t C, int64_t d_in, uint32_t K) {
    GatePlan P{};
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

extern "C" size_t dust_attn_gate_workspace(int64_t T, int64_t seq_len, int64_t C, int64_t d_in,
                                           uint32_t K) {
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || C < 8 || C % 8 != 0 || d_in < 1 || K < 2)
        return 0;
    return gate_plan(T, C, d_in, K).bytes;
}

dust_status dust::attn_gate_check(const float* z, const float* o, const float* E, const void* x,
                                  dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t C,
                                  int64_t d_in, const dust_noise& nz, const float* g_hat,
                                  const float* G_W, const void* ws, size_t ws_bytes) {
    if (!z || !o || !E || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || C < 1 || d_in < 1) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (nz.num_draws < 2 || !(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (!(nz.gamma >= 0.0f && nz.gamma <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (C % 8 != 0 || T > (1LL << 28) || C > (1LL << 16) || d_in > (1LL << 20) ||
        nz.num_draws > (1u << 24))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32) ||
        static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (!aligned(z, 16) || !aligned(o, 16) || !aligned(E, 16) || (g_hat && !aligned(g_hat, 16)))
        return DUST_ERR_INVALID_ARG;
    const GatePlan Pl = gate_plan(T, C, d_in, nz.num_draws);
    if (!ws || ws_bytes < Pl.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

extern "C" dust_status dust_attn_gate_estimate(const float* z, const float* o, const float* E,
                                               const void* x, dust_dtype x_dtype, int64_t T,
                                               int64_t seq_len, int64_t C, int64_t d_in,
                                               dust_noise nz, float* g_hat, float* G_W, void* ws,
                                               size_t ws_bytes, void* stream) {
    const dust_status chk = attn_gate_check(z, o, E, x, x_dtype, T, seq_len, C, d_in, nz, g_hat,
                                            G_W, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const GatePlan Pl = gate_plan(T, C, d_in, nz.num_draws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint32_t* status = static_cast<uint32_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    float* dl = reinterpret_cast<float*>(w + Pl.off_dl);
    float* mean = reinterpret_cast<float*>(w + Pl.off_m);
    float* r = reinterpret_cast<float*>(w + Pl.off_r);
    __nv_bfloat16* gbf = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_gbf);
    const PhiloxKeys keys = philox_round_keys(nz.seed);

    GateArgs ga{z, o, E, dl, static_cast<int>(T), static_cast<int>(C),
                static_cast<int>(nz.num_draws), nz.draw0, nz.token0, nz.layer, nz.sigma};
    timer_begin(s);
    attn_gate_dl_kernel<<<static_cast<unsigned>(ceil_div(T, 8)), 256, 0, s>>>(ga, keys);
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

namespace dust {
DUST_DEBUG_READER(6)
}  // namespace dust
