// reforward.cu -- the first contraction of the interior layer's re-forward,
// with its A operand generated on chip.
//
// A draw perturbs the layer output y1 and only the part after the layer is
// re-run (laoyaoba.com article, section 机制拆解; Dust translation,
// hn.213312.xyz, §2.3).  The first step after the layer is
//   du = dh W2^T,  dh = GELU(y1 + sigma a) - GELU(y1),
// with the noise a regenerated from its counter.  Instead of writing dh to
// memory and reading it back, producer warps compute each 128-token x
// 64-channel slice of dh, split it into bf16 hi and lo halves and store both
// straight into shared memory in the 128-byte-swizzled K-major layout the
// tensor cores read; W2's matching slice arrives by TMA.  One thread issues
// tcgen05.mma for hi and lo into the same fp32 accumulator in tensor memory
// (d_model <= 512 columns), so dh never leaves the chip and the noise and GELU
// arithmetic overlaps the MMAs of the previous slice.
//
// Rows are ordered (token block of 128, draw, token in block) like the rest of
// the interior pipeline; the output du (rows x d_model fp32) feeds the EMA.
#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"
#include "gelu.cuh"

namespace dust {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kStages = 2;
constexpr int kProducerWarps = 16;
constexpr int kThreads = 32 * (2 + kProducerWarps);
constexpr uint32_t kATile = kBM * kBK * 2;           // 16 KB per half
constexpr uint32_t kBTile = 512 * kBK * 2;           // 64 KB: up to 512 rows of W2
constexpr uint32_t kStageBytes = 2 * kATile + kBTile;  // 96 KB
constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + 256;

struct RefArgs {
    const float* y1;  // T x C
    const float* h0;  // T x C: GELU(y1) (exact path)
    const void* coef;    // Taylor coefficients of the GELU difference (GeluCoefs layout)
    int taylor;          // use the Taylor form (small sigma)
    float* du;        // rows x dm (plain epilogue)
    __nv_bfloat16* A2;  // rows x 2 dm: [hi | lo] of the EMA output (EMA epilogue)
    int T, C, dm, nd;
    int64_t rows;  // rows of du / A2: nd x the token count rounded up to a tile
    int ema;    // 1: work item = (sequence, draw), EMA in the epilogue
    int tiles;  // token blocks per sequence (EMA epilogue)
    float lam;  // EMA decay
    uint32_t draw_first, token0, layer;
    float sigma;
    float clog;  // the fast Box-Muller's constant for normals scaled by sigma
    uint32_t* status;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Named barrier over the 128 threads of one epilogue column group.
__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// True on every producer thread iff `ok` holds on all of them (barrier 5 over
// the producer warps only).
__device__ __forceinline__ bool producers_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, 5, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "n"(32 * kProducerWarps)
        : "memory");
    return r != 0;
}

// Barrier 6 over the producer warps only.
__device__ __forceinline__ void producers_sync() {
    asm volatile("bar.sync 6, %0;" ::"n"(32 * kProducerWarps) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    reforward1_kernel(const __grid_constant__ CUtensorMap tw2, const RefArgs a,
                      const PhiloxKeys keys) {
    extern __shared__ uint8_t smem_raw[];
    // EMA epilogue: end values of each quarter's walk from zero (two chunk
    // parities) and the carry into the next tile (two tile parities).
    __shared__ float s_end[2][4][4][32];
    __shared__ float s_carry[2][512];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t bars = base + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    const uint32_t acc_bar = bars + 16u * kStages;
    const uint32_t tmem_empty = acc_bar + 8u;
    const uint32_t tmem_slot = acc_bar + 16u;
    volatile uint32_t* tmem_slot_gen =
        reinterpret_cast<volatile uint32_t*>(base_gen + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nk = a.C / kBK;
    const int ngroups = (a.dm + 255) / 256;
    const uint32_t b_bytes = static_cast<uint32_t>(ngroups) * 256u * kBK * 2u;
    // Work item: one 128-row tile, or (EMA epilogue) the `tiles` token blocks
    // of one sequence for one draw, in token order.
    const int ntiles = a.ema ? a.tiles : 1;
    const int di = static_cast<int>(blockIdx.x) % a.nd;
    const int tb0 = a.ema ? (static_cast<int>(blockIdx.x) / a.nd) * a.tiles
                          : static_cast<int>(blockIdx.x) / a.nd;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 32 * kProducerWarps + 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        mbar_init(tmem_empty, kProducerWarps);
        mbar_fence_init();
        tma_prefetch_desc(&tw2);
    }
    for (int i = threadIdx.x; i < 512; i += blockDim.x) s_carry[0][i] = 0.f;
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot_gen;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int k = 0; k < ntiles; ++k) {
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (it >= kStages && !mbar_wait(empty_bar(s), ph ^ 1u, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), b_bytes);
                    const uint32_t b_dst = base + s * kStageBytes + 2 * kATile;
                    for (int g = 0; g < ngroups; ++g)
                        tma_load_2d(b_dst + g * (256u * kBK * 2u), &tw2, kb * kBK, g * 256,
                                    full_bar(s));
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, 256, false, false);
            int it = 0;
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k) {
                // The accumulator is reused: wait until the previous tile's
                // epilogue has read it.
                if (k > 0) {
                    if (!mbar_wait(tmem_empty, (k - 1) & 1, a.status)) break;
                    tc_fence_after();
                }
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(full_bar(s), ph, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + s * kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint64_t ad = sdesc_sw128(st + h * kATile + kk * 32u, 16u, 1024u);
                            for (int g = 0; g < ngroups; ++g) {
                                const uint64_t bd = sdesc_sw128(
                                    st + 2 * kATile + g * (256u * kBK * 2u) + kk * 32u, 16u, 1024u);
                                umma_bf16(tmem + g * 256, ad, bd, idesc,
                                          (kb | kk | h) != 0 ? 1u : 0u);
                            }
                        }
                    }
                    umma_commit(empty_bar(s));
                }
                if (ok) umma_commit(acc_bar);
            }
        }
    } else {
        // Producers: thread p owns channel block jj = p % 16 of the slice and
        // rows p / 16 + R m, R = 2 kProducerWarps.
        const int p = threadIdx.x - 64;
        const int jj = p & 15;
        const int r0 = p >> 4;  // 0 .. 2 kProducerWarps - 1
        constexpr int kRows = kBM / (2 * kProducerWarps);  // rows per thread
        // EMA epilogue constants: 1 - lam and lam^32 (one quarter of a tile).
        const float one_m = 1.0f - a.lam;
        float l32 = a.lam;
#pragma unroll
        for (int i = 0; i < 5; ++i) l32 *= l32;

        bool ok = true;
        int it = 0;
        for (int k = 0; k < ntiles; ++k) {
            const int tb = tb0 + k;
            const int mt = tb * a.nd + di;
            // The (draw, token) halves of Philox's first two rounds are the same
            // for every slice of a row: computed once per tile.
            DrawHalf2 dhalf[kRows];
#pragma unroll
            for (int m = 0; m < kRows; ++m)
                dhalf[m] = philox_draw_half2(philox_draw_half(
                    a.draw_first + di, a.token0 + tb * kBM + r0 + 2 * kProducerWarps * m, keys));
            for (int kb = 0; kb < nk; ++kb, ++it) {
                if (!ok) continue;
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1u;
                if (it >= kStages && !mbar_wait(empty_bar(s), ph ^ 1u, a.status)) {
                    ok = false;
                    continue;
                }
                const uint32_t st = base + s * kStageBytes;
                const int j = kb * (kBK / 4) + jj;  // global channel block
                const BlockHalf2 bhalf = philox_block_half2(philox_block_half(j, a.layer, keys), keys);
                if (a.taylor) {
                    // dh = d (c1 + d (c2 + d c3)), d = sigma a per channel (the noise
                    // comes out scaled by sigma); the coefficients' loads of every row
                    // first, then the arithmetic.
                    const GeluCoefs cf = gelu_coefs(a.coef, static_cast<int64_t>(a.T) * (a.C / 4));
                    float4 c1v[kRows];
                    uint4 c23v[kRows];
#pragma unroll
                    for (int m = 0; m < kRows; ++m) {
                        const int t = tb * kBM + r0 + 2 * kProducerWarps * m;
                        const int64_t e4 = static_cast<int64_t>(t) * (a.C / 4) + j;
                        if (t < a.T && DUST_IB(e4, static_cast<int64_t>(a.T) * (a.C / 4))) {
                            c1v[m] = __ldg(cf.c1 + e4);
                            c23v[m] = __ldg(cf.c23 + e4);
                        } else {
                            c1v[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                            c23v[m] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    // The noise of every row before any use of the loads: their latency
                    // hides behind it (measured 9 % faster than row by row).
                    float4 ev[kRows];
#pragma unroll
                    for (int m = 0; m < kRows; ++m)
                        ev[m] = words_to_normals_fast(philox_rest2(dhalf[m], bhalf, keys), a.clog);
#pragma unroll
                    for (int m = 0; m < kRows; ++m) {
                        const int r = r0 + 2 * kProducerWarps * m;
                        const int t = tb * kBM + r;
                        uint32_t hi0 = 0, hi1 = 0, lo0 = 0, lo1 = 0;
                        if (t < a.T) {
                            float2 d01, d23;
                            gelu_taylor_pairs(c1v[m], c23v[m], ev[m], d01, d23);
                            split_pair2(d01, hi0, lo0);
                            split_pair2(d23, hi1, lo1);
                        }
                        const uint32_t off =
                            r * 128u + ((((jj >> 1) ^ (r & 7)) & 7u) << 4) + (jj & 1) * 8u;
                        st_shared_v2(st + off, hi0, hi1);
                        st_shared_v2(st + kATile + off, lo0, lo1);
                    }
                } else {
                    // Issue the loads of every row first, then the arithmetic.
                    float4 yv[kRows], gv[kRows];
#pragma unroll
                    for (int m = 0; m < kRows; ++m) {
                        const int t = tb * kBM + r0 + 2 * kProducerWarps * m;
                        if (t < a.T && DUST_IB(static_cast<int64_t>(t) * (a.C / 4) + j,
                                               static_cast<int64_t>(a.T) * (a.C / 4))) {
                            const int64_t e4 = static_cast<int64_t>(t) * (a.C / 4) + j;
                            yv[m] = __ldg(reinterpret_cast<const float4*>(a.y1) + e4);
                            gv[m] = __ldg(reinterpret_cast<const float4*>(a.h0) + e4);
                        } else {
                            yv[m] = gv[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                    }
                    float4 nv[kRows];  // the noise of every row first, as above
#pragma unroll
                    for (int m = 0; m < kRows; ++m)
                        nv[m] = words_to_normals_fast(philox_rest2(dhalf[m], bhalf, keys));
#pragma unroll
                    for (int m = 0; m < kRows; ++m) {
                        const int r = r0 + 2 * kProducerWarps * m;
                        const int t = tb * kBM + r;
                        uint32_t hi0 = 0, hi1 = 0, lo0 = 0, lo1 = 0;
                        if (t < a.T) {
                            // channel pairs (0, 1) and (2, 3) on packed fp32 pairs
                            const float4 nrm = nv[m];
                            const float4 y = yv[m], g = gv[m];
                            const float2 sg = make_float2(a.sigma, a.sigma);
                            const float2 d01 = sub2(
                                gelu_as2(fma2(sg, make_float2(nrm.x, nrm.y), make_float2(y.x, y.y))),
                                make_float2(g.x, g.y));
                            const float2 d23 = sub2(
                                gelu_as2(fma2(sg, make_float2(nrm.z, nrm.w), make_float2(y.z, y.w))),
                                make_float2(g.z, g.w));
                            split_pair2(d01, hi0, lo0);
                            split_pair2(d23, hi1, lo1);
                        }
                        // 128-byte swizzle: 16-byte chunk c of row r sits at c ^ (r & 7).
                        const uint32_t off =
                            r * 128u + ((((jj >> 1) ^ (r & 7)) & 7u) << 4) + (jj & 1) * 8u;
                        st_shared_v2(st + off, hi0, hi1);
                        st_shared_v2(st + kATile + off, lo0, lo1);
                    }
                }
                fence_async_shared();
                mbar_arrive(full_bar(s));
            }
            if (ok) ok = mbar_wait(acc_bar, static_cast<uint32_t>(k & 1), a.status);
            // Every producer thread takes the same branch from here on, so the
            // group barriers of the epilogue are reached by all or by none.
            if (!producers_all(ok)) break;
            tc_fence_after();
            // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (rows of the tile).
            const int quarter = warp & 3;
            const int rit = quarter * 32 + lane;
            const int64_t row = static_cast<int64_t>(mt) * kBM + rit;
            if (a.ema) {
                // de_t = lam de_{t-1} + (1 - lam) du_t along the tile's rows,
                // started from the previous tile's last row; kept as
                // f_t = de_t / (1 - lam) = lam f_{t-1} + du_t.  Column group cg
                // (four warps, one per quarter of the rows) takes 32-column
                // chunks cg, cg + 4, ...  Each warp stages its 32 x 32 block
                // in shared memory (the A operand buffers, idle until every
                // producer has left the epilogue), then lane j walks column j:
                // once from zero for the quarter's end value, and, once the
                // quarters' end values have given it its carry in, again from
                // that carry, writing A2 = [hi | lo] a row at a time.
                const int cg = (warp - 2) >> 2;
                const int wp = warp - 2;
                const int par = k & 1;
                float* sc = reinterpret_cast<float*>(base_gen + (wp >> 3) * kStageBytes +
                                                     (wp & 7) * 4096);
                // Row r, 16-byte piece i of the block sits at piece i ^ (r & 7).
                int off[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) off[c8] = (((lane >> 2) ^ c8) << 2) + (lane & 3);
                const int64_t row0 = static_cast<int64_t>(mt) * kBM + quarter * 32;
                for (int c = cg, n = 0; c < (a.dm >> 5); c += 4, ++n) {
                    const int col0 = c * 32;
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + col0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(sc + lane * 32 + ((i ^ (lane & 7)) << 2)) =
                            make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                        __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    __syncwarp();
                    float f = 0.f;
#pragma unroll
                    for (int r = 0; r < 32; ++r) f = fmaf(a.lam, f, sc[r * 32 + off[r & 7]]);
                    s_end[n & 1][cg][quarter][lane] = f;
                    group_sync(1 + cg);
                    float cin = s_carry[par][col0 + lane];
                    for (int qq = 0; qq < quarter; ++qq)
                        cin = fmaf(l32, cin, s_end[n & 1][cg][qq][lane]);
                    if (quarter == 3) s_carry[par ^ 1][col0 + lane] = fmaf(l32, cin, f);
                    __nv_bfloat16* out = a.A2 + row0 * (2 * a.dm) + col0 + lane;
                    f = cin;
#pragma unroll 8
                    for (int r = 0; r < 32; ++r) {
                        f = fmaf(a.lam, f, sc[r * 32 + off[r & 7]]);
                        const float e = one_m * f;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(e);
                        if (DUST_IB((row0 + r) * (2 * a.dm) + col0 + lane + a.dm,
                                    a.rows * (2 * a.dm))) {
                            out[0] = hi;
                            out[a.dm] = __float2bfloat16_rn(e - __bfloat162float(hi));
                        }
                        out += 2 * a.dm;
                    }
                    __syncwarp();
                }
            } else {
                // du rows: the first four producer warps take columns 0..255,
                // the next four 256..511.
                const int g = (warp - 2) >> 2;
                if (g < ngroups && g < 2) {
                    float* drow = a.du + row * a.dm;
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        const int col0 = g * 256 + c * 32;
                        if (col0 >= a.dm) break;
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + col0, v);
                        tmem_wait_ld();
                        // (the TMEM load above is warp-collective; only the stores are checked)
                        if (!DUST_IB(row * a.dm + col0 + 31, a.rows * a.dm)) continue;
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4*>(drow + col0 + q) =
                                make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                            __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
            // The next tile's A operand overwrites the staging blocks.
            if (a.ema) producers_sync();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

bool reforward1_supported(int64_t C, int64_t dm) {
    return C % kBK == 0 && dm % 32 == 0 && dm <= 512;
}

// Taylor coefficients of d -> GELU(y + d) - GELU(y) about d = 0, with G(k)
// the k-th derivative of GELU, phi the standard normal density and Phi its
// distribution function:
//   c1 = G(1) = Phi + y phi,   c2 = G(2)/2 = phi (2 - y^2) / 2,
//   c3 = G(3)/6 = phi (y^3 - 4y) / 6,
// written in the GeluCoefs layout (c1 fp32, c2 and c3 fp16).  They use CUDA's
// accurate erfcf/expf, once per call.  The dropped term is
// d^4 G(4)/24 = d^4 phi (7y^2 - y^4 - 4) / 24, at most 0.067 d^4; the host
// takes this path only when 5.77 sigma <= 0.15 (5.77 bounds |a|).
__global__ void gelu_taylor_kernel(const float* __restrict__ y1, int64_t nblk,
                                   void* __restrict__ coef) {
    float4* c1 = static_cast<float4*>(coef);
    uint4* c23 = reinterpret_cast<uint4*>(c1 + nblk);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 y4 = __ldg(reinterpret_cast<const float4*>(y1) + i);
        const float ys[4] = {y4.x, y4.y, y4.z, y4.w};
        float c[3][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float y = ys[k], y2 = y * y;
            const float phi = 0.39894228040143268f * expf(-0.5f * y2);
            const float Phi = 0.5f * erfcf(-y * 0.70710678118654752f);
            c[0][k] = fmaf(y, phi, Phi);
            c[1][k] = phi * (2.0f - y2) * 0.5f;
            c[2][k] = phi * (y * (y2 - 4.0f)) * (1.0f / 6.0f);
        }
        auto h2 = [](float a, float b) {
            __half2 h = __floats2half2_rn(a, b);
            return *reinterpret_cast<uint32_t*>(&h);
        };
        c1[i] = make_float4(c[0][0], c[0][1], c[0][2], c[0][3]);
        c23[i] = make_uint4(h2(c[1][0], c[1][1]), h2(c[1][2], c[1][3]), h2(c[2][0], c[2][1]),
                            h2(c[2][2], c[2][3]));
    }
}

dust_status gelu_taylor_launch(const float* y, int64_t n, void* coef, cudaStream_t s) {
    const int64_t nblk = n / 4;
    int64_t b = ceil_div(nblk, 256);
    if (b > 148 * 32) b = 148 * 32;
    gelu_taylor_kernel<<<static_cast<unsigned>(b < 1 ? 1 : b), 256, 0, s>>>(y, nblk, coef);
    return launch_status();
}

// h0[i] = GELU(y1[i]), the clean activation the perturbed one is compared with.
__global__ void gelu_kernel(const float* __restrict__ y, int64_t n, float* __restrict__ h) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        h[i] = gelu_as(y[i]);
}

dust_status gelu_launch(const float* y, int64_t n, float* h, cudaStream_t s) {
    int64_t b = ceil_div(n, 256);
    if (b > 148 * 32) b = 148 * 32;
    gelu_kernel<<<static_cast<unsigned>(b < 1 ? 1 : b), 256, 0, s>>>(y, n, h);
    return launch_status();
}

dust_status reforward1_launch(const float* y1, const float* h0, const void* coef, bool taylor,
                              const void* W2, int64_t T, int64_t Tp, int64_t C,
                              int64_t dm, int nd, uint32_t draw_first, uint32_t token0,
                              uint32_t layer, float sigma, const PhiloxKeys& keys, float* du,
                              void* A2, int64_t seq_len, float lam, uint32_t* status,
                              cudaStream_t s) {
    CUtensorMap tw2;
    if (!encode_bf16_2d(&tw2, W2, C, dm, C, kBK, 256)) return DUST_ERR_CUDA;
    static std::atomic<uint64_t> smem_set{0};
    DUST_CUDA_TRY(set_smem_once(reforward1_kernel, static_cast<int>(kSmemBytes), smem_set));
    const bool ema = A2 != nullptr;
    if (ema && (seq_len % kBM != 0 || Tp != T)) return DUST_ERR_UNSUPPORTED;
    RefArgs a{};
    a.y1 = y1;
    a.h0 = h0;
    a.coef = coef;
    a.taylor = taylor ? 1 : 0;
    a.du = du;
    a.A2 = static_cast<__nv_bfloat16*>(A2);
    a.T = static_cast<int>(T);
    a.C = static_cast<int>(C);
    a.dm = static_cast<int>(dm);
    a.nd = nd;
    a.rows = static_cast<int64_t>(nd) * Tp;
    a.ema = ema ? 1 : 0;
    a.tiles = ema ? static_cast<int>(seq_len / kBM) : 1;
    a.lam = lam;
    a.draw_first = draw_first;
    a.token0 = token0;
    a.layer = layer;
    a.sigma = sigma;
    a.clog = static_cast<float>(-2.0 * 0.69314718055994531 * static_cast<double>(sigma) * sigma);
    a.status = status;
    const unsigned grid = static_cast<unsigned>(ema ? nd * (T / seq_len) : nd * (Tp / kBM));
    reforward1_kernel<<<grid, kThreads, kSmemBytes, s>>>(tw2, a, keys);
    return launch_status();
}

}  // namespace dust

namespace dust {
DUST_DEBUG_READER(5)
}  // namespace dust
