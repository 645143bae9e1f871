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
// Both contractions run on the tensor cores (attn_qk_tc_kernel below); the
// exponential, P and the causal mask sit between them on the CUDA cores.  A
// CTA covers one tile of 128 queries of one sequence for one draw and walks
// the heads in order, so the per-token sum over heads needs no second pass;
// the draws are the fastest grid index, so the CTAs resident at one time share
// P and V (and, for the queries, K) through L2.
#include <algorithm>
#include <cudaTypedefs.h>

#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {

bool encode_bf16_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                    int64_t stride_elems, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int kHd = 64;       // channels per head
constexpr int kQKRows = 128;  // query rows per CTA

// e^x - 1 for the score shifts (in the slice loop below, on channel pairs):
// x (1 + x/2 + x^2/6 + x^3/24) for |x| < 1/8 (truncation about 2e-6 relative
// at x = 1/8 and 2.2e-6 at x = -1/8, under the 2^-16 of the bf16 split the
// result goes through next, and no cancellation), else expm1f.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// ------------------------------------------------------------------------
// Per 64-key slice, two split-bf16 tcgen05 products (hi.hi + hi.lo + lo.hi,
// fp32 accumulation in tensor memory):
//   ds[128 x 64] = A[128 x 64 ch] B_slice^T,   acc[128 x 64 ch] += W[128 x 64] V_slice,
//   W = P (e^ds - 1), causal.
// Queries: A = (sigma / 8) x the queries' noise, B = the clean keys.  Keys:
// A = (sigma / 8) x the clean queries, B = the keys' noise (written for a
// group of draws by qk_key_noise_kernel).  Warp 0 brings each slice's B
// ([hi | lo], keys x channels) and V^T ([hi | lo], channels x keys) by TMA,
// warp 1 issues the MMAs, and warps 2..17 (four per tensor-memory lane
// quarter, 16 keys or channels each) generate A per head, turn each ds slice
// into W in shared memory, and reduce acc against E at the end of a head.  ds has two tensor-memory buffers and W two shared-memory
// buffers, so the next slice's score product runs while this one's W is
// formed.  Every wait is bounded; on a timeout the roles stop and the status
// word records it.
// ------------------------------------------------------------------------
constexpr int kTcKeys = 64;                  // keys per slice
constexpr int kTcGroups = 4;                 // epilogue warps per lane quarter
constexpr int kTcCols = 64 / kTcGroups;      // keys (channels) per epilogue thread
constexpr int kTcEpi = 128 * kTcGroups;
constexpr int kTcThreads = 64 + kTcEpi;      // TMA, MMA, epilogue
constexpr uint32_t kT8 = 64u * 128u;         // 64 rows x 128 bytes
constexpr uint32_t kT16 = 128u * 128u;       // 128 rows x 128 bytes
// K slices ([hi | lo], 16 KB), V^T slices ([hi | lo], 16 KB) and the tile's
// P (128 queries x 32 keys fp32, 16 KB: a slice in two halves) come by TMA in
// rings of their own, so each is loaded ahead of the product or the epilogue
// step that needs it.  P arrives 128-byte swizzled: a thread reads its query's
// row as 16-byte pieces spread over the banks, where reading it from global
// memory would touch a different line per lane.
constexpr int kNK = 2;                       // K ring stages
constexpr int kNV = 2;                       // V ring stages
constexpr int kNP = 3;                       // P ring stages (half slices)
constexpr uint32_t kTcHalf = 2u * kT8;       // one K or V stage: hi and lo
constexpr uint32_t kTcOffV = kNK * kTcHalf;
constexpr uint32_t kTcOffP = kTcOffV + kNV * kTcHalf;
constexpr uint32_t kTcOffA = kTcOffP + kNP * kT16;  // A_hi, A_lo
constexpr uint32_t kTcOffW = kTcOffA + 2u * kT16;  // W[2] = {hi, lo} each
constexpr uint32_t kTcOffBar = kTcOffW + 4u * kT16;
constexpr uint32_t kTcSmem = kTcOffBar + 256u + 1024u;

struct QKTcArgs {
    const float* Q;  // clean queries (keys mode: the thread side of the scores)
    const float* P;
    const float* O;
    const float* E;
    float* dl;
    int T, L, H;
    int i0;  // first draw of this launch within the call (dl row)
    uint32_t draw0, token0, layer;
    float scale;
    uint32_t* status;
};

__device__ __forceinline__ void tc_fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kTcEpi) : "memory");
}
// True on every epilogue thread iff `ok` holds on all of them.
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n"
        " bar.red.and.pred p, 2, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "n"(kTcEpi)
        : "memory");
    return r != 0;
}
// 32 lanes x 16 consecutive 32-bit columns of tensor memory.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ uint32_t bf16_pair(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
// hi and lo bf16 pairs of (a, b): hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = bf16_pair(a - __low2float(h), b - __high2float(h));
}
// Byte offset of the 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(c ^ (r & 7)) & 7u) << 4);
}

// KEYS: A is the scaled clean queries and the score product's B operand is
// the keys' noise (tk then maps the group's noise, draw d at rows d T ..);
// otherwise A is the queries' noise and B the clean keys.
template <bool KEYS>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_qk_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tp, const QKTcArgs a,
                      const PhiloxKeys keys) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ float s_w[2][kTcGroups][kQKRows];  // row sums of w per head parity and key group
    __shared__ float s_dl[kTcGroups][kQKRows];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t bars = base + kTcOffBar;
    auto k_full = [&](int s) { return bars + 8u * s; };
    auto k_empty = [&](int s) { return bars + 8u * (kNK + s); };
    auto v_full = [&](int s) { return bars + 8u * (2 * kNK + s); };
    auto v_empty = [&](int s) { return bars + 8u * (2 * kNK + kNV + s); };
    auto p_full = [&](int s) { return bars + 8u * (2 * kNK + 2 * kNV + s); };
    auto p_empty = [&](int s) { return bars + 8u * (2 * kNK + 2 * kNV + kNP + s); };
    const uint32_t bars2 = bars + 8u * (2 * kNK + 2 * kNV + 2 * kNP);
    auto ds_full = [&](int b) { return bars2 + 8u * b; };
    auto ds_empty = [&](int b) { return bars2 + 16u + 8u * b; };
    auto w_full = [&](int b) { return bars2 + 32u + 8u * b; };
    auto w_empty = [&](int b) { return bars2 + 48u + 8u * b; };
    const uint32_t a_full = bars2 + 64u, acc_full = bars2 + 72u, acc_empty = bars2 + 80u;
    const uint32_t tmem_slot = bars2 + 88u;
    volatile uint32_t* tmem_slot_gen =
        reinterpret_cast<volatile uint32_t*>(base_gen + (tmem_slot - base));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nseq = a.T / a.L;
    const int qb = a.L / kQKRows - 1 - static_cast<int>(blockIdx.y) / nseq;  // heavy first
    const int sq = static_cast<int>(blockIdx.y) % nseq;
    const int i = a.i0 + static_cast<int>(blockIdx.x);
    const uint32_t draw = a.draw0 + static_cast<uint32_t>(i);
    const int ns = (qb + 1) * (kQKRows / kTcKeys);  // key slices per head
    const int krow0 = (KEYS ? static_cast<int>(blockIdx.x) * a.T : 0) + sq * a.L;  // B rows
    const int64_t tok0 = static_cast<int64_t>(sq) * a.L + qb * kQKRows;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNK; ++b) {
            mbar_init(k_full(b), 1);
            mbar_init(k_empty(b), 1);
        }
        for (int b = 0; b < kNV; ++b) {
            mbar_init(v_full(b), 1);
            mbar_init(v_empty(b), 1);
        }
        for (int b = 0; b < kNP; ++b) {
            mbar_init(p_full(b), 1);
            mbar_init(p_empty(b), kTcEpi / 2);  // the threads of one half of the keys
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(ds_full(b), 1);
            mbar_init(ds_empty(b), kTcEpi);
            mbar_init(w_full(b), kTcEpi);
            mbar_init(w_empty(b), 1);
        }
        mbar_init(a_full, kTcEpi);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kTcEpi);
        mbar_fence_init();
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&tp);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot_gen;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            for (int h = 0, g = 0; h < a.H && ok; ++h) {
                for (int j = 0; j < ns; ++j, ++g) {
                    const int sk = g % kNK, sv = g % kNV;
                    const uint32_t uk = static_cast<uint32_t>(g / kNK), uv = static_cast<uint32_t>(g / kNV);
                    const int key0 = j * kTcKeys;
                    const int C = a.H * kHd;
                    if (g >= kNK && !mbar_wait(k_empty(sk), (uk & 1u) ^ 1u, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kd = base + sk * kTcHalf;
                    mbar_arrive_expect_tx(k_full(sk), kTcHalf);
                    tma_load_2d(kd, &tk, h * kHd, krow0 + key0, k_full(sk));               // K_hi
                    tma_load_2d(kd + kT8, &tk, C + h * kHd, krow0 + key0, k_full(sk));     // K_lo
                    if (g >= kNV && !mbar_wait(v_empty(sv), (uv & 1u) ^ 1u, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vd = base + kTcOffV + sv * kTcHalf;
                    mbar_arrive_expect_tx(v_full(sv), kTcHalf);
                    tma_load_2d(vd, &tv, key0, (sq * a.H + h) * kHd, v_full(sv));           // Vt_hi
                    tma_load_2d(vd + kT8, &tv, a.L + key0, (sq * a.H + h) * kHd, v_full(sv));  // Vt_lo
                    // P of the slice: keys key0 .. + 31, then + 32 .. + 63, of the tile's queries
                    for (int half = 0; half < 2 && ok; ++half) {
                        const int gp = 2 * g + half, sp = gp % kNP;
                        const uint32_t up = static_cast<uint32_t>(gp / kNP);
                        if (gp >= kNP && !mbar_wait(p_empty(sp), (up & 1u) ^ 1u, a.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(p_full(sp), kT16);
                        tma_load_2d(base + kTcOffP + sp * kT16, &tp, key0 + 32 * half,
                                    (sq * a.H + h) * a.L + qb * kQKRows, p_full(sp));
                    }
                    if (!ok) break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kQKRows, kTcKeys, false, false);
            const uint32_t a_hi = base + kTcOffA, a_lo = a_hi + kT16;
            bool ok = true;
            // score product of slice g into ds buffer g & 1
            auto g1 = [&](int g) -> bool {
                const int st = g & 1, sk = g % kNK;
                if (!mbar_wait(k_full(sk), static_cast<uint32_t>(g / kNK) & 1u, a.status)) return false;
                if (g >= 2 && !mbar_wait(ds_empty(st), ((g >> 1) & 1) ^ 1u, a.status)) return false;
                tc_fence_after();
                const uint32_t kh = base + sk * kTcHalf, kl = kh + kT8;
                const uint32_t d = tmem + kTcKeys * st;
#pragma unroll
                for (int kk = 0; kk < kHd / 16; ++kk) {
                    const uint64_t ah = sdesc_sw128(a_hi + kk * 32u, 16u, 1024u);
                    const uint64_t al = sdesc_sw128(a_lo + kk * 32u, 16u, 1024u);
                    const uint64_t bh = sdesc_sw128(kh + kk * 32u, 16u, 1024u);
                    const uint64_t bl = sdesc_sw128(kl + kk * 32u, 16u, 1024u);
                    umma_bf16(d, ah, bh, idesc, kk != 0 ? 1u : 0u);
                    umma_bf16(d, ah, bl, idesc, 1u);
                    umma_bf16(d, al, bh, idesc, 1u);
                }
                umma_commit(ds_full(st));
                umma_commit(k_empty(sk));
                return true;
            };
            // value product of slice g (j-th of its head) into acc
            auto g2 = [&](int g, int j) -> bool {
                const int st = g & 1, sv = g % kNV;
                if (!mbar_wait(v_full(sv), static_cast<uint32_t>(g / kNV) & 1u, a.status)) return false;
                if (!mbar_wait(w_full(st), (g >> 1) & 1, a.status)) return false;
                tc_fence_after();
                const uint32_t wh = base + kTcOffW + st * 2u * kT16, wl = wh + kT16;
                const uint32_t vh = base + kTcOffV + sv * kTcHalf, vl = vh + kT8;
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    const uint64_t ah = sdesc_sw128(wh + kk * 32u, 16u, 1024u);
                    const uint64_t al = sdesc_sw128(wl + kk * 32u, 16u, 1024u);
                    const uint64_t bh = sdesc_sw128(vh + kk * 32u, 16u, 1024u);
                    const uint64_t bl = sdesc_sw128(vl + kk * 32u, 16u, 1024u);
                    umma_bf16(tmem + 128, ah, bh, idesc, (j | kk) != 0 ? 1u : 0u);
                    umma_bf16(tmem + 128, ah, bl, idesc, 1u);
                    umma_bf16(tmem + 128, al, bh, idesc, 1u);
                }
                umma_commit(w_empty(st));
                umma_commit(v_empty(sv));
                return true;
            };
            for (int h = 0, g0 = 0; h < a.H && ok; ++h, g0 += ns) {
                if (!mbar_wait(a_full, h & 1, a.status)) break;
                tc_fence_after();
                ok = g1(g0);
                for (int j = 0; j < ns && ok; ++j) {
                    if (j + 1 < ns) ok = g1(g0 + j + 1);
                    if (ok && j == 0 && h > 0) {
                        ok = mbar_wait(acc_empty, (h - 1) & 1, a.status);
                        tc_fence_after();
                    }
                    if (ok) ok = g2(g0 + j, j);
                }
                if (ok) umma_commit(acc_full);
            }
        }
    } else {
        const int e = threadIdx.x - 64;
        const int quarter = warp & 3;           // tensor-memory lane quarter
        const int grp = e >> 7;                 // keys (channels) kTcCols grp .. + kTcCols - 1
        const int row = quarter * 32 + lane;    // query row in the tile
        const int s = qb * kQKRows + row;       // its position in the sequence
        const int C = a.H * kHd;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t a_hi = base + kTcOffA, a_lo = a_hi + kT16;
        const DrawHalf dh = philox_draw_half(draw, a.token0 + static_cast<uint32_t>(tok0 + row), keys);
        bool ok = true;
        float dl = 0.f;
        for (int h = 0, g = 0; h < a.H; ++h) {
            // A for this head: the row's channels kTcCols grp .. + kTcCols - 1, scaled and split
            if (ok) {
#pragma unroll
                for (int m = 0; m < kTcCols / 8; ++m) {  // 16-byte chunk: 8 channels
                    const int c8 = (kTcCols / 8) * grp + m;
                    const int jb = h * (kHd / 4) + 2 * c8;
                    float4 n0, n1;
                    if (KEYS) {
                        const int64_t qe = static_cast<int64_t>(a.T) * C;
                        n0 = ld4(a.Q + DUST_IDX((tok0 + row) * C + 4 * jb, 4, qe));
                        n1 = ld4(a.Q + DUST_IDX((tok0 + row) * C + 4 * jb + 4, 4, qe));
                    } else {
                        n0 = words_to_normals_fast(philox_rest(
                            dh, philox_block_half(static_cast<uint32_t>(jb), a.layer, keys), keys));
                        n1 = words_to_normals_fast(philox_rest(
                            dh, philox_block_half(static_cast<uint32_t>(jb + 1), a.layer, keys), keys));
                    }
                    uint32_t hi[4], lo[4];
                    split_pair(a.scale * n0.x, a.scale * n0.y, hi[0], lo[0]);
                    split_pair(a.scale * n0.z, a.scale * n0.w, hi[1], lo[1]);
                    split_pair(a.scale * n1.x, a.scale * n1.y, hi[2], lo[2]);
                    split_pair(a.scale * n1.z, a.scale * n1.w, hi[3], lo[3]);
                    const uint32_t off = sw128(row, c8);
                    st_shared_v4(a_hi + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(a_lo + off, lo[0], lo[1], lo[2], lo[3]);
                }
                tc_fence_async_shared();
            }
            mbar_arrive(a_full);
            float2 wsum2 = make_float2(0.f, 0.f);
            for (int j = 0; j < ns; ++j, ++g) {
                const int st = g & 1;
                const int k0 = j * kTcKeys + kTcCols * grp;  // this thread's first key
                if (!ok) continue;
                // this thread's 16 keys of P: half grp / 2 of the slice, 16-byte
                // pieces 4 (grp % 2) .. + 3 of its row, swizzled
                float4 pv[kTcCols / 4];
                {
                    const int gp = 2 * g + (grp >> 1), sp = gp % kNP;
                    ok = mbar_wait(p_full(sp), static_cast<uint32_t>(gp / kNP) & 1u, a.status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) continue;
                    const uint32_t prow = base + kTcOffP + sp * kT16 + static_cast<uint32_t>(row) * 128u;
#pragma unroll
                    for (int q = 0; q < kTcCols / 4; ++q) {
                        const uint32_t c = static_cast<uint32_t>(((grp & 1) * 4 + q) ^ (row & 7));
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(pv[q].x), "=f"(pv[q].y), "=f"(pv[q].z), "=f"(pv[q].w)
                                     : "r"(prow + (c << 4))
                                     : "memory");
                    }
                    // the reads above before the TMA's next write to the stage (a
                    // generic-proxy read, then an async-proxy write)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive(p_empty(sp));
                }
                ok = mbar_wait(ds_full(st), (g >> 1) & 1, a.status);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) continue;
                tc_fence_after();
                uint32_t r[kTcCols];
                tmem_ld_32x32b_x16(tmem + lane_off + kTcKeys * st + kTcCols * grp, r);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(ds_empty(st));
                // e^x - 1 on channel pairs: x (1 + x/2 + x^2/6 + x^3/24) for |x| < 1/8;
                // a warp with any larger x redoes those with expm1f.
                float2 ex[kTcCols / 2];
                bool big = false;
#pragma unroll
                for (int m = 0; m < kTcCols / 2; ++m) {
                    const float2 x = make_float2(__uint_as_float(r[2 * m]), __uint_as_float(r[2 * m + 1]));
                    big |= fabsf(x.x) >= 0.125f || fabsf(x.y) >= 0.125f;
                    float2 q = fma2(x, make_float2(1.0f / 24.0f, 1.0f / 24.0f),
                                    make_float2(1.0f / 6.0f, 1.0f / 6.0f));
                    q = fma2(x, q, make_float2(0.5f, 0.5f));
                    q = fma2(x, q, make_float2(1.0f, 1.0f));
                    ex[m] = mul2(x, q);
                }
                if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                    for (int m = 0; m < kTcCols / 2; ++m) {
                        const float x0 = __uint_as_float(r[2 * m]), x1 = __uint_as_float(r[2 * m + 1]);
                        if (fabsf(x0) >= 0.125f) ex[m].x = expm1f(x0);
                        if (fabsf(x1) >= 0.125f) ex[m].y = expm1f(x1);
                    }
                }
                // w = P (e^ds - 1), zero after the query (only the tile's diagonal slices)
                float2 w[kTcCols / 2];
#pragma unroll
                for (int q = 0; q < kTcCols / 4; ++q) {
                    w[2 * q] = mul2(make_float2(pv[q].x, pv[q].y), ex[2 * q]);
                    w[2 * q + 1] = mul2(make_float2(pv[q].z, pv[q].w), ex[2 * q + 1]);
                }
                if ((j + 1) * kTcKeys > qb * kQKRows) {
#pragma unroll
                    for (int m = 0; m < kTcCols / 2; ++m) {
                        if (k0 + 2 * m > s) w[m].x = 0.f;
                        if (k0 + 2 * m + 1 > s) w[m].y = 0.f;
                    }
                }
#pragma unroll
                for (int m = 0; m < kTcCols / 2; ++m) wsum2 = add2(wsum2, w[m]);
                if (g >= 2) {
                    ok = mbar_wait(w_empty(st), ((g >> 1) & 1) ^ 1u, a.status);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) continue;
                }
                const uint32_t wh = base + kTcOffW + st * 2u * kT16, wl = wh + kT16;
#pragma unroll
                for (int m = 0; m < kTcCols / 8; ++m) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) split_pair2(w[4 * m + u], hi[u], lo[u]);
                    const uint32_t off = sw128(row, (kTcCols / 8) * grp + m);
                    st_shared_v4(wh + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(wl + off, lo[0], lo[1], lo[2], lo[3]);
                }
                tc_fence_async_shared();
                mbar_arrive(w_full(st));
            }
            const float wsum = wsum2.x + wsum2.y;
            // end of the head: W_s, then <E, dO> over this thread's channels
            s_w[h & 1][grp][row] = wsum;
            ok = epi_all(ok);
            if (ok) {
                ok = mbar_wait(acc_full, h & 1, a.status);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok) {
                tc_fence_after();
                uint32_t r[kTcCols];
                tmem_ld_32x32b_x16(tmem + lane_off + 128 + kTcCols * grp, r);
                tmem_wait_ld();
                tc_fence_before();
                float W = 0.f;
#pragma unroll
                for (int q = 0; q < kTcGroups; ++q) W += s_w[h & 1][q][row];
                const int64_t off = (tok0 + row) * C + h * kHd + kTcCols * grp;
                float eo = 0.f;
#pragma unroll
                for (int q = 0; q < kTcCols / 4; ++q) {
                    const int64_t oi = DUST_IDX(off + 4 * q, 4, static_cast<int64_t>(a.T) * C);
                    const float4 o4 = ld4(a.O + oi), e4 = ld4(a.E + oi);
                    eo = fmaf(e4.x, fmaf(-W, o4.x, __uint_as_float(r[4 * q])), eo);
                    eo = fmaf(e4.y, fmaf(-W, o4.y, __uint_as_float(r[4 * q + 1])), eo);
                    eo = fmaf(e4.z, fmaf(-W, o4.z, __uint_as_float(r[4 * q + 2])), eo);
                    eo = fmaf(e4.w, fmaf(-W, o4.w, __uint_as_float(r[4 * q + 3])), eo);
                }
                dl += eo / (1.0f + W);
            }
            mbar_arrive(acc_empty);
        }
        s_dl[grp][row] = dl;
        epi_sync();
        if (ok && grp == 0 && DUST_IB(tok0 + row, a.T)) {
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < kTcGroups; ++q) sum += s_dl[q][row];
            a.dl[static_cast<int64_t>(i) * a.T + tok0 + row] = sum;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 256);
}

// The keys' noise of draws draw_first .. + nd - 1 as bf16 [hi | lo] rows of
// 2C, draw d at rows d T .. d T + T - 1 (the counter scheme of every layer).
__global__ void qk_key_noise_kernel(int nd, int64_t T, int C, uint32_t draw_first, uint32_t token0,
                                    uint32_t layer, PhiloxKeys keys, __nv_bfloat16* __restrict__ N2) {
    const int nb = C / 4;
    const int64_t n = static_cast<int64_t>(nd) * T * nb;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int jb = static_cast<int>(idx % nb);
        const int64_t dt = idx / nb;  // d T + t
        const int d = static_cast<int>(dt / T);
        const int64_t t = dt - static_cast<int64_t>(d) * T;
        const float4 v = words_to_normals_fast(philox4x32_10(static_cast<uint32_t>(jb),
                                                        token0 + static_cast<uint32_t>(t),
                                                        draw_first + static_cast<uint32_t>(d), layer,
                                                        keys));
        uint32_t hi0, lo0, hi1, lo1;
        split_pair(v.x, v.y, hi0, lo0);
        split_pair(v.z, v.w, hi1, lo1);
        __nv_bfloat16* row = N2 + dt * 2 * C;
        if (!DUST_IB(dt * 2 * C + C + 4 * jb + 3, n / nb * 2 * C)) continue;
        *reinterpret_cast<uint2*>(row + 4 * jb) = make_uint2(hi0, hi1);
        *reinterpret_cast<uint2*>(row + C + 4 * jb) = make_uint2(lo0, lo1);
    }
}

// K (T x C fp32) -> [K_hi | K_lo] rows of 2C bf16.
__global__ void qk_split_rows_kernel(const float* __restrict__ X, int64_t T, int C,
                                     __nv_bfloat16* __restrict__ X2) {
    const int64_t n2 = T * (C / 2);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n2;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / (C / 2);
        const int c = static_cast<int>(i - t * (C / 2)) * 2;
        if (!DUST_IB(t * C + c + 1, T * C)) continue;
        const float2 v = *reinterpret_cast<const float2*>(X + t * C + c);
        uint32_t hi, lo;
        split_pair(v.x, v.y, hi, lo);
        *reinterpret_cast<uint32_t*>(X2 + t * 2 * C + c) = hi;
        *reinterpret_cast<uint32_t*>(X2 + t * 2 * C + C + c) = lo;
    }
}

// V (T x C fp32) -> V^T per (sequence, head): row (sq H + h) 64 + c, columns
// [hi of keys 0 .. L-1 | lo of keys 0 .. L-1].  One 64-key x 64-channel tile
// per block through shared memory.
__global__ void __launch_bounds__(256) qk_split_vt_kernel(const float* __restrict__ V, int L, int H,
                                                          __nv_bfloat16* __restrict__ Vt2) {
    __shared__ float tile[64][65];
    const int kt = blockIdx.x;            // key tile
    const int sh = blockIdx.y;            // sq H + h
    const int h = sh % H, sq = sh / H;
    const int C = H * kHd;
    for (int e = threadIdx.x; e < 64 * 64; e += 256) {
        const int t = e / 64, c = e % 64;
        tile[t][c] = V[(static_cast<int64_t>(sq) * L + kt * 64 + t) * C + h * kHd + c];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 64 * 32; e += 256) {
        const int c = e / 32, t = 2 * (e % 32);
        uint32_t hi, lo;
        split_pair(tile[t][c], tile[t + 1][c], hi, lo);
        __nv_bfloat16* row = Vt2 + (static_cast<int64_t>(sh) * kHd + c) * (2 * static_cast<int64_t>(L));
        *reinterpret_cast<uint32_t*>(row + kt * 64 + t) = hi;
        *reinterpret_cast<uint32_t*>(row + L + kt * 64 + t) = lo;
    }
}

std::atomic<uint64_t> qk_tc_smem_set[2];
constexpr int kKeyGroup = 16;  // draws whose key noise is held at once (keys mode)

struct QKPlan {
    int64_t ldx;
    size_t off_dl, off_m, off_r, off_gbf, off_xbf, off_k2, off_v2, off_n2, bytes;
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
    P.off_k2 = w.take(static_cast<size_t>(T * C) * 4);  // [K_hi | K_lo] bf16
    P.off_v2 = w.take(static_cast<size_t>(T * C) * 4);  // V^T [hi | lo] bf16
    P.off_n2 = w.take(static_cast<size_t>(T * C) * 4 *  // keys' noise of a draw group
                      static_cast<size_t>(K < static_cast<uint32_t>(kKeyGroup) ? K : kKeyGroup));
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

dust_status dust::attn_qk_check(int which, const float* Q, const float* Kk, const float* V,
                                const float* O, const float* P, const float* E, const void* x,
                                dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t H,
                                int64_t dv, int64_t d_in, const dust_noise& nz,
                                const float* g_hat, const float* G_W, const void* ws,
                                size_t ws_bytes) {
    if (which != 0 && which != 1) return DUST_ERR_INVALID_ARG;
    if (!Q || !Kk || !V || !O || !P || !E || !x || !G_W) return DUST_ERR_INVALID_ARG;
    if (T < 1 || seq_len < 1 || T % seq_len != 0 || H < 1 || d_in < 1) return DUST_ERR_INVALID_ARG;
    if (x_dtype != DUST_F32 && x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
    if (nz.num_draws < 2 || !(nz.sigma > 0.0f) || !(nz.sigma < INFINITY)) return DUST_ERR_INVALID_ARG;
    if (!(nz.gamma >= 0.0f && nz.gamma <= 1.0f)) return DUST_ERR_INVALID_ARG;
    if (dv != kHd || seq_len % kQKRows != 0 || seq_len > 8192 || H > 64 || T / kQKRows > 65535 ||
        T / seq_len * H > 65535 || nz.num_draws > 65535 || d_in > (1LL << 20))
        return DUST_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(nz.token0) + static_cast<uint64_t>(T) > (1ULL << 32) ||
        static_cast<uint64_t>(nz.draw0) + nz.num_draws > (1ULL << 32))
        return DUST_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(Kk, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(P, 16) || !aligned(E, 16) || (g_hat && !aligned(g_hat, 16)))
        return DUST_ERR_INVALID_ARG;
    const QKPlan Pl = qk_plan(T, H, d_in, nz.num_draws);
    if (!ws || ws_bytes < Pl.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    return DUST_OK;
}

extern "C" dust_status dust_attn_qk_estimate(int which, const float* Q, const float* Kk,
                                             const float* V, const float* O, const float* P,
                                             const float* E, const void* x, dust_dtype x_dtype,
                                             int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                                             int64_t d_in, dust_noise nz, float* g_hat,
                                             float* G_W, void* ws, size_t ws_bytes, void* stream) {
    const dust_status chk = attn_qk_check(which, Q, Kk, V, O, P, E, x, x_dtype, T, seq_len, H, dv,
                                          d_in, nz, g_hat, G_W, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const QKPlan Pl = qk_plan(T, H, d_in, nz.num_draws);
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

    dust_status st = DUST_OK;
    {
        // K (queries) and V^T split once; the keys' noise per group of draws
        __nv_bfloat16* K2 = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_k2);
        __nv_bfloat16* V2 = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_v2);
        __nv_bfloat16* N2 = reinterpret_cast<__nv_bfloat16*>(w + Pl.off_n2);
        if (which == 0) {
            qk_split_rows_kernel<<<static_cast<unsigned>(std::min<int64_t>(ceil_div(T * C / 2, 256), 148 * 16)),
                                   256, 0, s>>>(Kk, T, static_cast<int>(C), K2);
            if ((st = launch_status()) != DUST_OK) return st;
        }
        qk_split_vt_kernel<<<dim3(static_cast<unsigned>(seq_len / 64),
                                  static_cast<unsigned>(T / seq_len * H)),
                             256, 0, s>>>(V, static_cast<int>(seq_len), static_cast<int>(H), V2);
        if ((st = launch_status()) != DUST_OK) return st;
        const int group = which == 0 ? static_cast<int>(nz.num_draws)
                                     : std::min(static_cast<int>(nz.num_draws), kKeyGroup);
        CUtensorMap tk, tv, tp;
        if (!encode_bf16_2d(&tk, which == 0 ? K2 : N2, 2 * C, which == 0 ? T : group * T, 2 * C,
                            kTcKeys, kTcKeys) ||
            !encode_bf16_2d(&tv, V2, 2 * seq_len, T / seq_len * H * kHd, 2 * seq_len, kTcKeys,
                            kHd) ||
            !encode_f32_2d(&tp, P, seq_len, T * H, seq_len, 32, kQKRows))
            return DUST_ERR_CUDA;
        if (which == 0)
            DUST_CUDA_TRY(set_smem_once(attn_qk_tc_kernel<false>, static_cast<int>(kTcSmem), qk_tc_smem_set[0]));
        else
            DUST_CUDA_TRY(set_smem_once(attn_qk_tc_kernel<true>, static_cast<int>(kTcSmem), qk_tc_smem_set[1]));
        for (int i0 = 0; i0 < static_cast<int>(nz.num_draws); i0 += group) {
            const int nd = std::min(group, static_cast<int>(nz.num_draws) - i0);
            if (which == 1) {
                const int64_t n = static_cast<int64_t>(nd) * T * (C / 4);
                qk_key_noise_kernel<<<static_cast<unsigned>(std::min<int64_t>(ceil_div(n, 256), 148 * 16)),
                                      256, 0, s>>>(nd, T, static_cast<int>(C),
                                                   nz.draw0 + static_cast<uint32_t>(i0), nz.token0,
                                                   nz.layer, keys, N2);
                if ((st = launch_status()) != DUST_OK) return st;
            }
            const QKTcArgs ta{Q, P, O, E, dl, static_cast<int>(T), static_cast<int>(seq_len),
                              static_cast<int>(H), i0, nz.draw0, nz.token0, nz.layer,
                              nz.sigma * 0.125f, status};
            const dim3 grid(static_cast<unsigned>(nd), static_cast<unsigned>(T / kQKRows));
            timer_begin(s);
            if (which == 0)
                attn_qk_tc_kernel<false><<<grid, kTcThreads, kTcSmem, s>>>(tk, tv, tp, ta, keys);
            else
                attn_qk_tc_kernel<true><<<grid, kTcThreads, kTcSmem, s>>>(tk, tv, tp, ta, keys);
            timer_end(s);
            if ((st = launch_status()) != DUST_OK) return st;
        }
    }
    if ((st = launch_status()) != DUST_OK) return st;
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
DUST_DEBUG_READER(7)
}  // namespace dust
