// gemm.cu -- bf16 x bf16 -> fp32 contractions on the tcgen05 tensor cores.
//
// Two users:
//   * the outer product G_W = sum_t g_t x_t^T (Dust translation,
//     hn.213312.xyz, §2.2 信用分配: the weight gradient has backprop's
//     outer-product form, only the error source differs), with a plain fp32
//     store epilogue;
//   * the interior layer's re-forward of the part after the perturbed layer
//     (laoyaoba.com article, section 机制拆解; Dust translation §2.3), whose
//     last contraction (the head) ends in a cross-entropy epilogue so that
//     the perturbed logits never reach memory.
//
// One CTA owns a 128-row tile of the output and walks n_per_cta column tiles
// of 256.  Warp 0's elected thread streams 64-deep K slices of both operands
// into a four-stage shared-memory ring with TMA (128-byte swizzle); warp 1's
// elected thread issues tcgen05.mma (M = 128, N = 256, K = 16) into one of two
// 256-column tensor-memory accumulators and releases each stage with
// tcgen05.commit; warps 2-5 read the finished accumulator with tcgen05.ld (one
// TMEM lane = one output row per thread) while the MMAs of the next column
// tile run into the other accumulator.
//
// Operands are K-major (rows of K elements) or MN-major (K rows of M or N
// elements).  b_kmod > 0 makes B's K coordinate wrap modulo b_kmod: the
// split-bf16 form A = [hi | lo] against B = W reads W twice without a copy.
#include <cudaTypedefs.h>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {

bool encode_bf16_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                    int64_t stride_elems, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr uint32_t kBBytes = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
// The cross-entropy epilogue also stages the softmax rows it needs: two
// 128 x 32 fp32 tiles (128-byte swizzle), filled by TMA from a seventh warp.
constexpr uint32_t kPTile = kBM * 32 * 4;
template <int EPI>
constexpr uint32_t smem_bytes() {
    return kStages * kStageBytes + (EPI == 1 ? 2 * kPTile : 0) + 1024 + 256;
}
template <int EPI>
constexpr int threads_of() {
    return EPI == 1 ? 224 : 192;
}

enum { EPI_STORE = 0, EPI_CE = 1 };

struct GemmShape {
    int M, N, K;
    int n_per_cta;
    int b_kmod;
    int n_fastest;  // grid.x walks N tiles (CTAs sharing an A tile run together)
};

struct EpiStore {
    float* D;
    int64_t ldd;
};

// Cross-entropy epilogue of the interior re-forward.  Rows are ordered
// (token block of 128, draw, token in block): row tile m covers draw
// i0 + m % ndraw and tokens (m / ndraw) * 128 .. + 127.  Per row it forms
// S = sum_v p_{t,v} (exp(dz_v) - 1) and dz_{y_t}, and writes
// dl[(i0 + i) * T + t] = log(1 + S) - dz_y, which equals
// CE(z + dz) - CE(z) because sum_v p_{t,v} = 1.  Summing the small terms
// e^dz - 1 keeps the fp32 rounding of the sum far below the loss change.
struct EpiCE {
    const float* p;  // T x V softmax of the clean logits (staged by TMA)
    const int32_t* targets;
    float* dl;       // K x T
    int T, V, ndraw, i0;
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// e^x - 1 without the cancellation of computing e^x first: the Taylor series
// to x^6 (truncation below 5e-8 relative for |x| < 1/4), else e^x - 1.
__device__ __forceinline__ float expm1_small(float x) {
    if (fabsf(x) < 0.25f) {
        float q = fmaf(x, 1.0f / 720.0f, 1.0f / 120.0f);
        q = fmaf(x, q, 1.0f / 24.0f);
        q = fmaf(x, q, 1.0f / 6.0f);
        q = fmaf(x, q, 0.5f);
        q = fmaf(x, q, 1.0f);
        return x * q;
    }
    return ex2_approx(x * 1.4426950408889634f) - 1.0f;
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(threads_of<EPI>(), 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                     const __grid_constant__ CUtensorMap tp, const GemmShape sh,
                     const EpiStore es, const EpiCE ec, uint32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_gen = smem_raw + (base - raw);
    const uint32_t pbuf = base + kStages * kStageBytes;  // CE epilogue only
    const uint32_t bars = pbuf + (EPI == EPI_CE ? 2 * kPTile : 0);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * kStages + 2 + b); };
    auto pfull_bar = [&](int b) { return bars + 8u * (2 * kStages + 4 + b); };
    auto pempty_bar = [&](int b) { return bars + 8u * (2 * kStages + 6 + b); };
    const uint32_t tmem_slot = bars + 8u * (2 * kStages + 8);
    volatile uint32_t* tmem_slot_gen =
        reinterpret_cast<volatile uint32_t*>(base_gen + (tmem_slot - base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mtile = sh.n_fastest ? blockIdx.y : blockIdx.x;
    const int m0 = mtile * kBM;
    const int ntiles = (sh.N + kBN - 1) / kBN;
    const int nt0 = (sh.n_fastest ? blockIdx.x : blockIdx.y) * sh.n_per_cta;
    const int nt_count = min(sh.n_per_cta, ntiles - nt0);
    const int nk = (sh.K + kBK - 1) / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);
            mbar_init(pfull_bar(b), 1);
            mbar_init(pempty_bar(b), 4);
        }
        mbar_fence_init();
        tma_prefetch_desc(&ta);
        tma_prefetch_desc(&tb);
        if (EPI == EPI_CE) tma_prefetch_desc(&tp);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot_gen;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int j = 0; j < nt_count && ok; ++j) {
                const int n0 = (nt0 + j) * kBN;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (it >= kStages && !mbar_wait(empty_bar(s), ph ^ 1u, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                    const uint32_t a_dst = base + s * kStageBytes;
                    const uint32_t b_dst = a_dst + kABytes;
                    const int k0 = kb * kBK;
                    const int kB = sh.b_kmod > 0 ? k0 % sh.b_kmod : k0;
                    if (A_MN) {
                        tma_load_2d(a_dst, &ta, m0, k0, full_bar(s));
                        tma_load_2d(a_dst + kABytes / 2, &ta, m0 + 64, k0, full_bar(s));
                    } else {
                        tma_load_2d(a_dst, &ta, k0, m0, full_bar(s));
                    }
                    if (B_MN) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tma_load_2d(b_dst + q * (kBBytes / 4), &tb, n0 + 64 * q, kB, full_bar(s));
                    } else {
                        tma_load_2d(b_dst, &tb, kB, n0, full_bar(s));
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, A_MN, B_MN);
            int it = 0;
            bool ok = true;
            for (int j = 0; j < nt_count; ++j) {
                const int buf = j & 1;
                if (ok && j >= 2 && !mbar_wait(acce_bar(buf), ((j >> 1) & 1u) ^ 1u, status)) ok = false;
                tc_fence_after();
                const uint32_t d = tmem + buf * kBN;
                for (int kb = 0; kb < nk && ok; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1u;
                    if (!mbar_wait(full_bar(s), ph, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = base + s * kStageBytes;
                    const uint32_t b = a + kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // MN-major: 16 K rows of 128 bytes per step, 64-element MN
                        // chunks one box apart.  K-major: 32 bytes along the
                        // swizzled row per step, 8-row groups 1 KB apart.
                        const uint64_t ad = A_MN ? sdesc_sw128(a + kk * 2048u, kABytes / 2, 1024u)
                                                 : sdesc_sw128(a + kk * 32u, 16u, 1024u);
                        const uint64_t bd = B_MN ? sdesc_sw128(b + kk * 2048u, kBBytes / 4, 1024u)
                                                 : sdesc_sw128(b + kk * 32u, 16u, 1024u);
                        umma_bf16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty_bar(s));
                }
                umma_commit(accf_bar(buf));  // also on failure, so nobody waits forever
            }
        }
    } else if (warp == 6) {
        // CE epilogue only: the softmax tile of every 32-column chunk, two
        // chunks ahead, rows = the tile's 128 tokens.
        if (EPI == EPI_CE && lane == 0) {
            const int tok0 = (blockIdx.x / ec.ndraw) * kBM;
            const int nq = nt_count * (kBN / 32);
            for (int q = 0; q < nq; ++q) {
                const int b = q & 1;
                if (q >= 2 && !mbar_wait(pempty_bar(b), ((q >> 1) - 1) & 1u, status)) break;
                mbar_arrive_expect_tx(pfull_bar(b), kPTile);
                const int col = (nt0 + q / (kBN / 32)) * kBN + (q % (kBN / 32)) * 32;
                tma_load_2d(pbuf + b * kPTile, &tp, col, tok0, pfull_bar(b));
            }
        }
    } else {
        // Epilogue warps 2..5; warp w may read TMEM lanes 32 (w % 4) .. + 31.
        const int quarter = warp & 3;
        const int rit = quarter * 32 + lane;  // row in tile
        const int row = m0 + rit;
        float ce_sum = 0.f, ce_zy = 0.f;
        int ce_t = 0, ce_i = 0, ce_y = -1;
        bool ce_valid = false;
        if (EPI == EPI_CE) {
            const int mt = blockIdx.x;
            ce_i = mt % ec.ndraw;
            ce_t = (mt / ec.ndraw) * kBM + rit;
            ce_valid = ce_t < ec.T;
            if (ce_valid) {
                ce_y = __ldg(ec.targets + ce_t);
                if (ce_y < 0 || ce_y >= ec.V) {
                    record_status(status, DUST_ERR_DEVICE_RANGE);
                    ce_y = -1;
                }
            }
        }
        bool ok = true;
        for (int j = 0; j < nt_count; ++j) {
            const int buf = j & 1;
            bool got = ok && mbar_wait(accf_bar(buf), (j >> 1) & 1u, status);
            got = __all_sync(0xFFFFFFFFu, got);
            if (!got) ok = false;
            tc_fence_after();
            const int n0 = (nt0 + j) * kBN;
            if (ok) {
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                           buf * kBN + c * 32,
                                       r);
                    tmem_wait_ld();
                    const int col0 = n0 + c * 32;
                    if (EPI == EPI_STORE) {
                        if (row < sh.M) {
                            float* drow = es.D + static_cast<int64_t>(row) * es.ldd;
                            const int64_t dext = static_cast<int64_t>(sh.M) * es.ldd;
                            if (((es.ldd & 3) == 0) && col0 + 32 <= sh.N &&
                                ((reinterpret_cast<uintptr_t>(es.D) & 15) == 0) &&
                                DUST_IB(static_cast<int64_t>(row) * es.ldd + col0 + 31, dext)) {
#pragma unroll
                                for (int q = 0; q < 32; q += 4)
                                    *reinterpret_cast<float4*>(drow + col0 + q) = make_float4(
                                        __uint_as_float(r[q]), __uint_as_float(r[q + 1]),
                                        __uint_as_float(r[q + 2]), __uint_as_float(r[q + 3]));
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; ++q)
                                    if (col0 + q < sh.N &&
                                        DUST_IB(static_cast<int64_t>(row) * es.ldd + col0 + q, dext))
                                        drow[col0 + q] = __uint_as_float(r[q]);
                            }
                        }
                    } else {
                        // chunk q = j * 8 + c uses p buffer q & 1
                        const int q = j * (kBN / 32) + c;
                        const int pb = q & 1;
                        bool pg = mbar_wait(pfull_bar(pb), (q >> 1) & 1u, status);
                        pg = __all_sync(0xFFFFFFFFu, pg);
                        if (pg && ce_valid) {
                            const uint32_t prow = pbuf + pb * kPTile + rit * 128u;
#pragma unroll
                            for (int g4 = 0; g4 < 8; ++g4) {
                                float4 p4;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(p4.x), "=f"(p4.y), "=f"(p4.z), "=f"(p4.w)
                                             : "r"(prow + (((g4 ^ (rit & 7)) & 7u) << 4))
                                             : "memory");
                                const int qq = 4 * g4;
                                ce_sum = fmaf(p4.x, expm1_small(__uint_as_float(r[qq])), ce_sum);
                                ce_sum = fmaf(p4.y, expm1_small(__uint_as_float(r[qq + 1])), ce_sum);
                                ce_sum = fmaf(p4.z, expm1_small(__uint_as_float(r[qq + 2])), ce_sum);
                                ce_sum = fmaf(p4.w, expm1_small(__uint_as_float(r[qq + 3])), ce_sum);
                            }
                        }
                        // the reads above before the TMA's next write to the buffer (a
                        // generic-proxy read, then an async-proxy write)
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(pempty_bar(pb));
                        if (!ce_valid) continue;
                        const int yo = ce_y - col0;
                        if (yo >= 0 && yo < 32) {
#pragma unroll
                            for (int qq = 0; qq < 32; ++qq)
                                if (qq == yo) ce_zy = __uint_as_float(r[qq]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(buf));
        }
        // (the launch writes rows i0 .. i0 + ndraw - 1 of dl)
        if (EPI == EPI_CE && ok && ce_valid &&
            DUST_IB(static_cast<int64_t>(ec.i0 + ce_i) * ec.T + ce_t,
                    static_cast<int64_t>(ec.i0 + ec.ndraw) * ec.T))
            ec.dl[static_cast<int64_t>(ec.i0 + ce_i) * ec.T + ce_t] = log1pf(ce_sum) - ce_zy;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

bool encode_operands(CUtensorMap* ta, CUtensorMap* tb, const void* A, bool a_mn, int64_t lda,
                     const void* B, bool b_mn, int64_t ldb, int64_t M, int64_t N, int64_t K,
                     int64_t b_kmod) {
    const int64_t KB = b_kmod > 0 ? b_kmod : K;
    bool ok = a_mn ? encode_bf16_2d(ta, A, M, K, lda, 64, kBK)
                   : encode_bf16_2d(ta, A, K, M, lda, kBK, kBM);
    ok = ok && (b_mn ? encode_bf16_2d(tb, B, N, KB, ldb, 64, kBK)
                     : encode_bf16_2d(tb, B, KB, N, ldb, kBK, kBN));
    return ok;
}

template <bool A_MN, bool B_MN, int EPI>
dust_status launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tp,
                     const GemmShape& sh, const EpiStore& es, const EpiCE& ec, uint32_t* status,
                     cudaStream_t s) {
    auto kern = gemm_bf16_kernel<A_MN, B_MN, EPI>;
    constexpr uint32_t smem = smem_bytes<EPI>();
    static std::atomic<uint64_t> smem_set{0};  // one per template instance
    DUST_CUDA_TRY(set_smem_once(kern, static_cast<int>(smem), smem_set));
    const int ntiles = (sh.N + kBN - 1) / kBN;
    const unsigned gm = static_cast<unsigned>(ceil_div(sh.M, kBM));
    const unsigned gn = static_cast<unsigned>(ceil_div(ntiles, sh.n_per_cta));
    const dim3 grid = sh.n_fastest ? dim3(gn, gm) : dim3(gm, gn);
    kern<<<grid, threads_of<EPI>(), smem, s>>>(ta, tb, tp, sh, es, ec, status);
    return launch_status();
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D bf16 tensor (inner x outer elements, row stride in elements) with a
// 128-byte-swizzled box of box_inner x box_outer; out-of-range reads are 0.
bool encode_bf16_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                    int64_t stride_elems, uint32_t box_inner, uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_elems) * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D fp32 tensor (inner x outer elements, row stride in elements) with a
// 128-byte-swizzled box of box_inner (32) x box_outer; out-of-range reads are 0.
bool encode_f32_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                   int64_t stride_elems, uint32_t box_inner, uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_elems) * 4};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ in, int64_t rows, int64_t cols,
                                   int64_t ld_in, __nv_bfloat16* __restrict__ out,
                                   int64_t ld_out) {
    const int64_t n = rows * ld_out;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / ld_out, c = i - r * ld_out;
        const bool in_b = c < cols && DUST_IB(r * ld_in + c, (rows - 1) * ld_in + cols);
        out[i] = __float2bfloat16_rn(in_b ? in[r * ld_in + c] : 0.0f);
    }
}

__global__ void bf16_pad_kernel(const __nv_bfloat16* __restrict__ in, int64_t rows, int64_t cols,
                                int64_t ld_in, __nv_bfloat16* __restrict__ out, int64_t ld_out) {
    const int64_t n = rows * ld_out;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / ld_out, c = i - r * ld_out;
        const bool in_b = c < cols && DUST_IB(r * ld_in + c, (rows - 1) * ld_in + cols);
        out[i] = in_b ? in[r * ld_in + c] : __float2bfloat16_rn(0.0f);
    }
}

static unsigned grid_for(int64_t n) {
    int64_t b = ceil_div(n, 256);
    if (b > 148 * 32) b = 148 * 32;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

dust_status f32_to_bf16_launch(const float* in, int64_t rows, int64_t cols, int64_t ld_in,
                               void* out, int64_t ld_out, cudaStream_t s) {
    if (rows * ld_out == 0) return DUST_OK;
    f32_to_bf16_kernel<<<grid_for(rows * ld_out), 256, 0, s>>>(
        in, rows, cols, ld_in, static_cast<__nv_bfloat16*>(out), ld_out);
    return launch_status();
}

dust_status bf16_pad_launch(const void* in, int64_t rows, int64_t cols, int64_t ld_in, void* out,
                            int64_t ld_out, cudaStream_t s) {
    if (rows * ld_out == 0) return DUST_OK;
    bf16_pad_kernel<<<grid_for(rows * ld_out), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(in), rows, cols, ld_in,
        static_cast<__nv_bfloat16*>(out), ld_out);
    return launch_status();
}

dust_status gemm_bf16_launch(const void* A, bool a_mn, int64_t lda, const void* B, bool b_mn,
                             int64_t ldb, int64_t M, int64_t N, int64_t K, int64_t b_kmod,
                             int n_per_cta, float* G, int64_t ldg, uint32_t* status,
                             cudaStream_t s) {
    CUtensorMap ta, tb;
    if (!encode_operands(&ta, &tb, A, a_mn, lda, B, b_mn, ldb, M, N, K, b_kmod))
        return DUST_ERR_CUDA;
    // One N tile per CTA, N tiles of the same A tile launched together, when
    // the caller asks for a single tile per CTA: the A tile is then read from
    // HBM once and served from L2 to its neighbours.
    GemmShape sh{static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), n_per_cta,
                 static_cast<int>(b_kmod), n_per_cta == 1 ? 1 : 0};
    EpiStore es{G, ldg};
    EpiCE ec{};
    if (a_mn && b_mn) return launch_t<true, true, EPI_STORE>(ta, tb, ta, sh, es, ec, status, s);
    if (a_mn) return launch_t<true, false, EPI_STORE>(ta, tb, ta, sh, es, ec, status, s);
    if (b_mn) return launch_t<false, true, EPI_STORE>(ta, tb, ta, sh, es, ec, status, s);
    return launch_t<false, false, EPI_STORE>(ta, tb, ta, sh, es, ec, status, s);
}

dust_status gemm_ce_launch(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M,
                           int64_t V, int64_t K, int64_t b_kmod, const float* p, int64_t ldp,
                           const int32_t* targets, int64_t T, int ndraw, int i0, float* dl,
                           uint32_t* status, cudaStream_t s) {
    CUtensorMap ta, tb;
    if (!encode_operands(&ta, &tb, A, false, lda, B, false, ldb, M, V, K, b_kmod))
        return DUST_ERR_CUDA;
    const int ntiles = static_cast<int>(ceil_div(V, kBN));
    GemmShape sh{static_cast<int>(M), static_cast<int>(V), static_cast<int>(K), ntiles,
                 static_cast<int>(b_kmod), 0};
    EpiStore es{};
    EpiCE ec{p, targets, dl, static_cast<int>(T), static_cast<int>(V), ndraw, i0};
    // softmax rows: T x V fp32, row stride ldp (a multiple of 4), 128 x 32 boxes
    CUtensorMap tp;
    {
        auto enc = tensor_map_encoder();
        if (enc == nullptr) return DUST_ERR_CUDA;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(T)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldp) * 4};
        cuuint32_t box[2] = {32, kBM};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&tp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DUST_ERR_CUDA;
    }
    timer_begin(s);
    const dust_status st = launch_t<false, false, EPI_CE>(ta, tb, tp, sh, es, ec, status, s);
    timer_end(s);
    return st;
}

}  // namespace dust

extern "C" dust_status dust_gemm_bf16(const void* A, int a_mn, int64_t lda, const void* B,
                                      int b_mn, int64_t ldb, int64_t M, int64_t N, int64_t K,
                                      float* G, int64_t ldg, void* ws, size_t ws_bytes,
                                      void* stream) {
    using namespace dust;
    if (!A || !B || !G || M < 1 || N < 1 || K < 1) return DUST_ERR_INVALID_ARG;
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return DUST_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < kCtlBytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    const int64_t a_inner = a_mn ? M : K, b_inner = b_mn ? N : K;
    if (lda < a_inner || ldb < b_inner || ldg < N) return DUST_ERR_INVALID_ARG;
    if ((lda % 8) || (ldb % 8) || !aligned(A, 16) || !aligned(B, 16)) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    return gemm_bf16_launch(A, a_mn != 0, lda, B, b_mn != 0, ldb, M, N, K, 0, 1, G, ldg,
                            static_cast<uint32_t*>(ws), s);
}

namespace dust {
DUST_DEBUG_READER(4)
}  // namespace dust
