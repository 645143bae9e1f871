// internal.h -- host-side pieces shared by the entry points: workspace
// carving, CUDA error mapping and the launchers one entry point borrows from
// another (the outer-product GEMM, the bf16 conversion).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <atomic>
#include <stdint.h>

#include "../../include/dust.h"

namespace dust {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Offsets of the pieces of a caller-owned workspace; every piece is 256-byte
// aligned.  The same function computes the layout for the size query and for
// the call, so the two always agree.
struct WsLayout {
    size_t used = 0;
    size_t take(size_t bytes) {
        used = static_cast<size_t>(round_up(static_cast<int64_t>(used), 256));
        const size_t off = used;
        used += bytes;
        return off;
    }
};

inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

#define DUST_CUDA_TRY(expr)                                    \
    do {                                                       \
        cudaError_t e_ = (expr);                               \
        if (e_ != cudaSuccess) {                               \
            (void)cudaGetLastError();                          \
            return DUST_ERR_CUDA;                              \
        }                                                      \
    } while (0)

// Raises a kernel's dynamic shared-memory limit once per device: the
// attribute belongs to the device that is current when it is set, so a
// process that drives several GPUs needs it on each (bit d of `done` records
// device d; a race only repeats a harmless call).
template <typename K>
inline cudaError_t set_smem_once(K kern, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launch-error check after a kernel launch.
inline dust_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DUST_OK : DUST_ERR_CUDA;
}

// Debug build: the first out-of-bounds index each source file's kernels met
// since the last read, as (file id << 32) | line, or 0 (always 0 in the
// release build); reading clears it.  File ids: 1 head, 2 interior,
// 3 embed, 4 gemm, 5 reforward, 6 attention, 7 attention_qk, 8 optim, 9 es,
// 10 abi (the index self-check).
uint64_t debug_fault_file_1();
uint64_t debug_fault_file_2();
uint64_t debug_fault_file_3();
uint64_t debug_fault_file_4();
uint64_t debug_fault_file_5();
uint64_t debug_fault_file_6();
uint64_t debug_fault_file_7();
uint64_t debug_fault_file_8();
uint64_t debug_fault_file_9();
uint64_t debug_fault_file_10();

// Optional event pairs around the dominant kernel of each entry point (the
// benchmark hook of dust_set_kernel_events).
struct KernelTimer {
    void* const* start = nullptr;
    void* const* stop = nullptr;
    int capacity = 0;
    int count = 0;
};
KernelTimer& kernel_timer();
inline void timer_begin(cudaStream_t s) {
    KernelTimer& k = kernel_timer();
    if (k.start && k.count < k.capacity)
        cudaEventRecord(static_cast<cudaEvent_t>(k.start[k.count]), s);
}
inline void timer_end(cudaStream_t s) {
    KernelTimer& k = kernel_timer();
    if (k.stop && k.count < k.capacity) {
        cudaEventRecord(static_cast<cudaEvent_t>(k.stop[k.count]), s);
        ++k.count;
    }
}

// G[m][n] = sum_k A(m,k) B(n,k) on the tensor cores (bf16 in, fp32 out).
// a_mn: A stored as K rows of M elements (row stride lda), else M rows of K.
// b_kmod > 0: B's K index wraps modulo b_kmod.  n_per_cta: 256-column tiles
// walked by one CTA.
dust_status gemm_bf16_launch(const void* A, bool a_mn, int64_t lda, const void* B, bool b_mn,
                             int64_t ldb, int64_t M, int64_t N, int64_t K, int64_t b_kmod,
                             int n_per_cta, float* G, int64_t ldg, uint32_t* status,
                             cudaStream_t s);

// Same contraction (both operands K-major) ending in the cross-entropy
// epilogue: rows ordered (token block of 128, draw, token in block) for
// ndraw draws starting at draw index i0; writes dl[(i0 + i) T + t] =
// log sum_v p[t][v] exp(dz_v) - dz_{targets[t]}; p has row stride ldp, a
// multiple of 4.
dust_status gemm_ce_launch(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M,
                           int64_t V, int64_t K, int64_t b_kmod, const float* p, int64_t ldp,
                           const int32_t* targets, int64_t T, int ndraw, int i0, float* dl,
                           uint32_t* status, cudaStream_t s);

// 2-D bf16 TMA descriptor (inner x outer elements, row stride in elements),
// 128-byte swizzle, box box_inner x box_outer, zero fill out of range.
bool encode_bf16_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                    int64_t stride_elems, uint32_t box_inner, uint32_t box_outer);
// The same for fp32 (box_inner 32: one 128-byte row of the box).
bool encode_f32_2d(CUtensorMap* map, const void* ptr, int64_t inner, int64_t outer,
                   int64_t stride_elems, uint32_t box_inner, uint32_t box_outer);

struct PhiloxKeys;

// From per-draw loss changes dl (K x T): the centring by the mean over draws,
// the gamma-discounted suffix scan per sequence (r, K x T), and
// g = -(1/(K sigma)) sum_i r a with the noise regenerated over C channels
// (C % 8 == 0), written as fp32 (g_hat, optional) and bf16 (gbf, T x C).
dust_status credit_and_ghat_launch(const float* dl, float* mean, float* r, int T, int seq_len,
                                   int C, const dust_noise& nz, const PhiloxKeys& keys,
                                   float* g_hat, __nv_bfloat16* gbf, cudaStream_t s);

// Interior GEMM 1 with its A operand (the GELU difference of the perturbed
// output, split bf16) generated on chip: du = dh W2^T for nd draws.  With A2
// non-null (seq_len a multiple of 128, T = Tp) the epilogue also runs the
// per-sequence EMA and writes A2 = [hi | lo] of de instead of du.
bool reforward1_supported(int64_t C, int64_t dm);
dust_status gelu_launch(const float* y, int64_t n, float* h, cudaStream_t s);
// Taylor coefficients (4 per channel, T x C/4 x 4 float4) of the GELU difference.
dust_status gelu_taylor_launch(const float* y, int64_t n, void* coef, cudaStream_t s);
dust_status reforward1_launch(const float* y1, const float* h0, const void* coef, bool taylor,
                              const void* W2, int64_t T, int64_t Tp, int64_t C,
                              int64_t dm, int nd, uint32_t draw_first, uint32_t token0,
                              uint32_t layer, float sigma, const PhiloxKeys& keys, float* du,
                              void* A2, int64_t seq_len, float lam, uint32_t* status,
                              cudaStream_t s);

// Host-side argument checks of the estimator entry points, workspace size
// included: exactly what each entry point verifies before it enqueues
// anything (the block scheduler runs them on every job first).
dust_status head_estimate_check(const float* logits, const int32_t* targets, const void* x,
                                dust_dtype x_dtype, int64_t T, int64_t V, int64_t d,
                                const dust_noise& nz, dust_baseline baseline, const float* g_hat,
                                const float* G_W, const void* ws, size_t ws_bytes);
dust_status linear_estimate_check(const void* x, const float* y1, const void* W2,
                                  float ema_decay, const void* W_head, const float* z_clean,
                                  const int32_t* targets, int64_t T, int64_t seq_len,
                                  int64_t d_in, int64_t C, int64_t d_model, int64_t V,
                                  const dust_noise& nz, const float* g_hat, const float* G_W1,
                                  const void* ws, size_t ws_bytes);
dust_status attn_value_check(const float* P, const float* E, const void* x, dust_dtype x_dtype,
                             int64_t T, int64_t seq_len, int64_t H, int64_t dv, int64_t d_in,
                             const dust_noise& nz, const float* g_hat, const float* G_W,
                             const void* ws, size_t ws_bytes);
dust_status attn_gate_check(const float* z, const float* o, const float* E, const void* x,
                            dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t C,
                            int64_t d_in, const dust_noise& nz, const float* g_hat,
                            const float* G_W, const void* ws, size_t ws_bytes);
dust_status attn_qk_check(int which, const float* Q, const float* Kk, const float* V,
                          const float* O, const float* P, const float* E, const void* x,
                          dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                          int64_t d_in, const dust_noise& nz, const float* g_hat,
                          const float* G_W, const void* ws, size_t ws_bytes);

// rows x cols fp32 (row stride ld_in) -> bf16 (row stride ld_out, padding
// columns set to zero).
dust_status f32_to_bf16_launch(const float* in, int64_t rows, int64_t cols, int64_t ld_in,
                               void* out, int64_t ld_out, cudaStream_t s);
// bf16 -> bf16 copy into a padded layout.
dust_status bf16_pad_launch(const void* in, int64_t rows, int64_t cols, int64_t ld_in,
                            void* out, int64_t ld_out, cudaStream_t s);

}  // namespace dust
