// dust_common.cuh -- device helpers shared by the engine's kernels: the
// workspace status word, bounded mbarrier waits, and thin inline-PTX wrappers
// for the sm_103a asynchronous machinery (TMA bulk tensor copies, mbarriers,
// tcgen05 tensor-memory MMAs).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dust.h"

namespace dust {

// Every workspace starts with this many bytes of control words; word 0 is the
// status word that kernels write a dust_status into.
constexpr size_t kCtlBytes = 256;

// Default limit of a bounded in-kernel wait.  Large next to any legitimate
// wait of these kernels (microseconds), small enough that a broken pipeline
// returns an error instead of holding the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void record_status(uint32_t* status, uint32_t code) {
    if (status != nullptr) atomicCAS(status, 0u, code);
}

// ------------------------------------------------------------ debug build ----
// In the debug build (-DDUST_DEBUG, libdust_debug.so) DUST_IB(i, n) checks a
// computed index against the extent of the buffer it addresses before the
// access it guards: an index outside [0, n) records the first such fault of
// its source file (the line) and the access is skipped instead of reaching
// memory.  In the release build DUST_IB is the constant true and compiles
// away.  DUST_IDX(i, w, n) is the form for code whose control flow must stay
// uniform across a warp (around warp-collective TMEM loads and barriers): for
// an access of w elements from index i it checks i and i + w - 1, records a
// fault the same way and yields index 0 in place of a bad i, so the access
// still happens, at the buffer's start (every such buffer holds at least w
// elements).  In release it is i.  DUST_DEBUG_READER(file_id) defines the host reader of a file's word.
#ifdef DUST_DEBUG
namespace {
__device__ unsigned long long g_debug_fault;  // 0, or the faulting line
}
__device__ __forceinline__ bool debug_in_bounds(int64_t i, int64_t n, unsigned line) {
    if (i >= 0 && i < n) return true;
    atomicCAS(&g_debug_fault, 0ull, static_cast<unsigned long long>(line));
    return false;
}
#define DUST_IB(i, n) \
    (::dust::debug_in_bounds(static_cast<int64_t>(i), static_cast<int64_t>(n), __LINE__))
#define DUST_IDX(i, w, n)                                                   \
    (DUST_IB(i, n) && DUST_IB(static_cast<int64_t>(i) + (w) - 1, n) ? static_cast<int64_t>(i) \
                                                                      : int64_t{0})
#define DUST_DEBUG_READER(file_id)                                                     \
    uint64_t debug_fault_file_##file_id() {                                            \
        unsigned long long v = 0, zero = 0;                                            \
        if (cudaMemcpyFromSymbol(&v, g_debug_fault, sizeof(v)) != cudaSuccess ||       \
            cudaMemcpyToSymbol(g_debug_fault, &zero, sizeof(zero)) != cudaSuccess) {   \
            (void)cudaGetLastError();                                                  \
            return ~0ull;                                                              \
        }                                                                              \
        return v ? ((static_cast<uint64_t>(file_id) << 32) | v) : 0;                   \
    }
#else
#define DUST_IB(i, n) true
#define DUST_IDX(i, w, n) (i)
#define DUST_DEBUG_READER(file_id) \
    uint64_t debug_fault_file_##file_id() { return 0; }
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns, records DUST_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) {
            record_status(status, DUST_ERR_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------ TMA ----
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// -------------------------------------------------------------- tcgen05 ----
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     slot_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
// lbo / sbo are byte offsets: for a K-major tile sbo is the distance between
// 8-row groups (lbo unused); for an MN-major tile lbo is the distance between
// 64-element MN chunks and sbo the distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version of the tcgen05 family
    d |= 2ull << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with bf16 operands and an fp32
// accumulator: M = 128 rows, N columns, A/B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                  // D: f32
           | (1u << 7) | (1u << 10)                   // A, B: bf16
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the mbarrier when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace dust
