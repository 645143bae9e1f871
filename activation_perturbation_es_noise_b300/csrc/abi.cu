// abi.cu -- status strings, the workspace status read-back and the noise
// regenerator test hooks.
#include "dust_common.cuh"
#include "internal.h"
#include "noise.cuh"

namespace dust {
namespace {

// One thread per (token, channel block of 4): the words and normals of the
// block, written for the channels below nchan.
__global__ void philox_fill_kernel(PhiloxKeys keys, uint32_t layer, uint32_t draw,
                                   uint32_t token0, int64_t ntok, int64_t nchan,
                                   uint32_t* __restrict__ words, float* __restrict__ normals) {
    const int64_t nblk = (nchan + 3) / 4;
    const int64_t n = ntok * nblk;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / nblk, j = i - t * nblk;
        const uint4 w = philox4x32_10(static_cast<uint32_t>(j), token0 + static_cast<uint32_t>(t),
                                      draw, layer, keys);
        const float4 a = words_to_normals(w);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = 4 * j + k;
            if (c < nchan) {
                if (words) words[t * nchan + c] = wv[k];
                if (normals) normals[t * nchan + c] = av[k];
            }
        }
    }
}

// The kernels' fast Box-Muller at scale 1: one thread per two pairs of words
// through words_to_normals_fast (the packed form every estimator kernel
// runs), and the last pair of an odd count through box_muller_fast (the
// scalar form it must equal bit for bit).
__global__ void box_muller_fast_kernel(const uint2* __restrict__ words, int64_t npairs,
                                       float2* __restrict__ normals) {
    const int64_t nquads = npairs / 2;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i <= nquads;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i < nquads) {
            const uint2 w0 = words[2 * i], w1 = words[2 * i + 1];
            const float4 a = words_to_normals_fast(make_uint4(w0.x, w0.y, w1.x, w1.y), kClogUnit);
            normals[2 * i] = make_float2(a.x, a.y);
            normals[2 * i + 1] = make_float2(a.z, a.w);
        } else if (2 * nquads < npairs) {
            const uint2 w = words[2 * nquads];
            float2 a;
            box_muller_fast(w.x, w.y, a.x, a.y, kClogUnit);
            normals[2 * nquads] = a;
        }
    }
}

// Waits on an mbarrier that nothing arrives at, with the caller's limit, the
// way every pipeline wait in the library is bounded; records
// DUST_ERR_TIMEOUT when the limit runs out and returns.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(b, 0, status, limit_ns);
    __syncthreads();
}

// The debug build's index check on its own: one thread evaluates the check
// of index i against extent n and writes whether it passed.  Nothing is
// addressed with i, so an out-of-range i only records the fault (in the
// debug build; the release check is the constant true).
__global__ void debug_check_index_kernel(int64_t i, int64_t n, int* in_bounds) {
    *in_bounds = DUST_IB(i, n) ? 1 : 0;
}

// Issue-rate probe: every thread runs `iters` rounds over eight independent
// chains of one operation kind, so that throughput, not latency, bounds it.
//   kind 0: the Philox step, a 32 x 32 -> 64-bit multiply and an xor of its
//           halves (2 operations per chain and round);
//   kind 1: ex2.approx (1 XU operation per chain and round);
//   kind 2: fp32 fma (1 operation per chain and round);
//   kind 5: packed fp32 fma, fma.rn.f32x2 (2 operations per chain and round).
// The chains' results go to `sink` so that nothing is optimised away.
__global__ void __launch_bounds__(256) issue_probe_kernel(int kind, int64_t iters,
                                                          uint32_t* sink) {
    const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t acc = 0;
    if (kind == 0) {
        uint32_t x[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = tid * 2654435761u + c;
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint64_t pr = static_cast<uint64_t>(x[c]) * 0xD2511F53u;
                x[c] = static_cast<uint32_t>(pr >> 32) ^ static_cast<uint32_t>(pr);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc ^= x[c];
    } else if (kind == 3 || kind == 4) {
        // the same step with the product's halves as two 32-bit multiplies,
        // written as PTX (3) or as C (4)
        uint32_t x[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = tid * 2654435761u + c;
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t lo, hi;
                if (kind == 3) {
                    asm("mul.lo.u32 %0, %1, %2;" : "=r"(lo) : "r"(x[c]), "r"(0xD2511F53u));
                    asm("mul.hi.u32 %0, %1, %2;" : "=r"(hi) : "r"(x[c]), "r"(0xD2511F53u));
                } else {
                    lo = x[c] * 0xD2511F53u;
                    hi = __umulhi(x[c], 0xD2511F53u);
                }
                x[c] = hi ^ lo;
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc ^= x[c];
    } else if (kind == 5) {
        float2 f[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            f[c] = make_float2(0.001f * static_cast<float>((tid + c) & 255),
                               0.002f * static_cast<float>((tid + c) & 127));
        const float2 m = make_float2(0.999f, 0.998f), k = make_float2(0.0001f, 0.0002f);
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int c = 0; c < 8; ++c) f[c] = fma2(f[c], m, k);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc ^= __float_as_uint(f[c].x) ^ __float_as_uint(f[c].y);
    } else if (kind == 1) {
        float f[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) f[c] = 0.001f * static_cast<float>((tid + c) & 255);
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float y;
                asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(-f[c]));
                f[c] = y;  // stays in (0, 1]
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc ^= __float_as_uint(f[c]);
    } else {
        float f[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) f[c] = 0.001f * static_cast<float>((tid + c) & 255);
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int c = 0; c < 8; ++c) f[c] = fmaf(f[c], 0.999f, 0.0001f);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc ^= __float_as_uint(f[c]);
    }
    if (acc == 0x12345678u) sink[tid & 255] = acc;  // practically never taken
}

}  // namespace

KernelTimer& kernel_timer() {
    static KernelTimer t;
    return t;
}

}  // namespace dust

using namespace dust;

extern "C" dust_status dust_set_kernel_events(void* const* start_events, void* const* stop_events,
                                              int capacity) {
    KernelTimer& k = kernel_timer();
    if ((start_events == nullptr) != (stop_events == nullptr) || capacity < 0)
        return DUST_ERR_INVALID_ARG;
    k.start = start_events;
    k.stop = stop_events;
    k.capacity = start_events ? capacity : 0;
    k.count = 0;
    return DUST_OK;
}

extern "C" int dust_kernel_event_count(void) { return kernel_timer().count; }

extern "C" dust_status dust_wait_selftest(void* ws, uint64_t limit_ns, void* stream) {
    if (!ws || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<uint32_t*>(ws), limit_ns);
    return launch_status();
}

extern "C" dust_status dust_debug_check_index(int64_t i, int64_t n, int* in_bounds,
                                              void* stream) {
    if (!in_bounds || !aligned(in_bounds, 4)) return DUST_ERR_INVALID_ARG;
    debug_check_index_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(i, n, in_bounds);
    return launch_status();
}

extern "C" int dust_abi_version(void) { return 100; }

extern "C" const char* dust_status_string(dust_status s) {
    switch (s) {
        case DUST_OK: return "ok";
        case DUST_ERR_INVALID_ARG: return "invalid argument";
        case DUST_ERR_UNSUPPORTED: return "size not supported";
        case DUST_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case DUST_ERR_CUDA: return "CUDA call failed";
        case DUST_ERR_TIMEOUT: return "bounded in-kernel wait ran out";
        case DUST_ERR_DEVICE_RANGE: return "device-side id out of range";
    }
    return "unknown status";
}

extern "C" dust_status dust_workspace_status(void* ws, void* stream, dust_status* status_out) {
    if (!ws || !status_out || !aligned(ws, 256)) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    DUST_CUDA_TRY(cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s));
    DUST_CUDA_TRY(cudaStreamSynchronize(s));
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(word), s));
    *status_out = static_cast<dust_status>(word);
    return DUST_OK;
}

extern "C" dust_status dust_philox_fill(uint64_t seed, uint32_t layer, uint32_t draw,
                                        int64_t token0, int64_t ntok, int64_t nchan,
                                        uint32_t* words, float* normals, void* stream) {
    if (ntok < 0 || nchan < 0 || token0 < 0) return DUST_ERR_INVALID_ARG;
    if (token0 + ntok > (1LL << 32)) return DUST_ERR_INVALID_ARG;
    if (nchan > (1LL << 34)) return DUST_ERR_UNSUPPORTED;
    if (ntok == 0 || nchan == 0) return DUST_OK;
    if (!words && !normals) return DUST_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t n = ntok * ((nchan + 3) / 4);
    int64_t blocks = ceil_div(n, 256);
    if (blocks > 148 * 64) blocks = 148 * 64;
    philox_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        philox_round_keys(seed), layer, draw, static_cast<uint32_t>(token0), ntok, nchan, words,
        normals);
    return launch_status();
}

extern "C" dust_status dust_box_muller_fast(const uint32_t* words, int64_t npairs,
                                            float* normals, void* stream) {
    if (npairs < 0 || npairs > (1LL << 40)) return DUST_ERR_INVALID_ARG;
    if (npairs == 0) return DUST_OK;
    if (!words || !normals || !aligned(words, 8) || !aligned(normals, 8))
        return DUST_ERR_INVALID_ARG;
    int64_t blocks = ceil_div(npairs, 256);
    if (blocks > 148 * 64) blocks = 148 * 64;
    box_muller_fast_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                             static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint2*>(words), npairs, reinterpret_cast<float2*>(normals));
    return launch_status();
}

extern "C" dust_status dust_issue_probe(int kind, int64_t iters, int64_t* threads_out,
                                        void* sink, void* stream) {
    if (kind < 0 || kind > 5 || iters < 1 || iters > (1LL << 32) || !threads_out || !sink ||
        !aligned(sink, 4))
        return DUST_ERR_INVALID_ARG;
    constexpr int kBlocks = 148 * 8, kThreads = 256;
    *threads_out = static_cast<int64_t>(kBlocks) * kThreads;
    issue_probe_kernel<<<kBlocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        kind, iters, static_cast<uint32_t*>(sink));
    return launch_status();
}

extern "C" int dust_debug_build(void) {
#ifdef DUST_DEBUG
    return 1;
#else
    return 0;
#endif
}

extern "C" uint64_t dust_debug_fault(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) {
        (void)cudaGetLastError();
        return ~0ull;
    }
    uint64_t (*const readers[])() = {debug_fault_file_1, debug_fault_file_2, debug_fault_file_3,
                                     debug_fault_file_4, debug_fault_file_5, debug_fault_file_6,
                                     debug_fault_file_7, debug_fault_file_8, debug_fault_file_9,
                                     debug_fault_file_10};
    uint64_t first = 0;
    for (auto r : readers) {
        const uint64_t v = r();
        if (v && !first) first = v;
    }
    return first;
}

namespace dust {
DUST_DEBUG_READER(10)
}  // namespace dust
