// embed.cu -- the embedding's weight gradient.  Its input is one-hot, so the
// outer product sum_t g_t onehot(id_t)^T is a scatter-add of g_t into row
// id_t (Dust translation, hn.213312.xyz, §2.2 信用分配, last sentences).
//
// Done without floating-point atomics so that the result is bitwise
// reproducible:
//   1. stable LSD radix sort of the ids (8-bit digits, 1024-token chunks):
//      perm lists the tokens ordered by (id, t);
//   2. every id's run of sorted tokens is cut into pieces of at most kPiece
//      tokens; a CTA sums one piece's rows of g in ascending t;
//   3. rows with one piece were written directly; rows with several pieces
//      add their partial sums in piece order; rows no token hits are zero.
#include <algorithm>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {
namespace {

constexpr int kChunk = 1024;   // tokens per radix-sort CTA
constexpr int kPiece = 32;     // tokens per partial row sum
constexpr int64_t kMaxT = 1LL << 26;
constexpr int64_t kMaxV = 1LL << 24;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Keys: valid ids as they are; an id outside [0, V) becomes V (sorted last,
// left out of every row) and is recorded in the status word.
__global__ void embed_keys_kernel(const int32_t* __restrict__ ids, int T, int V,
                                  uint32_t* __restrict__ keys, int32_t* __restrict__ vals,
                                  uint32_t* status) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    int id = ids[t];
    if (id < 0 || id >= V) {
        record_status(status, DUST_ERR_DEVICE_RANGE);
        id = V;
    }
    keys[t] = static_cast<uint32_t>(id);
    vals[t] = t;
}

// Per-chunk digit counts, stored digit-major: hist[digit * nchunks + chunk].
__global__ void __launch_bounds__(kChunk)
    radix_hist_kernel(const uint32_t* __restrict__ keys, int T, int shift, int nchunks,
                      uint32_t* __restrict__ hist) {
    __shared__ uint32_t cnt[256];
    const int c = blockIdx.x;
    if (threadIdx.x < 256) cnt[threadIdx.x] = 0;
    __syncthreads();
    const int i = c * kChunk + threadIdx.x;
    if (i < T) atomicAdd(&cnt[(keys[i] >> shift) & 255u], 1u);
    __syncthreads();
    if (threadIdx.x < 256) hist[static_cast<int64_t>(threadIdx.x) * nchunks + c] = cnt[threadIdx.x];
}

// Exclusive prefix sum of n words in one CTA of 1024 threads; out[n] = total.
// Block 1 of a two-block launch scans (in2, out2) instead, with each word w
// taken as ceil(w / kPiece) when pieces2 is set (the pieces of each id).
__global__ void __launch_bounds__(1024)
    exclusive_scan_kernel(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int64_t n,
                          const uint32_t* __restrict__ in2 = nullptr,
                          uint32_t* __restrict__ out2 = nullptr, int pieces2 = 0) {
    const bool second = blockIdx.x == 1;
    if (second) {
        in = in2;
        out = out2;
    }
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += 4 * 1024) {
        uint32_t v[4];
        uint32_t local = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = base + 4 * tid + k;
            v[k] = i < n ? in[i] : 0u;
            if (second && pieces2) v[k] = (v[k] + kPiece - 1) / kPiece;
            local += v[k];
        }
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = wsum[lane];
            uint32_t wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
                if (lane >= o) wi += y;
            }
            wsum[lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
        const uint32_t carry = carry_s;
        uint32_t run = carry + wsum[warp] + incl - local;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = base + 4 * tid + k;
            if (i < n) out[i] = run;
            run += v[k];
        }
        __syncthreads();
        if (tid == 1023) carry_s = run;
        __syncthreads();
    }
    if (tid == 0) out[n] = carry_s;
}

// Stable scatter of one radix pass.  Within a chunk the rank of a token among
// earlier tokens with the same digit is (tokens of that digit in earlier
// warps) + (earlier lanes of this warp with that digit).
__global__ void __launch_bounds__(kChunk)
    radix_scatter_kernel(const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
                         int T, int shift, int nchunks, const uint32_t* __restrict__ offs,
                         uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out) {
    __shared__ uint32_t wcnt[32][256];
    const int c = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int k = tid; k < 32 * 256; k += kChunk) (&wcnt[0][0])[k] = 0;
    __syncthreads();
    const int i = c * kChunk + tid;
    const bool valid = i < T;
    const uint32_t key = valid ? keys_in[i] : 0u;
    const uint32_t dig = valid ? (key >> shift) & 255u : 256u;  // 256: padding lane
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dig);
    const uint32_t lrank = __popc(peers & lanemask_lt());
    if (valid && lrank == 0) wcnt[warp][dig] = __popc(peers);
    __syncthreads();
    if (tid < 256) {
        uint32_t acc = 0;
        for (int w = 0; w < 32; ++w) {
            const uint32_t x = wcnt[w][tid];
            wcnt[w][tid] = acc;
            acc += x;
        }
    }
    __syncthreads();
    if (valid) {
        const uint32_t pos = offs[static_cast<int64_t>(dig) * nchunks + c] + wcnt[warp][dig] + lrank;
        keys_out[pos] = key;
        vals_out[pos] = vals_in[i];
    }
}

// counts[v] = number of sorted tokens with key v (keys sorted; v < V).
__global__ void key_counts_kernel(const uint32_t* __restrict__ keys, int T, int V,
                                  uint32_t* __restrict__ counts) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= T) return;
    const uint32_t key = keys[k];
    if (key >= static_cast<uint32_t>(V)) return;
    const bool first = (k == 0) || keys[k - 1] != key;
    if (!first) return;
    int e = k + 1;  // run end by binary search over the sorted keys
    int lo = k + 1, hi = T;
    while (lo < hi) {
        const int mid = lo + ((hi - lo) >> 1);
        if (keys[mid] == key) lo = mid + 1; else hi = mid;
    }
    e = lo;
    counts[key] = static_cast<uint32_t>(e - k);
}

struct Piece {
    int32_t v, start, len, multi;
};

__global__ void piece_table_kernel(const uint32_t* __restrict__ seg, const uint32_t* __restrict__ counts,
                                   const uint32_t* __restrict__ poff, int V, Piece* __restrict__ table) {
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= V) return;
    const uint32_t n = counts[v], p0 = poff[v], np = poff[v + 1] - p0;
    for (uint32_t k = 0; k < np; ++k) {
        Piece pc;
        pc.v = v;
        pc.start = static_cast<int32_t>(seg[v] + k * kPiece);
        pc.len = static_cast<int32_t>(min(static_cast<uint32_t>(kPiece), n - k * kPiece));
        pc.multi = np > 1;
        table[p0 + k] = pc;
    }
}

// One CTA per piece: rows g[perm[start .. start+len)] summed in that order.
// The piece's token indices are staged in shared memory first, so the row
// loads of a thread do not wait on index loads and can all be in flight.
template <bool VEC>
__global__ void piece_sum_kernel(const float* __restrict__ g, const int32_t* __restrict__ perm,
                                 const Piece* __restrict__ table, const uint32_t* __restrict__ poff,
                                 int V, int d, float* __restrict__ G_E, float* __restrict__ partial) {
    __shared__ int32_t rows[kPiece];
    const int npieces = static_cast<int>(poff[V]);
    for (int pi = blockIdx.x; pi < npieces; pi += gridDim.x) {
        const Piece pc = table[pi];
        __syncthreads();
        if (threadIdx.x < pc.len) rows[threadIdx.x] = __ldg(perm + pc.start + threadIdx.x);
        __syncthreads();
        float* dst = pc.multi ? partial + static_cast<int64_t>(pi) * d
                              : G_E + static_cast<int64_t>(pc.v) * d;
        if (VEC) {
            const int d4 = d >> 2;
            for (int c = threadIdx.x; c < d4; c += blockDim.x) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                for (int r = 0; r < pc.len; ++r) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(
                                               g + static_cast<int64_t>(rows[r]) * d) + c);
                    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
                }
                reinterpret_cast<float4*>(dst)[c] = acc;
            }
        } else {
            for (int c = threadIdx.x; c < d; c += blockDim.x) {
                float acc = 0.f;
#pragma unroll 8
                for (int r = 0; r < pc.len; ++r) acc += __ldg(g + static_cast<int64_t>(rows[r]) * d + c);
                dst[c] = acc;
            }
        }
    }
}

// Rows with no token -> 0; rows with several pieces -> sum of partials in
// piece order; rows with one piece are already final.  blockIdx.y = row.
template <bool VEC>
__global__ void rows_finish_kernel(const uint32_t* __restrict__ poff, int V, int d,
                                   const float* __restrict__ partial, float* __restrict__ G_E) {
    for (int v = blockIdx.y; v < V; v += gridDim.y) {
        const uint32_t p0 = __ldg(poff + v), np = __ldg(poff + v + 1) - p0;
        if (np == 1) continue;
        const int w = VEC ? d >> 2 : d;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < w; c += gridDim.x * blockDim.x) {
            if (VEC) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (uint32_t k = 0; k < np; ++k) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(
                                               partial + static_cast<int64_t>(p0 + k) * d) + c);
                    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
                }
                reinterpret_cast<float4*>(G_E + static_cast<int64_t>(v) * d)[c] = acc;
            } else {
                float acc = 0.f;
                for (uint32_t k = 0; k < np; ++k)
                    acc += __ldg(partial + static_cast<int64_t>(p0 + k) * d + c);
                G_E[static_cast<int64_t>(v) * d + c] = acc;
            }
        }
    }
}

struct EmbedPlan {
    int nchunks, passes;
    int64_t np_max;
    size_t off_k0, off_v0, off_k1, off_v1, off_hist, off_offs, off_cnt, off_seg, off_poff,
        off_table, off_part, bytes;
};

EmbedPlan embed_plan(int64_t T, int64_t d, int64_t V) {
    EmbedPlan P{};
    P.nchunks = static_cast<int>(ceil_div(T > 0 ? T : 1, kChunk));
    int bits = 1;
    while ((1LL << bits) <= V) ++bits;  // keys are in [0, V]
    P.passes = (bits + 7) / 8;
    P.np_max = ceil_div(T, kPiece) + (T < V ? T : V) + 1;
    const size_t Tn = static_cast<size_t>(T > 0 ? T : 1);
    const size_t Vn = static_cast<size_t>(V) + 1;
    WsLayout w;
    w.take(kCtlBytes);
    P.off_k0 = w.take(Tn * 4);
    P.off_v0 = w.take(Tn * 4);
    P.off_k1 = w.take(Tn * 4);
    P.off_v1 = w.take(Tn * 4);
    P.off_hist = w.take(static_cast<size_t>(256) * P.nchunks * 4);
    P.off_offs = w.take((static_cast<size_t>(256) * P.nchunks + 1) * 4);
    P.off_cnt = w.take(Vn * 4);
    P.off_seg = w.take(Vn * 4);
    P.off_poff = w.take(Vn * 4);
    P.off_table = w.take(static_cast<size_t>(P.np_max) * sizeof(Piece));
    P.off_part = w.take(static_cast<size_t>(P.np_max) * static_cast<size_t>(d) * 4);
    P.bytes = w.used;
    return P;
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" size_t dust_embed_workspace(int64_t T, int64_t d, int64_t V) {
    if (T < 0 || d < 1 || V < 1 || T > kMaxT || V > kMaxV) return 0;
    return embed_plan(T, d, V).bytes;
}

extern "C" dust_status dust_embed_scatter(const float* g_hat, const int32_t* ids, int64_t T,
                                          int64_t d, int64_t V, float* G_E, int32_t* perm_out,
                                          void* ws, size_t ws_bytes, void* stream) {
    if (!G_E || d < 1 || V < 1 || T < 0) return DUST_ERR_INVALID_ARG;
    if (T > 0 && (!g_hat || !ids)) return DUST_ERR_INVALID_ARG;
    if (T > kMaxT || V > kMaxV || d > (1LL << 24)) return DUST_ERR_UNSUPPORTED;
    const EmbedPlan P = embed_plan(T, d, V);
    if (!ws || ws_bytes < P.bytes || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint32_t* status = static_cast<uint32_t*>(ws);
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
    if (T == 0) {
        DUST_CUDA_TRY(cudaMemsetAsync(G_E, 0, static_cast<size_t>(V * d) * 4, s));
        return DUST_OK;
    }
    const int Ti = static_cast<int>(T), Vi = static_cast<int>(V), di = static_cast<int>(d);
    uint32_t* k0 = reinterpret_cast<uint32_t*>(w + P.off_k0);
    int32_t* v0 = reinterpret_cast<int32_t*>(w + P.off_v0);
    uint32_t* k1 = reinterpret_cast<uint32_t*>(w + P.off_k1);
    int32_t* v1 = reinterpret_cast<int32_t*>(w + P.off_v1);
    uint32_t* hist = reinterpret_cast<uint32_t*>(w + P.off_hist);
    uint32_t* offs = reinterpret_cast<uint32_t*>(w + P.off_offs);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(w + P.off_cnt);
    uint32_t* seg = reinterpret_cast<uint32_t*>(w + P.off_seg);
    uint32_t* poff = reinterpret_cast<uint32_t*>(w + P.off_poff);
    Piece* table = reinterpret_cast<Piece*>(w + P.off_table);
    float* part = reinterpret_cast<float*>(w + P.off_part);
    dust_status st;

    const unsigned tb = static_cast<unsigned>(ceil_div(T, 256));
    embed_keys_kernel<<<tb, 256, 0, s>>>(ids, Ti, Vi, k0, v0, status);
    if ((st = launch_status()) != DUST_OK) return st;
    for (int pass = 0; pass < P.passes; ++pass) {
        const int shift = 8 * pass;
        // the last pass writes the permutation straight into perm_out
        int32_t* vout = (pass == P.passes - 1 && perm_out) ? perm_out : v1;
        radix_hist_kernel<<<P.nchunks, kChunk, 0, s>>>(k0, Ti, shift, P.nchunks, hist);
        exclusive_scan_kernel<<<1, 1024, 0, s>>>(hist, offs, static_cast<int64_t>(256) * P.nchunks);
        radix_scatter_kernel<<<P.nchunks, kChunk, 0, s>>>(k0, v0, Ti, shift, P.nchunks, offs, k1,
                                                          vout);
        if (vout != v1) v1 = vout;
        if ((st = launch_status()) != DUST_OK) return st;
        uint32_t* tk = k0; k0 = k1; k1 = tk;
        int32_t* tv = v0; v0 = v1; v1 = tv;
    }
    // k0/v0 now hold the sorted keys and the permutation.
    DUST_CUDA_TRY(cudaMemsetAsync(cnt, 0, static_cast<size_t>(V + 1) * 4, s));
    key_counts_kernel<<<tb, 256, 0, s>>>(k0, Ti, Vi, cnt);
    // segment starts and piece offsets in one launch
    exclusive_scan_kernel<<<2, 1024, 0, s>>>(cnt, seg, V, cnt, poff, 1);
    const unsigned vb = static_cast<unsigned>(ceil_div(V, 256));
    piece_table_kernel<<<vb, 256, 0, s>>>(seg, cnt, poff, Vi, table);
    if ((st = launch_status()) != DUST_OK) return st;
    // Pieces are at most np_max; launch enough CTAs to cover the usual count
    // and let the grid-stride loop take the rest.
    const bool vec = (d % 4 == 0) && aligned(g_hat, 16) && aligned(G_E, 16);
    // one CTA per piece
    const int threads = static_cast<int>(std::min<int64_t>(256, round_up(vec ? d / 4 : d, 32)));
    const unsigned pgrid = static_cast<unsigned>(std::min<int64_t>(P.np_max, 148 * 64));
    timer_begin(s);
    if (vec)
        piece_sum_kernel<true><<<pgrid, threads, 0, s>>>(g_hat, v0, table, poff, Vi, di, G_E,
                                                         part);
    else
        piece_sum_kernel<false><<<pgrid, threads, 0, s>>>(g_hat, v0, table, poff, Vi, di, G_E,
                                                          part);
    timer_end(s);
    if ((st = launch_status()) != DUST_OK) return st;
    {
        const int64_t w = vec ? d / 4 : d;
        const dim3 fg(static_cast<unsigned>(ceil_div(w, 128)),
                      static_cast<unsigned>(std::min<int64_t>(V, 65535)));
        if (vec)
            rows_finish_kernel<true><<<fg, 128, 0, s>>>(poff, Vi, di, part, G_E);
        else
            rows_finish_kernel<false><<<fg, 128, 0, s>>>(poff, Vi, di, part, G_E);
    }
    if ((st = launch_status()) != DUST_OK) return st;
    return DUST_OK;
}
