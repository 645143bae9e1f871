// embed.cu -- the embedding's weight gradient.  Its input is one-hot, so the
// outer product sum_t g_t onehot(id_t)^T is a scatter-add of g_t into row
// id_t (Dust translation, hn.213312.xyz, §2.2 信用分配, last sentences).
//
// Done without floating-point atomics so that the result is bitwise
// reproducible, in two launches after one memset (the control words, every
// counter and the rows kernel's completion counters):
//   1. sort, one cooperative launch.  For up to 8190 ids and 64 chunks of
//      1024 tokens (the pages' 4096-token vocabulary over a batch) it is the
//      counting pass of embed_count_sort_kernel below: one grid barrier.
//      Otherwise (a bounded grid-wide barrier between radix passes): per
//      1024-token chunk
//      the sort keys (an id outside [0, V) becomes V, sorted last and left
//      out), the first pass's digit counts and every id's token count
//      (integer atomics, warp-aggregated: the same sums in any order); then
//      one stable LSD radix scatter per 8-bit digit, each CTA deriving its
//      chunk's scatter offsets from the digit counts of all chunks and
//      counting the next pass's digits per output chunk; the last pass writes
//      the permutation (tokens ordered by (id, t)).  Alongside, CTA 0 scans
//      the id counts into segment starts, piece offsets (pieces of at most
//      kPiece sorted tokens of one id) and the offsets of the ids no token
//      hits, and every CTA then writes part of the piece table and the list
//      of empty ids;
//   2. rows: one warp per work unit, (piece, 512-column slice) or (empty id,
//      slice).  A piece sums its rows of g in ascending t; a row with one
//      piece is written directly.  A row with several writes partials and
//      adds them as a two-level tree in a fixed order: the warp that finishes
//      the last piece of a group of kGroup consecutive pieces (an integer
//      counter per group and slice) adds the group's partials in piece order
//      into the group's first partial, and the warp that finishes the row's
//      last group adds the group sums in group order.  Empty rows are zero.
#include <algorithm>
#include <atomic>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {
namespace {

constexpr int kChunk = 1024;   // tokens per radix-sort chunk (one CTA's threads)
constexpr int kPiece = 32;     // tokens per partial row sum
constexpr int kGroup = 8;      // partials added together at the first level
// (wider slices, 256 and 384 float4 columns, measured slower: more registers, fewer warps)
constexpr int kSliceF4 = 128;  // float4 columns (512 floats) per row work unit
constexpr int kSliceF = 128;   // float columns per work unit without float4 rows
constexpr int kLaneF4 = kSliceF4 / 32;  // float4 columns of a lane
constexpr int kLaneF = kSliceF / 32;    // float columns of a lane
constexpr int kRowThreads = 256;
constexpr int64_t kMaxT = 1LL << 26;
// The counting pass, for few ids and few tokens (the pages' 4096-token
// vocabulary over one batch): every CTA takes one chunk, sorts it stably in
// shared memory and counts its ids; after one grid barrier every CTA finds
// each id's place from all chunks' counts.  Keys are below 8192 (13 bits; 8191
// pads a chunk's tail).
constexpr int kCountV = 8190;       // largest V the counting pass takes
constexpr int kCountBins = 8192;
constexpr int kCountChunks = 64;    // largest chunk count it takes
constexpr uint32_t kPadKey = 8191u;
constexpr size_t kCountSmem = (4 * kCountBins + 8 + 4 * 1024 + 32 * 128 + 128 + 4 * 32 + 32) * 4;
constexpr int64_t kMaxV = 1LL << 24;

// Control words after the status word (word 0) of the workspace.
enum { kBarCount = 8,   // grid barrier: CTAs arrived
       kBarGen = 9,     // grid barrier: generation
       kNPieces = 16,   // pieces in the table
       kNEmpty = 17 };  // ids no token hits

struct Piece {
    int32_t v, start, len, multi;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive prefix sums of NC word sequences at once, over n elements, by one
// CTA of 1024 threads (4096 elements per round, with carries); f(i, v) fills
// v[0..NC) for element i, out[c][i] receives the prefixes, tot[c] the totals.
// Every thread of the CTA must call it.
template <int NC, typename F>
__device__ void cta_exclusive_scan(int64_t n, F f, uint32_t* const (&out)[NC],
                                   uint32_t (&tot)[NC]) {
    __shared__ uint32_t wsum[NC][32];
    __shared__ uint32_t carry[NC];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < NC) carry[tid] = 0;
    __syncthreads();
    for (int64_t base = 0; base < n; base += 4 * 1024) {
        uint32_t v[4][NC], local[NC], incl[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) local[c] = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t i = base + 4 * tid + k;
            if (i < n) {
                f(i, v[k]);
            } else {
#pragma unroll
                for (int c = 0; c < NC; ++c) v[k][c] = 0;
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) local[c] += v[k][c];
        }
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            incl[c] = local[c];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl[c], o);
                if (lane >= o) incl[c] += y;
            }
            if (lane == 31) wsum[c][warp] = incl[c];
        }
        __syncthreads();
        if (warp < NC) {
            const uint32_t w = wsum[warp][lane];
            uint32_t wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
                if (lane >= o) wi += y;
            }
            wsum[warp][lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            uint32_t run = carry[c] + wsum[c][warp] + incl[c] - local[c];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t i = base + 4 * tid + k;
                if (i < n) out[c][i] = run;
                run += v[k][c];
            }
            if (tid == 1023) incl[c] = run;  // this round's end
        }
        __syncthreads();
        if (tid == 1023) {
#pragma unroll
            for (int c = 0; c < NC; ++c) carry[c] = incl[c];
        }
        __syncthreads();
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) tot[c] = carry[c];
    __syncthreads();  // every thread has read the totals before carry[] is reused
}

// Grid-wide barrier of the cooperative sort launch (all CTAs resident):
// ctl[kBarCount] counts arrivals, the last arriver resets it and bumps
// ctl[kBarGen].  The wait is bounded: past kWaitLimitNs the CTA records
// DUST_ERR_TIMEOUT and the barrier returns false in all its threads.
__device__ bool grid_barrier(uint32_t* ctl) {
    __shared__ bool ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile uint32_t* gen = ctl + kBarGen;
        const uint32_t g0 = *gen;
        __threadfence();
        bool good = true;
        if (atomicAdd(ctl + kBarCount, 1u) + 1 == gridDim.x) {
            atomicExch(ctl + kBarCount, 0u);
            __threadfence();
            atomicAdd(ctl + kBarGen, 1u);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (*gen == g0) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    record_status(ctl, DUST_ERR_TIMEOUT);
                    good = false;
                    break;
                }
            }
        }
        __threadfence();
        ok = good;
    }
    __syncthreads();
    return ok;
}

struct SortArgs {
    const int32_t* ids;
    int T, V, nchunks, passes, nslices;
    uint32_t* keys[2];  // ping-pong sort keys (id, or V for an invalid id)
    int32_t* vals[2];   // ping-pong token indices
    int32_t* perm_out;  // the last pass's values, or null
    uint32_t* hist;     // passes x 256 x nchunks digit counts
    uint32_t* offs;     // their exclusive prefix sums
    uint32_t* cnt;      // V tokens per id
    uint32_t* seg;      // V first sorted position of every id
    uint32_t* poff;     // V + 1 first piece of every id
    uint32_t* eoff;     // V empty ids before every id
    Piece* table;
    int32_t* empty;     // ids with no token, in order
    uint32_t* row_done; // V x nslices counters of the rows kernel (zeroed by the caller)
    uint32_t* group_done;  // np_max x nslices counters of the rows kernel (zeroed by the caller)
    int64_t np_max;
    uint32_t* ctl;      // workspace control words (status word 0)
    uint32_t* chist;    // counting pass: (V + 1) x nchp tokens per id and chunk (zeroed)
    int nchp;
    int32_t* perm_dst;  // counting pass: where the permutation goes
};

// offs[d] for chunk c: tokens of every chunk with a smaller digit, plus
// tokens of digit d in earlier chunks (the exclusive prefix of the
// digit-major counts hist[d][c]).  Threads 0..255 take one digit each.
__device__ void chunk_offsets(const uint32_t* hist, int nchunks, int c, uint32_t* offs) {
    __shared__ uint32_t tot[256];
    const int tid = threadIdx.x;
    uint32_t pre = 0;
    if (tid < 256) {
        uint32_t t = 0;
        const uint32_t* row = hist + static_cast<int64_t>(tid) * nchunks;
        for (int k = 0; k < nchunks; ++k) {
            const uint32_t h =
                DUST_IB(static_cast<int64_t>(tid) * nchunks + k, static_cast<int64_t>(256) * nchunks)
                    ? __ldcg(row + k)
                    : 0u;
            pre += k < c ? h : 0u;
            t += h;
        }
        tot[tid] = t;
    }
    __syncthreads();
    if (tid < 32) {  // exclusive scan of the 256 digit totals, 8 per lane
        uint32_t v[8], local = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[k] = tot[8 * tid + k];
            local += v[k];
        }
        uint32_t incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (tid >= o) incl += y;
        }
        uint32_t run = incl - local;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            tot[8 * tid + k] = run;
            run += v[k];
        }
    }
    __syncthreads();
    if (tid < 256) offs[tid] = tot[tid] + pre;
    __syncthreads();
}

__global__ void __launch_bounds__(kChunk) embed_sort_kernel(const SortArgs a) {
    __shared__ uint32_t wcnt[32][256];
    __shared__ uint32_t choffs[256];
    const int tid = threadIdx.x;
    const int64_t gthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
    const int64_t hist_words = static_cast<int64_t>(256) * a.nchunks;


    // Keys, the first digit's counts per chunk, tokens per id (cnt and the
    // later passes' digit counts were cleared by the caller's memset).
    uint32_t* h = &wcnt[0][0];
    for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
        __syncthreads();
        if (tid < 256) h[tid] = 0;
        __syncthreads();
        const int t = c * kChunk + tid;
        const bool valid = t < a.T;
        uint32_t key = 0xFFFFFFFFu;
        if (valid && DUST_IB(t, a.T)) {
            int id = __ldg(a.ids + t);
            if (id < 0 || id >= a.V) {
                record_status(a.ctl, DUST_ERR_DEVICE_RANGE);
                id = a.V;
            }
            key = static_cast<uint32_t>(id);
            a.keys[0][t] = key;
            a.vals[0][t] = t;
            atomicAdd(&h[key & 255u], 1u);
        }
        // one atomic per distinct id in the warp
        const bool counted = valid && key < static_cast<uint32_t>(a.V);
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, counted ? key : 0xFFFFFFFFu);
        if (counted && (peers & lanemask_lt()) == 0 && DUST_IB(key, a.V))
            atomicAdd(a.cnt + key, __popc(peers));
        __syncthreads();
        if (tid < 256 && DUST_IB(static_cast<int64_t>(tid) * a.nchunks + c, hist_words))
            a.hist[static_cast<int64_t>(tid) * a.nchunks + c] = h[tid];
    }

    int cur = 0;
    for (int pass = 0; pass < a.passes; ++pass) {
        if (!grid_barrier(a.ctl)) return;
        if (pass == 1) {
            // the piece table and the empty-id list (offsets from CTA 0, before
            // the barrier just passed)
            for (int64_t v = gtid; v < a.V; v += gthreads) {
                const uint32_t n = __ldcg(a.cnt + v);
                if (n == 0) {
                    const uint32_t e = __ldcg(a.eoff + v);
                    if (DUST_IB(e, a.V)) a.empty[e] = static_cast<int32_t>(v);
                    continue;
                }
                const uint32_t p0 = __ldcg(a.poff + v), s0 = __ldcg(a.seg + v);
                const uint32_t np = (n + kPiece - 1) / kPiece;
                for (uint32_t k = 0; k < np; ++k) {
                    Piece pc;
                    pc.v = static_cast<int32_t>(v);
                    pc.start = static_cast<int32_t>(s0 + k * kPiece);
                    pc.len = static_cast<int32_t>(min(static_cast<uint32_t>(kPiece), n - k * kPiece));
                    pc.multi = np > 1;
                    if (DUST_IB(p0 + k, a.np_max)) a.table[p0 + k] = pc;
                }
            }
        }
        const bool last = pass == a.passes - 1;
        const uint32_t* hist_cur = a.hist + pass * hist_words;
        uint32_t* hist_next = last ? nullptr : a.hist + (pass + 1) * hist_words;
        const uint32_t* keys_in = a.keys[cur];
        const int32_t* vals_in = a.vals[cur];
        uint32_t* keys_out = a.keys[cur ^ 1];
        int32_t* vals_out = (last && a.perm_out) ? a.perm_out : a.vals[cur ^ 1];
        const int shift = 8 * pass;
        const int lane = tid & 31, warp = tid >> 5;
        // Stable scatter of each chunk of this CTA: the rank of a token among
        // earlier tokens of its chunk with the same digit is (tokens of that
        // digit in earlier warps) + (earlier lanes of this warp with it).
        for (int c = blockIdx.x; c < a.nchunks; c += gridDim.x) {
            chunk_offsets(hist_cur, a.nchunks, c, choffs);
            for (int k = tid; k < 32 * 256; k += kChunk) (&wcnt[0][0])[k] = 0;
            __syncthreads();
            const int i = c * kChunk + tid;
            const bool valid = i < a.T;
            const uint32_t key = (valid && DUST_IB(i, a.T)) ? __ldcg(keys_in + i) : 0u;
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
                const uint32_t pos = choffs[dig] + wcnt[warp][dig] + lrank;
                if (DUST_IB(pos, a.T) && DUST_IB(i, a.T)) {
                    keys_out[pos] = key;
                    vals_out[pos] = __ldcg(vals_in + i);
                }
                if (hist_next) {
                    const uint32_t d2 = (key >> (shift + 8)) & 255u;
                    const int64_t hi = static_cast<int64_t>(d2) * a.nchunks + pos / kChunk;
                    if (DUST_IB(hi, hist_words)) atomicAdd(hist_next + hi, 1u);
                }
            }
            __syncthreads();  // wcnt and choffs are reused by the next chunk
        }
        if (pass == 0 && blockIdx.x == 0) {
            // segment starts, piece offsets and empty-id offsets of every id
            uint32_t* const out[3] = {a.seg, a.poff, a.eoff};
            uint32_t tot[3];
            cta_exclusive_scan<3>(a.V,
                                  [&](int64_t v, uint32_t* x) {
                                      const uint32_t n = __ldcg(a.cnt + v);
                                      x[0] = n;
                                      x[1] = (n + kPiece - 1) / kPiece;
                                      x[2] = n == 0 ? 1u : 0u;
                                  },
                                  out, tot);
            if (tid == 0) {
                a.poff[a.V] = tot[1];
                a.ctl[kNPieces] = tot[1];
                a.ctl[kNEmpty] = tot[2];
            }
        }
        cur ^= 1;
    }
    if (a.passes == 1) {  // (V < 256: no second pass to build the table beside)
        if (!grid_barrier(a.ctl)) return;
        for (int64_t v = gtid; v < a.V; v += gthreads) {
            const uint32_t n = __ldcg(a.cnt + v);
            if (n == 0) {
                const uint32_t e = __ldcg(a.eoff + v);
                if (DUST_IB(e, a.V)) a.empty[e] = static_cast<int32_t>(v);
                continue;
            }
            const uint32_t p0 = __ldcg(a.poff + v), s0 = __ldcg(a.seg + v);
            const uint32_t np = (n + kPiece - 1) / kPiece;
            for (uint32_t k = 0; k < np; ++k) {
                Piece pc;
                pc.v = static_cast<int32_t>(v);
                pc.start = static_cast<int32_t>(s0 + k * kPiece);
                pc.len = static_cast<int32_t>(min(static_cast<uint32_t>(kPiece), n - k * kPiece));
                pc.multi = np > 1;
                if (DUST_IB(p0 + k, a.np_max)) a.table[p0 + k] = pc;
            }
        }
    }
}

// Exclusive prefix sums of four per-thread values over the CTA's 1024 threads
// (in thread order); tot receives the four totals.  Every thread must call it.
__device__ void block_exclusive_scan4(const uint32_t (&x)[4], uint32_t (&pre)[4],
                                      uint32_t (&tot)[4], uint32_t* wsum /* [4][32] */) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t incl[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        incl[c] = x[c];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl[c], o);
            if (lane >= o) incl[c] += y;
        }
        if (lane == 31) wsum[c * 32 + warp] = incl[c];
    }
    __syncthreads();
    if (warp < 4) {
        const uint32_t w = wsum[warp * 32 + lane];
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += y;
        }
        wsum[warp * 32 + lane] = wi - w;  // exclusive prefix of the warp totals
        if (lane == 31) wsum[128 + warp] = wi;  // the CTA total
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        pre[c] = wsum[c * 32 + warp] + incl[c] - x[c];
        tot[c] = wsum[128 + c];
    }
    __syncthreads();  // wsum is free again
}

// Piece k of id v's n sorted tokens, which start at s0.
__device__ __forceinline__ Piece make_piece(uint32_t v, uint32_t s0, uint32_t n, uint32_t k) {
    Piece pc;
    pc.v = static_cast<int32_t>(v);
    pc.start = static_cast<int32_t>(s0 + k * kPiece);
    pc.len = static_cast<int32_t>(min(static_cast<uint32_t>(kPiece), n - k * kPiece));
    pc.multi = n > static_cast<uint32_t>(kPiece);
    return pc;
}

// The counting pass (V <= kCountV, nchunks <= kCountChunks, one CTA per chunk,
// cooperative launch with kCountSmem bytes of dynamic shared memory).
//   1. The chunk's sort keys (an id outside [0, V) becomes V, counted and
//      sorted last, then left out), its count per key (warp-aggregated
//      shared-memory atomics: exact in any order), and the chunk's (key,
//      token) pairs sorted stably by key in shared memory (two passes of
//      7-bit digits, ranks from per-warp digit counts as in the radix sort).
//      The counts go to chist[chunk][key].
//   2. After one grid barrier, thread i of every CTA owns keys 8i .. 8i + 7:
//      their totals over all chunks and over the chunks before this one, and
//      this chunk's counts, scanned over the keys give each key's first
//      sorted position seg, its first piece and its place among the ids no
//      token hits.  A token at place p of the chunk's sorted list with key v
//      lands at seg[v] + (tokens of v in earlier chunks) + (p - first place
//      of v in this chunk).  Every CTA scans all keys; CTA b writes the piece
//      table, the empty ids and poff of the keys owned by its threads
//      i = b, b + grid, ...
__global__ void __launch_bounds__(kChunk) embed_count_sort_kernel(const SortArgs a) {
    extern __shared__ uint32_t csm[];
    uint32_t* bins = csm;              // this chunk's counts per key, then the scatter bases
    uint32_t* tot_s = bins + kCountBins;           // tokens per key, all chunks
    uint32_t* pre_s = tot_s + kCountBins;          // ... in earlier chunks, then each key's seg
    uint32_t* poff_s = pre_s + kCountBins;         // first piece of each key (kCountBins + 8)
    uint32_t* lk0 = poff_s + kCountBins + 8;
    uint32_t* lk1 = lk0 + kChunk;
    int32_t* lv0 = reinterpret_cast<int32_t*>(lk1 + kChunk);
    int32_t* lv1 = lv0 + kChunk;
    uint32_t* wc = reinterpret_cast<uint32_t*>(lv1 + kChunk);  // [32 warps][128 digits]
    uint32_t* dt = wc + 32 * 128;                              // [128] digit starts
    uint32_t* wsum = dt + 128;                                 // [4][32] + [4]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x;
    const int V1 = a.V + 1;

    for (int v = tid; v < kCountBins; v += kChunk) bins[v] = 0;
    __syncthreads();
    const int t = c * kChunk + tid;
    uint32_t key = kPadKey;
    if (t < a.T && DUST_IB(t, a.T)) {
        int id = __ldg(a.ids + t);
        if (id < 0 || id >= a.V) {
            record_status(a.ctl, DUST_ERR_DEVICE_RANGE);
            id = a.V;
        }
        key = static_cast<uint32_t>(id);
    }
    {
        // this chunk's count per key, and every chunk's total in cnt (integer
        // atomics, one per distinct key of a warp: the same sums in any order)
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        if (key != kPadKey && (peers & lanemask_lt()) == 0 && DUST_IB(key, kCountBins)) {
            atomicAdd(&bins[key], static_cast<uint32_t>(__popc(peers)));
            if (DUST_IB(key, a.V + 1)) atomicAdd(a.cnt + key, static_cast<uint32_t>(__popc(peers)));
        }
    }
    lk0[tid] = key;
    lv0[tid] = t;
    for (int pass = 0; pass < 2; ++pass) {
        const uint32_t* ki = pass ? lk1 : lk0;
        const int32_t* vi = pass ? lv1 : lv0;
        uint32_t* ko = pass ? lk0 : lk1;
        int32_t* vo = pass ? lv0 : lv1;
        for (int k = tid; k < 32 * 128; k += kChunk) wc[k] = 0;
        __syncthreads();
        const uint32_t k = ki[tid];
        const int32_t val = vi[tid];
        const uint32_t dig = (k >> (7 * pass)) & 127u;
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, dig);
        const uint32_t lrank = __popc(peers & lanemask_lt());
        if (lrank == 0) wc[warp * 128 + dig] = __popc(peers);
        __syncthreads();
        if (tid < 128) {  // digit tid: prefix over the warps, then the digit's total
            uint32_t acc = 0;
            for (int w = 0; w < 32; ++w) {
                const uint32_t x = wc[w * 128 + tid];
                wc[w * 128 + tid] = acc;
                acc += x;
            }
            dt[tid] = acc;
        }
        __syncthreads();
        if (warp == 0) {  // exclusive prefix of the 128 digit totals, four per lane
            uint32_t x[4], sum = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                x[q] = dt[4 * lane + q];
                sum += x[q];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t run = incl - sum;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dt[4 * lane + q] = run;
                run += x[q];
            }
        }
        __syncthreads();
        const uint32_t pos = dt[dig] + wc[warp * 128 + dig] + lrank;
        if (DUST_IB(pos, kChunk)) {
            ko[pos] = k;
            vo[pos] = val;
        }
    }
    __syncthreads();  // lk0/lv0: the chunk sorted by key, ties by token
    // this chunk's counts into column c of chist (zeroed by the caller: only the
    // keys the chunk holds are written)
    const int64_t ch_words = static_cast<int64_t>(V1) * a.nchp;
    for (int v = tid; v < V1; v += kChunk) {
        const uint32_t n = bins[v];
        if (n != 0 && DUST_IB(static_cast<int64_t>(v) * a.nchp + c, ch_words))
            a.chist[static_cast<int64_t>(v) * a.nchp + c] = n;
    }
    if (!grid_barrier(a.ctl)) return;

    // For the keys this chunk holds, their counts in the earlier chunks: a
    // key's row of chist is nchp words, 16-byte aligned, so four chunks per
    // load; thread i takes keys i + 1024 k, which spreads the keys that every
    // chunk holds (the frequent ids) over the threads.
    for (int k = 0; k < kCountBins / kChunk; ++k) {
        const int v = tid + kChunk * k;
        uint32_t acc = 0;
        if (v < V1 && c > 0 && bins[v] != 0) {
            const int64_t r0 = static_cast<int64_t>(v) * a.nchp;
            if (a.nchp <= 16) {
                uint4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    q[u] = (4 * u < c && DUST_IB(r0 + 4 * u + 3, ch_words))
                               ? __ldcg(reinterpret_cast<const uint4*>(a.chist + r0 + 4 * u))
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int cc = 4 * u;
                    acc += (cc < c ? q[u].x : 0u) + (cc + 1 < c ? q[u].y : 0u) +
                           (cc + 2 < c ? q[u].z : 0u) + (cc + 3 < c ? q[u].w : 0u);
                }
            } else {
                for (int c4 = 0; c4 < c; c4 += 4) {
                    if (!DUST_IB(r0 + c4 + 3, ch_words)) break;
                    const uint4 q = __ldcg(reinterpret_cast<const uint4*>(a.chist + r0 + c4));
                    acc += q.x + (c4 + 1 < c ? q.y : 0u) + (c4 + 2 < c ? q.z : 0u) +
                           (c4 + 3 < c ? q.w : 0u);
                }
            }
        }
        pre_s[v] = acc;
    }
    __syncthreads();
    // Keys v0 .. v0 + 7 of this thread, in order, for the scans: totals (cnt),
    // this chunk's counts, the earlier chunks' counts.
    const int v0 = 8 * tid;
    uint32_t tot[8], pre[8], own[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int v = v0 + k;
        tot[k] = (v < V1 && DUST_IB(v, a.V + 1)) ? __ldcg(a.cnt + v) : 0u;
        own[k] = v < V1 ? bins[v] : 0u;
        pre[k] = pre_s[v];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tot_s[v0 + k] = tot[k];
    // per-thread sums: tokens, pieces, ids no token hits (v < V), this chunk's tokens
    uint32_t x4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int v = v0 + k;
        x4[0] += tot[k];
        if (v < a.V) {
            x4[1] += (tot[k] + kPiece - 1) / kPiece;
            x4[2] += tot[k] == 0 ? 1u : 0u;
        }
        x4[3] += own[k];
    }
    uint32_t p4[4], t4[4];
    block_exclusive_scan4(x4, p4, t4, wsum);  // (its barriers also order the reads of bins above)
    const bool writer = (tid % static_cast<int>(gridDim.x)) == c;
    uint32_t seg = p4[0], pof = p4[1], eof = p4[2], lst = p4[3];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int v = v0 + k;
        if (v >= V1) break;
        bins[v] = seg + pre[k] - lst;  // scatter base: position = base + place in the chunk
        pre_s[v] = seg;
        poff_s[v] = v < a.V ? pof : t4[1];
        if (writer && v < a.V) {
            if (DUST_IB(v, a.V + 1)) a.poff[v] = pof;
            if (tot[k] == 0 && DUST_IB(eof, a.V)) a.empty[eof] = v;
        }
        seg += tot[k];
        if (v < a.V) {
            pof += (tot[k] + kPiece - 1) / kPiece;
            eof += tot[k] == 0 ? 1u : 0u;
        }
        lst += own[k];
    }
    if (c == 0 && tid == 0) {
        a.poff[a.V] = t4[1];
        a.ctl[kNPieces] = t4[1];
        a.ctl[kNEmpty] = t4[2];
    }
    __syncthreads();
    // The piece table, pieces q = c, c + grid, ... of this CTA: q's key is the
    // last v < V with poff[v] <= q (binary search), k = q - poff[v] its place.
    const uint32_t npieces = t4[1];
    for (uint32_t q = static_cast<uint32_t>(c) + static_cast<uint32_t>(gridDim.x) * tid; q < npieces;
         q += static_cast<uint32_t>(gridDim.x) * kChunk) {
        int lo = 0, hi = a.V - 1;  // poff_s[lo] <= q < poff_s[hi + 1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (poff_s[mid] <= q) lo = mid;
            else hi = mid - 1;
        }
        if (DUST_IB(q, a.np_max))
            a.table[q] = make_piece(static_cast<uint32_t>(lo), pre_s[lo], tot_s[lo], q - poff_s[lo]);
    }
    const uint32_t kk = lk0[tid];
    if (kk != kPadKey && DUST_IB(kk, kCountBins)) {
        const uint32_t pos = bins[kk] + static_cast<uint32_t>(tid);
        if (DUST_IB(pos, a.T)) a.perm_dst[pos] = lv0[tid];
    }
}

struct RowArgs {
    const float* g;
    const int32_t* perm;
    const Piece* table;
    const uint32_t* poff;
    const int32_t* empty;
    const uint32_t* ctl;
    uint32_t* row_done;    // V x nslices counters of finished groups (zeroed by the caller)
    uint32_t* group_done;  // pieces x nslices counters of finished pieces, at a group's
                           // first piece (zeroed by the caller)
    int d, nslices;
    float* G_E;
    float* partial;  // npieces x d
    int T, V;        // extents the debug build checks indices against
    int64_t np_max;
};

// out[c] = sum_{q < n} rows[q * d + c], in order q = 0, 1, ..., for the warp's
// four columns of a slice; the loads of two rows are in flight together.
template <bool VEC>
__device__ __forceinline__ void add_rows_in_order(const float* rows, uint32_t n, int64_t d,
                                                  int c0, int w, float* out) {
    if (VEC) {
        float4 acc[kLaneF4];
#pragma unroll
        for (int k = 0; k < kLaneF4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t q = 0; q < n; q += 2) {
            float4 x[2][kLaneF4];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int k = 0; k < kLaneF4; ++k) {
                    const int c = c0 + 32 * k;
                    x[j][k] = (q + j < n && c < w)
                                  ? __ldcg(reinterpret_cast<const float4*>(rows + (q + j) * d) + c)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (q + j < n)
#pragma unroll
                    for (int k = 0; k < kLaneF4; ++k) {
                        acc[k].x += x[j][k].x; acc[k].y += x[j][k].y;
                        acc[k].z += x[j][k].z; acc[k].w += x[j][k].w;
                    }
        }
#pragma unroll
        for (int k = 0; k < kLaneF4; ++k) {
            const int c = c0 + 32 * k;
            if (c < w) reinterpret_cast<float4*>(out)[c] = acc[k];
        }
    } else {
        float acc[kLaneF] = {};
        for (uint32_t q = 0; q < n; q += 2) {
            float x[2][kLaneF];
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int k = 0; k < kLaneF; ++k) {
                    const int c = c0 + 32 * k;
                    x[j][k] = (q + j < n && c < w) ? __ldcg(rows + (q + j) * d + c) : 0.f;
                }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (q + j < n)
#pragma unroll
                    for (int k = 0; k < kLaneF; ++k) acc[k] += x[j][k];
        }
#pragma unroll
        for (int k = 0; k < kLaneF; ++k) {
            const int c = c0 + 32 * k;
            if (c < w) out[c] = acc[k];
        }
    }
}

// One warp per work unit: (piece, column slice) for every piece, then (empty
// id, slice).  Lane l takes columns l, l + 32, l + 64, l + 96 of the slice
// (float4 columns when VEC: d % 4 == 0 and 16-byte aligned rows).  The rows'
// token indices are read once per lane and passed round by shuffles.
template <bool VEC>
__global__ void __launch_bounds__(kRowThreads) embed_rows_kernel(const RowArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int npieces = static_cast<int>(__ldg(a.ctl + kNPieces));
    const int nempty = static_cast<int>(__ldg(a.ctl + kNEmpty));
    const int64_t nunits = static_cast<int64_t>(npieces + nempty) * a.nslices;
    const int w = VEC ? a.d >> 2 : a.d;  // columns of the element type
    const int per = VEC ? kSliceF4 : kSliceF;
    // A unit's piece and this lane's row index (one unit ahead: the next
    // unit's table entry and row indices are read while this one streams).
    auto fetch = [&](int64_t u, Piece& pc, int& myrow) {
        pc.v = -1;
        pc.len = 0;
        myrow = 0;
        if (u >= nunits) return;
        const int item = static_cast<int>(u / a.nslices);
        if (item >= npieces) {
            pc.v = DUST_IB(item - npieces, a.V) ? __ldg(a.empty + (item - npieces)) : 0;
            return;
        }
        if (!DUST_IB(item, a.np_max)) return;
        pc = a.table[item];
        myrow = (lane < pc.len && DUST_IB(pc.start + lane, a.T)) ? __ldg(a.perm + pc.start + lane)
                                                                 : 0;
        if (!DUST_IB(myrow, a.T)) myrow = 0;
    };
    Piece pc;
    int myrow;
    fetch(gwarp, pc, myrow);
    for (int64_t u = gwarp; u < nunits; u += nwarps) {
        Piece pn;
        int rown;
        fetch(u + nwarps, pn, rown);
        const int item = static_cast<int>(u / a.nslices);
        const int s = static_cast<int>(u - static_cast<int64_t>(item) * a.nslices);
        const int c0 = s * per + lane;
        if (item >= npieces) {  // an id no token hits: zeros
            const int64_t v = pc.v;
#pragma unroll
            for (int k = 0; k < (VEC ? kLaneF4 : kLaneF); ++k) {
                const int c = c0 + 32 * k;
                if (c < w && DUST_IB(v, a.V)) {
                    if (VEC)
                        reinterpret_cast<float4*>(a.G_E + v * a.d)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                    else
                        a.G_E[v * a.d + c] = 0.f;
                }
            }
            pc = pn;
            myrow = rown;
            continue;
        }
        if (!DUST_IB(pc.multi ? item : pc.v, pc.multi ? a.np_max : a.V)) {
            pc = pn;
            myrow = rown;
            continue;
        }
        float* dst = pc.multi ? a.partial + static_cast<int64_t>(item) * a.d
                              : a.G_E + static_cast<int64_t>(pc.v) * a.d;
        if (VEC) {
            float4 acc[kLaneF4];
#pragma unroll
            for (int k = 0; k < kLaneF4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
            for (int r = 0; r < pc.len; ++r) {
                const float4* src = reinterpret_cast<const float4*>(
                    a.g + static_cast<int64_t>(__shfl_sync(0xFFFFFFFFu, myrow, r)) * a.d);
#pragma unroll
                for (int k = 0; k < kLaneF4; ++k) {
                    const int c = c0 + 32 * k;
                    if (c < w) {
                        const float4 x = __ldg(src + c);
                        acc[k].x += x.x; acc[k].y += x.y; acc[k].z += x.z; acc[k].w += x.w;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kLaneF4; ++k) {
                const int c = c0 + 32 * k;
                if (c < w) reinterpret_cast<float4*>(dst)[c] = acc[k];
            }
        } else {
            float acc[kLaneF] = {};
#pragma unroll 4
            for (int r = 0; r < pc.len; ++r) {
                const float* src =
                    a.g + static_cast<int64_t>(__shfl_sync(0xFFFFFFFFu, myrow, r)) * a.d;
#pragma unroll
                for (int k = 0; k < kLaneF; ++k) {
                    const int c = c0 + 32 * k;
                    if (c < w) acc[k] += __ldg(src + c);
                }
            }
#pragma unroll
            for (int k = 0; k < kLaneF; ++k) {
                const int c = c0 + 32 * k;
                if (c < w) dst[c] = acc[k];
            }
        }
        if (pc.multi) {
            // Two-level tree: the warp that completes a group of kGroup pieces
            // adds them into the group's first partial; the warp that
            // completes the row's last group adds the group sums into the row.
            __threadfence();
            __syncwarp();
            const uint32_t p0 = a.poff[pc.v], np = a.poff[pc.v + 1] - p0;
            const uint32_t k = static_cast<uint32_t>(item) - p0;  // piece within the row
            const bool counters_ok =
                DUST_IB(static_cast<int64_t>(p0) + np - 1, a.np_max) &&
                DUST_IB(static_cast<int64_t>(pc.v) * a.nslices + s, static_cast<int64_t>(a.V) * a.nslices);
            if (!counters_ok) {
                pc = pn;
                myrow = rown;
                continue;
            }
            const uint32_t gfirst = p0 + (k / kGroup) * kGroup;    // the group's first piece
            const uint32_t gsize = min(static_cast<uint32_t>(kGroup), p0 + np - gfirst);
            uint32_t fin = 0;
            if (lane == 0)
                fin = atomicAdd(a.group_done + static_cast<int64_t>(gfirst) * a.nslices + s,
                                1u) == gsize - 1;
            if (__shfl_sync(0xFFFFFFFFu, fin, 0)) {
                __threadfence();
                float* gdst = a.partial + static_cast<int64_t>(gfirst) * a.d;
                add_rows_in_order<VEC>(gdst, gsize, a.d, c0, w, gdst);
                __threadfence();
                __syncwarp();
                const uint32_t ng = (np + kGroup - 1) / kGroup;
                fin = 0;
                if (lane == 0)
                    fin = atomicAdd(a.row_done + static_cast<int64_t>(pc.v) * a.nslices + s, 1u) ==
                          ng - 1;
                if (__shfl_sync(0xFFFFFFFFu, fin, 0)) {
                    __threadfence();
                    add_rows_in_order<VEC>(a.partial + static_cast<int64_t>(p0) * a.d, ng,
                                           static_cast<int64_t>(kGroup) * a.d, c0, w,
                                           a.G_E + static_cast<int64_t>(pc.v) * a.d);
                }
            }
        }
        pc = pn;
        myrow = rown;
    }
}

struct EmbedPlan {
    int nchunks, passes, nslices;
    int nchp;           // counting pass: chunk counts per key, padded to 4 words
    bool counting;      // the counting pass (one grid barrier) instead of the radix sort
    int64_t np_max;
    size_t zero_bytes;  // [ctl | digit counts | id counts | chunk counts | the rows kernel's
                        // counters]: cleared before the sort
    size_t off_hist, off_cnt, off_eoff, off_done, off_gdone, off_k0, off_v0, off_k1, off_v1, off_offs,
        off_seg, off_poff, off_table, off_empty, off_part, off_chist, bytes;
};

EmbedPlan embed_plan(int64_t T, int64_t d, int64_t V) {
    EmbedPlan P{};
    P.nchunks = static_cast<int>(ceil_div(T > 0 ? T : 1, kChunk));
    int bits = 1;
    while ((1LL << bits) <= V) ++bits;  // keys are in [0, V]
    P.passes = (bits + 7) / 8;
    // column slices per row: ceil(d/4 / 128) float4 or ceil(d / 128) float
    // slices; the counters are sized for the larger count
    P.nslices = static_cast<int>(ceil_div(d, kSliceF));
    P.np_max = ceil_div(T, kPiece) + (T < V ? T : V) + 1;
    const size_t Tn = static_cast<size_t>(T > 0 ? T : 1);
    const size_t Vn = static_cast<size_t>(V);
    const size_t hist_words = static_cast<size_t>(256) * P.nchunks;
    WsLayout w;
    w.take(kCtlBytes);
    P.off_hist = w.take(static_cast<size_t>(P.passes) * hist_words * 4);
    P.off_cnt = w.take((Vn + 1) * 4);  // (the counting pass counts the invalid key V too)
    P.counting = V <= kCountV && P.nchunks <= kCountChunks;
    P.nchp = static_cast<int>(round_up(P.nchunks, 4));
    P.off_chist = w.take(P.counting ? (Vn + 1) * static_cast<size_t>(P.nchp) * 4 : 0);
    P.off_done = w.take(Vn * static_cast<size_t>(P.nslices) * 4);
    P.off_gdone = w.take(static_cast<size_t>(P.np_max) * static_cast<size_t>(P.nslices) * 4);
    P.zero_bytes = w.used;
    P.off_eoff = w.take(Vn * 4);
    P.off_k0 = w.take(Tn * 4);
    P.off_v0 = w.take(Tn * 4);
    P.off_k1 = w.take(Tn * 4);
    P.off_v1 = w.take(Tn * 4);
    P.off_offs = w.take(static_cast<size_t>(P.passes) * hist_words * 4);
    P.off_seg = w.take(Vn * 4);
    P.off_poff = w.take((Vn + 1) * 4);
    P.off_table = w.take(static_cast<size_t>(P.np_max) * sizeof(Piece));
    P.off_empty = w.take(Vn * 4);
    P.off_part = w.take(static_cast<size_t>(P.np_max) * static_cast<size_t>(d) * 4);
    P.bytes = w.used;
    return P;
}

// CTAs of a sort kernel that fit on the current device at once (the grid of
// its cooperative launch is at most this), looked up once per device: the
// radix sort (counting = false) or the counting pass with its shared memory.
int sort_grid_limit(bool counting) {
    static std::atomic<int> limits[2][64];
    std::atomic<int>* limit = limits[counting ? 1 : 0];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 0 || dev >= 64) return 0;
    int cached = limit[dev].load(std::memory_order_acquire);
    if (cached > 0) return cached;
    int per_sm = 0, sms = 0;
    const cudaError_t occ =
        counting ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                       &per_sm, embed_count_sort_kernel, kChunk, static_cast<size_t>(kCountSmem))
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, embed_sort_kernel,
                                                                 kChunk, 0);
    if (occ != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cached = per_sm * sms;
    limit[dev].store(cached, std::memory_order_release);
    return cached;
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
    uint32_t* ctl = static_cast<uint32_t*>(ws);
    if (T == 0) {
        DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlBytes, s));
        DUST_CUDA_TRY(cudaMemsetAsync(G_E, 0, static_cast<size_t>(V * d) * 4, s));
        return DUST_OK;
    }
    if (P.counting) {
        static std::atomic<uint64_t> smem_set{0};
        DUST_CUDA_TRY(set_smem_once(embed_count_sort_kernel, static_cast<int>(kCountSmem), smem_set));
    }
    const int limit = sort_grid_limit(P.counting);
    if (limit < 1) return DUST_ERR_CUDA;
    const bool vec = (d % 4 == 0) && aligned(g_hat, 16) && aligned(G_E, 16);

    SortArgs sa{};
    sa.ids = ids;
    sa.T = static_cast<int>(T);
    sa.V = static_cast<int>(V);
    sa.nchunks = P.nchunks;
    sa.passes = P.passes;
    sa.nslices = P.nslices;
    sa.keys[0] = reinterpret_cast<uint32_t*>(w + P.off_k0);
    sa.keys[1] = reinterpret_cast<uint32_t*>(w + P.off_k1);
    sa.vals[0] = reinterpret_cast<int32_t*>(w + P.off_v0);
    sa.vals[1] = reinterpret_cast<int32_t*>(w + P.off_v1);
    sa.perm_out = perm_out;
    sa.hist = reinterpret_cast<uint32_t*>(w + P.off_hist);
    sa.offs = reinterpret_cast<uint32_t*>(w + P.off_offs);
    sa.cnt = reinterpret_cast<uint32_t*>(w + P.off_cnt);
    sa.seg = reinterpret_cast<uint32_t*>(w + P.off_seg);
    sa.poff = reinterpret_cast<uint32_t*>(w + P.off_poff);
    sa.eoff = reinterpret_cast<uint32_t*>(w + P.off_eoff);
    sa.table = reinterpret_cast<Piece*>(w + P.off_table);
    sa.empty = reinterpret_cast<int32_t*>(w + P.off_empty);
    sa.row_done = reinterpret_cast<uint32_t*>(w + P.off_done);
    sa.group_done = reinterpret_cast<uint32_t*>(w + P.off_gdone);
    sa.np_max = P.np_max;
    sa.ctl = ctl;
    sa.chist = reinterpret_cast<uint32_t*>(w + P.off_chist);
    sa.nchp = P.nchp;
    // the last pass's values: perm_out, or the ping-pong buffer it lands in
    sa.perm_dst = perm_out ? perm_out : sa.vals[0];
    const int32_t* perm = P.counting ? sa.perm_dst : perm_out ? perm_out : sa.vals[P.passes & 1];
    if (P.counting && P.nchunks > limit) return DUST_ERR_CUDA;

    timer_begin(s);  // the benchmark hook times the whole call
    // status and barrier words, the later passes' digit counts, the id counts
    DUST_CUDA_TRY(cudaMemsetAsync(ws, 0, P.zero_bytes, s));
    if (P.counting) {
        void* args[] = {&sa};
        DUST_CUDA_TRY(cudaLaunchCooperativeKernel(
            reinterpret_cast<const void*>(embed_count_sort_kernel), dim3(P.nchunks), dim3(kChunk),
            args, kCountSmem, s));
    } else {
        const unsigned grid = static_cast<unsigned>(std::min(P.nchunks, limit));
        void* args[] = {&sa};
        DUST_CUDA_TRY(cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(embed_sort_kernel),
                                                  dim3(grid), dim3(kChunk), args, 0, s));
    }
    RowArgs ra{g_hat, perm, reinterpret_cast<const Piece*>(w + P.off_table),
               reinterpret_cast<const uint32_t*>(w + P.off_poff),
               reinterpret_cast<const int32_t*>(w + P.off_empty), ctl,
               reinterpret_cast<uint32_t*>(w + P.off_done),
               reinterpret_cast<uint32_t*>(w + P.off_gdone), static_cast<int>(d),
               static_cast<int>(vec ? ceil_div(d / 4, kSliceF4) : ceil_div(d, kSliceF)), G_E,
               reinterpret_cast<float*>(w + P.off_part), static_cast<int>(T), static_cast<int>(V),
               P.np_max};
    const unsigned rgrid = 148 * 8;
    if (vec)
        embed_rows_kernel<true><<<rgrid, kRowThreads, 0, s>>>(ra);
    else
        embed_rows_kernel<false><<<rgrid, kRowThreads, 0, s>>>(ra);
    timer_end(s);
    return launch_status();
}

namespace dust {
DUST_DEBUG_READER(3)
}  // namespace dust
