/*
 * dust.h -- C ABI of the B300 (sm_103a) engine for the Dust virtual-population
 * gradient estimator ("Dust: Pretraining Transformers Without
 * Backpropagation", Q Labs).
 *
 * The method (Dust translation, hn.213312.xyz, §2.2 信用分配): a linear layer
 * y_t = W x_t has its output perturbed per token, y_t + sigma a_t with
 * a_t ~ N(0, I).  For each of K draws the per-token loss is re-evaluated from
 * cached clean activations; the centred loss decrease c_s of token s gives the
 * reward r_t = sum_{s>=t} gamma^(s-t) c_s (gamma = 0: own token only); the
 * error estimate is g_t = -(1/(K sigma)) sum_i r_t^(i) a_t^(i) and the weight
 * gradient is G_W = sum_t g_t x_t^T.  For an embedding (one-hot input) the
 * outer product is a scatter-add of g_t into row id_t.  The LM head is
 * perturbed directly on its cached logits and only the cross-entropy is
 * recomputed (same page, §2.3 干扰与调优; laoyaoba.com article, section
 * 机制拆解).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer named as device memory must point to memory of the current
 *    CUDA device; host pointers are named as such.  Arrays are row-major and
 *    contiguous.  The caller owns every buffer; the library never allocates,
 *    frees or synchronises (apart from dust_workspace_status, which reads a
 *    word back on purpose).  All work is enqueued on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream).
 *  - Outputs are overwritten, never accumulated into.  Inputs are not
 *    modified.
 *  - Arguments are checked on the host before any launch; a bad argument
 *    returns an error status and enqueues nothing.  Values that live on the
 *    device (target ids, embedding ids) are checked by the kernels: an id out
 *    of range is skipped and recorded in the workspace status word, which
 *    dust_workspace_status reads back.  No kernel traps or asserts.
 *  - Every wait inside a kernel is bounded; a wait that runs out records
 *    DUST_ERR_TIMEOUT in the workspace status word and the kernel returns.
 *  - Results are deterministic: the same inputs and the same dust_noise give
 *    bitwise-identical outputs (no floating-point atomics).
 *  - The workspace (`ws`, `ws_bytes`) is device memory of at least the size
 *    returned by the matching *_workspace query, 256-byte aligned.  Calls that
 *    share one workspace must be ordered on the GPU (same stream).
 */
#ifndef DUST_H
#define DUST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DUST_OK = 0,
    DUST_ERR_INVALID_ARG = 1,  /* null pointer, bad size, sigma <= 0, ... */
    DUST_ERR_UNSUPPORTED = 2,  /* a size beyond what the kernels handle   */
    DUST_ERR_WORKSPACE = 3,    /* workspace null, too small or unaligned  */
    DUST_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed       */
    DUST_ERR_TIMEOUT = 5,      /* a bounded in-kernel wait ran out        */
    DUST_ERR_DEVICE_RANGE = 6  /* a device-side id was out of range       */
} dust_status;

typedef enum { DUST_F32 = 0, DUST_BF16 = 1 } dust_dtype;

/*
 * Noise and credit parameters of one estimator call.
 *
 * The noise a_{i,t}[c] of draw i, token t, output channel c is regenerated
 * from a counter, never stored: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11) of the counter
 * (c / 4, token0 + t, draw0 + i, layer) under the key (seed low word, seed
 * high word); each 32-bit word w becomes u = ((w >> 9) + 0.5) * 2^-23 and the
 * pairs (word 0, word 1), (word 2, word 3) become two normals each by
 * Box-Muller: rho = sqrt(-2 ln u_even), theta = 2 pi u_odd, channel 4j+2p gets
 * rho cos theta and 4j+2p+1 gets rho sin theta.  The pages say only that the
 * noise is Gaussian and independent per token and per layer; the generator and
 * counter layout are this library's convention.
 */
typedef struct {
    uint64_t seed;
    uint32_t layer;      /* layer id, the fourth counter word                 */
    uint32_t draw0;      /* draws are draw0 .. draw0 + num_draws - 1          */
    uint32_t num_draws;  /* K >= 2 (centring needs two draws)                 */
    uint32_t token0;     /* global index of the call's first token            */
    float sigma;         /* noise scale, > 0                                  */
    float gamma;         /* reward discount in [0, 1]; ignored by the head    */
} dust_noise;

const char* dust_status_string(dust_status s);

/* Version of this ABI (major * 100 + minor). */
int dust_abi_version(void);

/*
 * Reads the workspace status word left by the last call that used `ws`
 * (waits for `stream` first) into *status_out and clears it.  DUST_OK means no
 * kernel recorded a device-side error.
 */
dust_status dust_workspace_status(void* ws, void* stream, dust_status* status_out);

/* ------------------------------------------------------------------------ */
/* LM head (configs with gamma = 0)                                          */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for dust_head_estimate with these sizes. */
size_t dust_head_workspace(int64_t T, int64_t V, int64_t d, uint32_t K);

/*
 * LM-head estimator, perturbed directly on the cached logits (Dust
 * translation §2.3; laoyaoba.com section 机制拆解).
 *
 *   logits  device, T x V fp32: the cached clean logits z_t.
 *   targets device, T int32: next-token ids in [0, V).
 *   x       device, T x d, dtype x_dtype: the head's input activations.
 *   g_hat   device, T x V fp32 output, or NULL: the error estimate
 *           g_t[v] = -(1/(K sigma)) sum_i c_{i,t} a_{i,t}[v], with
 *           c_{i,t} = -(dl_{i,t} - mean_j dl_{j,t}) and
 *           dl_{i,t} = CE(z_t + sigma a_{i,t}) - CE(z_t) (natural log, full
 *           vocabulary).  gamma is not used: the head has no path from one
 *           token's logits to another token's loss, so r = c.
 *   G_W     device, V x d fp32 output: sum_t g_t x_t^T, computed from g
 *           rounded to bf16 and x rounded to bf16, accumulated in fp32.
 *
 * Limits: 1 <= V <= 8192, 1 <= d, 1 <= T <= 2^30, 2 <= K <= 2^30,
 *         token0 + T <= 2^32, draw0 + K <= 2^32.
 */
dust_status dust_head_estimate(const float* logits, const int32_t* targets, const void* x,
                               dust_dtype x_dtype, int64_t T, int64_t V, int64_t d,
                               dust_noise nz, float* g_hat, float* G_W, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * How the loss changes of the K draws become centred decreases c.  The pages
 * centre by the mean over draws (Dust translation §2.2); the two others are
 * the common variance-reduction baselines, which the pages do not describe:
 *   DUST_BASELINE_MEAN           c_i = -(dl_i - mean_j dl_j)     (the pages)
 *   DUST_BASELINE_LEAVE_ONE_OUT  c_i = -(dl_i - mean_{j != i} dl_j)
 *                                (= K/(K-1) times the mean-centred estimate)
 *   DUST_BASELINE_ANTITHETIC     each draw's noise is evaluated as +a and -a,
 *                                c_i = -(dl_i(+a) - dl_i(-a)) / 2: 2K
 *                                perturbed evaluations from K noise draws.
 */
typedef enum {
    DUST_BASELINE_MEAN = 0,
    DUST_BASELINE_LEAVE_ONE_OUT = 1,
    DUST_BASELINE_ANTITHETIC = 2
} dust_baseline;

/*
 * dust_head_estimate with a choice of baseline; everything else (arguments,
 * limits, workspace from dust_head_workspace with the same K, errors) is as
 * there.  With DUST_BASELINE_ANTITHETIC, nz.num_draws counts noise draws
 * (pairs); draw i uses the noise of counter draw0 + i for both signs.  An
 * unknown baseline value is INVALID_ARG.
 */
dust_status dust_head_estimate_baseline(const float* logits, const int32_t* targets,
                                        const void* x, dust_dtype x_dtype, int64_t T, int64_t V,
                                        int64_t d, dust_noise nz, dust_baseline baseline,
                                        float* g_hat, float* G_W, void* ws, size_t ws_bytes,
                                        void* stream);

/* Workspace bytes for dust_head_estimate_chunked (0 if the shape is invalid). */
size_t dust_head_chunked_workspace(int64_t T, int64_t V, int64_t d, uint32_t K, int64_t chunk);

/*
 * The head with one vocabulary chunk perturbed per draw (the pages' head
 * recomputes the cross-entropy of only a small chunk of the vocabulary per
 * round: laoyaoba.com, section 机制拆解).  Chunks of width `chunk` tile the
 * vocabulary; draw j (counter draw0 + j) perturbs chunk j mod (V/chunk) only:
 *   dl = log(1 + sum_{v in chunk} p_v (e^{sigma a_v} - 1)) - sigma a_y [y in chunk],
 * p the softmax of the full row.  Each chunk's draws are centred by their own
 * mean, and each column of g averages over its chunk's K chunk / V draws:
 *   g_t[v] = -(1/(K_c sigma)) sum_{draws i of v's chunk} c_{i,t} a_{i,t}[v].
 * With chunk = V it is dust_head_estimate.  Arguments and outputs as there;
 * chunk must be a multiple of 4 dividing V (<= 8192), and V/chunk must divide
 * K with at least 2 draws per chunk (INVALID_ARG otherwise).
 */
dust_status dust_head_estimate_chunked(const float* logits, const int32_t* targets,
                                       const void* x, dust_dtype x_dtype, int64_t T, int64_t V,
                                       int64_t d, dust_noise nz, int64_t chunk, float* g_hat,
                                       float* G_W, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Interior linear layer with causal credit                                  */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for dust_linear_estimate with these sizes. */
size_t dust_linear_workspace(int64_t T, int64_t d_in, int64_t C, int64_t d_model, int64_t V,
                             uint32_t K);

/*
 * Interior linear layer y1 = W1 x whose output is perturbed; only the part
 * after it is re-run, from cached clean activations (laoyaoba.com section
 * 机制拆解; Dust translation §2.3).  The downstream is fixed:
 * GELU (exact erf) -> W2 -> causal per-sequence EMA
 * e_t = ema_decay e_{t-1} + (1 - ema_decay) u_t (e = 0 before each sequence
 * start) -> W_head -> cross-entropy.  Because W2, the EMA and W_head are
 * linear, a draw's perturbed logits are z_clean + W_head EMA(W2 dh) with
 * dh = GELU(y1 + sigma a) - GELU(y1).
 *
 *   x       device, T x d_in bf16: the layer input.
 *   y1      device, T x C fp32: cached clean output of the layer.
 *   W2      device, d_model x C bf16.
 *   W_head  device, V x d_model bf16.
 *   z_clean device, T x V fp32: cached clean logits.
 *   targets device, T int32 in [0, V).
 *   seq_len tokens per sequence; T is a multiple of it.  Credit and the EMA
 *           never cross a sequence boundary.
 *   g_hat   device, T x C fp32 output, or NULL.
 *   G_W1    device, C x d_in fp32 output: sum_t g_t x_t^T (g rounded to bf16).
 *
 * Reward: r_{i,t} = sum_{s >= t, same sequence} gamma^(s-t) c_{i,s}.
 */
dust_status dust_linear_estimate(const void* x, const float* y1, const void* W2,
                                 float ema_decay, const void* W_head, const float* z_clean,
                                 const int32_t* targets, int64_t T, int64_t seq_len,
                                 int64_t d_in, int64_t C, int64_t d_model, int64_t V,
                                 dust_noise nz, float* g_hat, float* G_W1, void* ws,
                                 size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Embedding: one-hot input, so the outer product is a scatter-add            */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for dust_embed_scatter with these sizes. */
size_t dust_embed_workspace(int64_t T, int64_t d, int64_t V);

/*
 * Embedding gradient (Dust translation §2.2, last sentences): with one-hot
 * inputs, sum_t g_t onehot(id_t)^T is the scatter-add G_E[id_t] += g_t.
 *
 *   g_hat   device, T x d fp32.
 *   ids     device, T int32 in [0, V).
 *   G_E     device, V x d fp32 output, fully overwritten; rows no token hits
 *           are zero.  Row v is the sum of the g_t with id_t = v, in a fixed
 *           order that depends only on the ids (bitwise reproducible).
 *   perm_out device, T int32 output, or NULL: the tokens ordered by
 *           (id, t) ascending -- a stable sort of the ids.
 *
 * Limits: 1 <= V <= 2^24, 1 <= d, 0 <= T < 2^31.
 */
dust_status dust_embed_scatter(const float* g_hat, const int32_t* ids, int64_t T, int64_t d,
                               int64_t V, float* G_E, int32_t* perm_out, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * dust_embed_scatter without a caller-provided workspace, for callers that
 * cannot allocate device memory where they need the embedding gradient (code
 * running under a host framework that owns every device allocation, or in a
 * hook that runs while the caller's memory pool is locked).  The pages have no
 * counterpart: this is an interface convenience, not a step of the method.
 *
 * Same arguments, results and limits as dust_embed_scatter, except that the
 * scratch is a fixed 32 MiB array inside the library (held on every GPU that
 * loads the library until the process exits).  Sizes whose workspace
 * (dust_embed_workspace) exceeds 32 MiB return DUST_ERR_UNSUPPORTED.  The
 * first call on a device looks up the array's device address (and so does the
 * first call after the device's context was reset and recreated, where the
 * array may have moved), so make it before any stream capture.  All calls
 * share the array: calls that overlap on
 * the GPU race, so order them (one stream).  Device-side id errors go to the
 * shared array's status word and cannot be read back through this call.
 * Allocates nothing (no cudaMalloc, no allocating library routine).
 */
dust_status dust_embed_scatter_static(const float* g_hat, const int32_t* ids, int64_t T,
                                      int64_t d, int64_t V, float* G_E, int32_t* perm_out,
                                      void* stream);

/* ------------------------------------------------------------------------ */
/* Test hooks                                                               */
/* ------------------------------------------------------------------------ */

/*
 * The noise regenerator alone, for tokens token0 .. token0 + ntok - 1 and
 * channels 0 .. nchan - 1 of one draw (counter layout as in dust_noise).
 *   words   device, ntok x nchan uint32 output, or NULL: word (c % 4) of the
 *           Philox block of channel c.
 *   normals device, ntok x nchan fp32 output, or NULL: the normal of channel c.
 */
dust_status dust_philox_fill(uint64_t seed, uint32_t layer, uint32_t draw, int64_t token0,
                             int64_t ntok, int64_t nchan, uint32_t* words, float* normals,
                             void* stream);

/*
 * The Box-Muller step that the throughput-bound kernels use (the head's draw
 * kernels), on caller-chosen words: for pair k, words[2k] (even) and
 * words[2k+1] (odd) become normals[2k] = rho cos theta and
 * normals[2k+1] = rho sin theta with rho = sqrt(-2 ln u(w_even)),
 * theta = 2 pi u(w_odd) and u(w) = ((w >> 9) + 0.5) 2^-23, computed with the
 * hardware log2, square root and sin/cos (the map of dust_noise, to within
 * the error those approximations leave).  Pairs are taken two at a time by
 * the packed-pair form the estimator kernels run and the last pair of an odd
 * count by the scalar form; both give the same bits.  words and normals are
 * device arrays of 2 npairs elements, 8-byte aligned.  INVALID_ARG for a
 * negative count or a NULL or misaligned array.
 */
dust_status dust_box_muller_fast(const uint32_t* words, int64_t npairs, float* normals,
                                 void* stream);

/*
 * The debug build.  libdust_debug.so is the same library compiled with every
 * computed global-memory index of the CUDA-core code checked against the
 * extent of the buffer it addresses: an index out of range skips its access
 * (nothing outside the caller's buffers is read or written) and records the
 * first such fault per source file.  dust_debug_build returns 1 for that
 * library, 0 for libdust.so.  dust_debug_fault synchronises the device,
 * returns the first recorded fault as (file id << 32) | source line, or 0 if
 * no checked access failed since the last call (always 0 in libdust.so), and
 * clears the record.
 */
int dust_debug_build(void);
uint64_t dust_debug_fault(void);

/*
 * The debug build's index check by itself: one device thread checks index i
 * against extent n and writes 1 (in range) or 0 to the device int
 * `in_bounds`, addressing nothing with i.  In libdust_debug.so an i outside
 * [0, n) also records a fault that dust_debug_fault then returns (file id
 * 10); libdust.so always writes 1.  Asynchronous on `stream`.  Returns
 * DUST_ERR_INVALID_ARG for a null or unaligned `in_bounds`.
 */
dust_status dust_debug_check_index(int64_t i, int64_t n, int* in_bounds, void* stream);

/*
 * The outer-product GEMM alone: G[m][n] = sum_k A(m, k) B(n, k) in fp32 from
 * bf16 operands on the tensor cores.  A is stored M-major (k rows of M
 * elements, row stride lda elements) when a_mn != 0, else K-major (M rows of
 * K elements); likewise B with b_mn.  All device; G is M x N fp32 (row stride
 * ldg).  Strides are multiples of 8 elements; the bases are 16-byte aligned.
 * `ws` holds the status word (>= 256 bytes).
 */
dust_status dust_gemm_bf16(const void* A, int a_mn, int64_t lda, const void* B, int b_mn,
                           int64_t ldb, int64_t M, int64_t N, int64_t K, float* G, int64_t ldg,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Inside attention: the values, scored by the attention-output error        */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for dust_attn_value_estimate with these sizes (0 if they
 * are invalid). */
size_t dust_attn_value_workspace(int64_t T, int64_t seq_len, int64_t H, int64_t dv,
                                 int64_t d_in, uint32_t K);

/*
 * Estimator for the value projection v = W_v x of a causal attention layer,
 * perturbed per token inside the attention and scored by the attention-output
 * error (Dust translation §2.3: perturbations inside attention are scored by
 * the error of the attention output, with a decay gamma close to 1 for later
 * tokens).  With the cached clean probabilities P, perturbing every value by
 * sigma a_t changes head h's output of token s by
 *   dO_s = sigma sum_{t <= s} P_{s,t} a_t[h]   (exactly, values enter linearly);
 * the loss change of token s is read to first order as dl_s = <E_s, dO_s> over
 * all heads, and then c = -(dl - mean over draws),
 * r_t = sum_{s >= t, same sequence} gamma^(s-t) c_s,
 * g_t = -(1/(K sigma)) sum_i r a, G_W = sum_t g_t x_t^T.
 *
 *   P    device fp32, (T/seq_len) x H x seq_len x seq_len: row s = query,
 *        column t = key; entries with t > s are ignored (treated as 0).
 *   E    device fp32, T x (H dv): the error estimate of the attention output
 *        (head h in columns h dv .. h dv + dv - 1).
 *   x    device, T x d_in, dtype x_dtype: the input of W_v.
 *   g_hat device fp32 T x (H dv) output or NULL; G_W device fp32 (H dv) x d_in
 *        output (g and x rounded to bf16, fp32 accumulation).
 *   nz   noise of channel c = h dv + j of token t, draw i: the Philox counter
 *        (c/4, token0 + t, draw0 + i, layer) as for the other estimators.
 * Limits: dv = 64, seq_len a multiple of 128 (<= 8192), T a multiple of
 * seq_len, 1 <= H <= 64, K >= 2.  Workspace from dust_attn_value_workspace
 * (it holds P as split bf16, 2 x 2 bytes per entry of P).
 */
dust_status dust_attn_value_estimate(const float* P, const float* E, const void* x,
                                     dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t H,
                                     int64_t dv, int64_t d_in, dust_noise nz, float* g_hat,
                                     float* G_W, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for dust_attn_gate_estimate with these sizes (0 if invalid). */
size_t dust_attn_gate_workspace(int64_t T, int64_t seq_len, int64_t C, int64_t d_in, uint32_t K);

/*
 * Estimator for the gate projection z = W_g x of a gated attention output
 * o~ = sig(z) * o (per channel, sig the logistic function), perturbed per
 * token and scored like the values by the error E of the gated output
 * (Dust translation §2.3):
 *   d(o~)_s = (sig(z_s + sigma a_s) - sig(z_s)) * o_s,   dl_s = <E_s, d(o~)_s>,
 * then the same centring, gamma-scan, g and G_W = g^T x as the values.
 *   z, o, E  device fp32, T x C (16-byte aligned): gate pre-activations, the
 *            attention output before the gate, the error of the gated output.
 *   x        device, T x d_in (x_dtype): the input of W_g.
 *   g_hat    T x C fp32 or NULL; G_W C x d_in fp32.
 * Limits: C a multiple of 8, T a multiple of seq_len, K >= 2.
 */
dust_status dust_attn_gate_estimate(const float* z, const float* o, const float* E,
                                    const void* x, dust_dtype x_dtype, int64_t T, int64_t seq_len,
                                    int64_t C, int64_t d_in, dust_noise nz, float* g_hat,
                                    float* G_W, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for dust_attn_qk_estimate with these sizes (0 if invalid). */
size_t dust_attn_qk_workspace(int64_t T, int64_t seq_len, int64_t H, int64_t dv, int64_t d_in,
                              uint32_t K);

/*
 * Estimator for the query projection (which = 0) or the key projection
 * (which = 1) of a causal softmax attention layer, perturbed per token inside
 * the attention and scored like the values by the attention-output error
 * (Dust translation §2.3).  Perturbing every query by sigma a_s (or every key
 * by sigma a_t) moves the scores by ds_{s,t} = sigma <a_s, k_t> / sqrt(dv)
 * (or sigma <q_s, a_t> / sqrt(dv)); with the cached clean probabilities P and
 * output O the perturbed output of token s is, exactly,
 *   dO_s = (sum_{t<=s} w_{s,t} v_t - W_s o_s) / (1 + W_s),
 *   w_{s,t} = P_{s,t} (exp(ds_{s,t}) - 1),   W_s = sum_{t<=s} w_{s,t},
 * since the perturbed softmax row is P e^{ds} / sum P e^{ds}.  Then
 * dl_s = <E_s, dO_s> over all heads, and the same centring, gamma-scan, g and
 * G_W = g^T x as the values.
 *
 *   which  0 queries, 1 keys.
 *   Q, Kk, V, O, E  device fp32, T x (H dv), 16-byte aligned: the clean
 *          queries, keys and values, the clean attention output (head h in
 *          columns h dv .. h dv + dv - 1) and its error estimate.
 *   P      device fp32, (T/seq_len) x H x seq_len x seq_len, the clean
 *          probabilities of the same forward (row s = query, column t = key;
 *          entries with t > s are not read).  P and O must come from Q, Kk and
 *          V (rows of P summing to 1, O = P V): the formula above uses both.
 *   x      device, T x d_in (x_dtype): the input of W_q (or W_k).
 *   g_hat  T x (H dv) fp32 or NULL: the estimate for the queries (keys).
 *   G_W    (H dv) x d_in fp32 (g and x rounded to bf16, fp32 accumulation).
 *   nz     noise of channel c of token t, draw i: the Philox counter
 *          (c/4, token0 + t, draw0 + i, layer), as for the other estimators.
 * Limits: dv = 64, seq_len a multiple of 128 (<= 8192), T a multiple of
 * seq_len, 1 <= H <= 64, T/128 <= 65535, (T/seq_len) H <= 65535,
 * 2 <= K <= 65535.  Both products (the score shifts and the reweighted
 * values) run on the tensor cores as split-bf16 (hi/lo) operands with fp32
 * accumulation, per 128-query tile and 64-key slice, heads summed in order.
 * The workspace (from dust_attn_qk_workspace) holds the loss changes, the
 * credits, the bf16 copies for the outer product, K and V^T split into bf16
 * hi/lo, and for the keys the split noise of up to 16 draws at a time.
 */
dust_status dust_attn_qk_estimate(int which, const float* Q, const float* Kk, const float* V,
                                  const float* O, const float* P, const float* E, const void* x,
                                  dust_dtype x_dtype, int64_t T, int64_t seq_len, int64_t H,
                                  int64_t dv, int64_t d_in, dust_noise nz, float* g_hat,
                                  float* G_W, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Weight-space ES for the residual-mixing scalars                           */
/* ------------------------------------------------------------------------ */

/*
 * The pages estimate every weight by perturbing activations except the 2L
 * residual-mixing scalars (Dust translation §2.1); read plainly, those stay
 * with weight-space ES.  The library supplies the population side, with the
 * noise of the same counter scheme (parameter j as channel j of "token"
 * nz.token0, draw nz.draw0 + i):
 *   dust_es_perturb:  theta_out[i][j] = theta[j] + sigma eps_i[j]   (K x n)
 *   dust_es_estimate: g[j] = (1/(K sigma)) sum_i (L_i - mean L) eps_i[j],
 * an estimate of +dL/dtheta from the caller's K losses L (device, K fp32).
 * theta, theta_out, losses and g are device fp32 arrays; 1 <= n <= 2^26,
 * 2 <= K <= 2^20, sigma > 0; INVALID_ARG otherwise.  Asynchronous on stream.
 */
dust_status dust_es_perturb(const float* theta, int64_t n, dust_noise nz, float* theta_out,
                            void* stream);
dust_status dust_es_estimate(const float* losses, int64_t n, dust_noise nz, float* g,
                             void* stream);

/* ------------------------------------------------------------------------ */
/* Using the estimate: optimiser step and the backprop reference             */
/* ------------------------------------------------------------------------ */

/*
 * One step of SGD with momentum on n fp32 parameters, with the estimated
 * gradient G (the pages train with SGD and momentum: Dust translation,
 * experiment set-up; the form is the textbook heavy-ball one):
 *   b <- momentum b + (G + weight_decay W),   W <- W - lr b.
 * W and momentum_buf (device, n fp32, caller-owned, updated in place; the
 * buffer starts at zero) and G (device, n fp32, read) must not overlap.
 * W_bf16 (device, n bf16, or NULL) receives the updated W rounded to bf16,
 * the operand of the next forward's tensor-core GEMM.  n = 0 does nothing
 * and returns DUST_OK (the arrays may then be NULL).
 * INVALID_ARG: a NULL array, n < 0, misaligned elements, lr or weight_decay
 * not finite, weight_decay < 0, momentum outside [0, 1].  Asynchronous on
 * `stream`; allocates nothing.
 */
dust_status dust_sgd_step(float* W, const float* G, float* momentum_buf, int64_t n, float lr,
                          float momentum, float weight_decay, void* W_bf16, void* stream);

/*
 * One step of Adam (Kingma & Ba, 2015) with decoupled weight decay (AdamW) on
 * n fp32 parameters (the pages report that Adam works on the estimate
 * unchanged: Dust translation §3.3):
 *   m <- beta1 m + (1 - beta1) G,   v <- beta2 v + (1 - beta2) G^2,
 *   W <- W - lr ( (m / (1 - beta1^step)) / (sqrt(v / (1 - beta2^step)) + eps)
 *                 + weight_decay W ).
 * step counts from 1; m and v (device, n fp32, caller-owned) start at zero.
 * Arrays as for dust_sgd_step.  INVALID_ARG also for step < 1, beta outside
 * [0, 1), eps <= 0.
 */
dust_status dust_adam_step(float* W, const float* G, float* m, float* v, int64_t n, float lr,
                           float beta1, float beta2, float eps, float weight_decay,
                           int64_t step, void* W_bf16, void* stream);

/* Workspace bytes for dust_head_backprop with these sizes. */
size_t dust_head_backprop_workspace(int64_t T, int64_t V, int64_t d);

/*
 * The exact head gradient that the estimate is compared with (the pages tune
 * by the single-batch cosine with backprop: Dust translation §2.3, §4.2):
 *   g_t = softmax(z_t) - e_{y_t},   G_W = sum_t g_t x_t^T.
 * Arguments as for dust_head_estimate (no noise): g_out (T x V fp32) may be
 * NULL; G_W (V x d fp32) is computed from g and x rounded to bf16 with fp32
 * accumulation.  A target outside [0, V) sets DUST_ERR_DEVICE_RANGE in the
 * workspace status word (its row then has no -1 term).
 */
dust_status dust_head_backprop(const float* logits, const int32_t* targets, const void* x,
                               dust_dtype x_dtype, int64_t T, int64_t V, int64_t d,
                               float* g_out, float* G_W, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * Failure-path check of the bounded waits: a one-warp kernel waits on a
 * barrier that nothing arrives at, gives up after limit_ns (1 .. 1e9) and
 * records DUST_ERR_TIMEOUT in the status word of `ws` (>= 256 bytes), exactly
 * as a stalled pipeline inside the estimators would.  Read it back with
 * dust_workspace_status.
 */
dust_status dust_wait_selftest(void* ws, uint64_t limit_ns, void* stream);

/*
 * Issue-rate probe for the benchmark's rooflines: launches 148 x 8 CTAs of 256
 * threads (*threads_out receives the count) on `stream`, each thread running
 * `iters` rounds over eight independent chains of one operation:
 *   kind 0: a 32 x 32 -> 64-bit multiply and an xor of its halves (Philox's
 *           step; 16 operations per thread and round),
 *   kind 1: ex2.approx (8 XU operations per thread and round),
 *   kind 2: fp32 fma (8 operations per thread and round),
 *   kind 3, 4: kind 0's step with the product's halves as two 32-bit
 *           multiplies, written as PTX (3) or as C (4) (16 per round),
 *   kind 5: packed fp32 fma, fma.rn.f32x2 (2 operations per instruction; 16
 *           operations per thread and round).
 * The caller times it with events on `stream`.  `sink` (device, >= 1 KB) only
 * keeps the results alive.  INVALID_ARG for another kind, iters outside
 * [1, 2^32], or a NULL pointer.
 */
dust_status dust_issue_probe(int kind, int64_t iters, int64_t* threads_out, void* sink,
                             void* stream);

/* ------------------------------------------------------------------------ */
/* A whole block: one perturbed pass per layer type                           */
/* ------------------------------------------------------------------------ */

/*
 * The pages perturb the different layer types of a block in separate
 * forwards, so that one type's noise never moves another type's loss
 * (Dust translation §2.3; laoyaoba.com section 机制拆解).  A dust_layer_job
 * describes one such pass, for one weight, from the block's cached clean
 * activations; dust_block_estimate validates a list of them, gives each its
 * own slice of one workspace, requires their noise layer ids to differ, and
 * runs them as separate estimator calls, spread round-robin over the
 * caller's streams.
 */
typedef enum {
    DUST_JOB_HEAD = 0,        /* dust_head_estimate                            */
    DUST_JOB_LINEAR = 1,      /* dust_linear_estimate (interior, MLP input)    */
    DUST_JOB_ATTN_VALUE = 2,  /* dust_attn_value_estimate                      */
    DUST_JOB_ATTN_GATE = 3,   /* dust_attn_gate_estimate                       */
    DUST_JOB_ATTN_QUERY = 4,  /* dust_attn_qk_estimate, which = 0              */
    DUST_JOB_ATTN_KEY = 5     /* dust_attn_qk_estimate, which = 1              */
} dust_job_type;

/*
 * One layer type's pass.  `in` holds the entry point's device inputs in its
 * own argument order; `x`/`x_dtype`/`d_in` are the weight's input; the sizes
 * n1..n3 are the entry point's remaining dimensions:
 *
 *   HEAD        in = {logits, targets}                  n1 = V
 *   LINEAR      in = {y1, W2, W_head, z_clean, targets}  n1 = C, n2 = d_model,
 *                                                        n3 = V, ema_decay
 *   ATTN_VALUE  in = {P, E}                              n1 = H
 *   ATTN_GATE   in = {z, o, E}                           n1 = C
 *   ATTN_QUERY,
 *   ATTN_KEY    in = {Q, Kk, V, O, P, E}                 n1 = H
 *
 * (head: d = d_in; attention: dv = 64; LINEAR: x must be DUST_BF16, as
 * dust_linear_estimate reads it).  Unused `in` entries and sizes are
 * ignored.  nz is the pass's noise (its `layer` must differ from every other
 * job's); g_hat (or NULL) and G_W are the outputs, as for the entry point.
 */
typedef struct {
    int type;             /* dust_job_type */
    const void* in[6];
    const void* x;
    dust_dtype x_dtype;
    int64_t T, seq_len, d_in;
    int64_t n1, n2, n3;
    float ema_decay;
    dust_noise nz;
    float* g_hat;
    float* G_W;
} dust_layer_job;

/* Workspace bytes for the jobs: each job's own workspace, 256-byte aligned,
 * in list order.  0 if n < 1, a type is unknown or a job's sizes are
 * invalid for its entry point. */
size_t dust_block_workspace(const dust_layer_job* jobs, int n);

/* Byte offset of job j's slice in that workspace (its status word is the
 * slice's first word: dust_workspace_status(ws + offset, ...)); (size_t)-1
 * if j is out of range or the jobs are invalid. */
size_t dust_block_job_offset(const dust_layer_job* jobs, int n, int j);

/*
 * Runs the jobs: job j on streams[j % nstreams] (or on the default stream
 * when streams is NULL or nstreams < 1).  With several streams, every stream
 * first waits for the work already queued on streams[0], and streams[0]
 * finally waits for all of them, so the call is ordered on streams[0] like a
 * single estimator call.  Checked before anything is queued: n >= 1, known
 * types, distinct nz.layer across jobs, non-NULL G_W, bf16 x for LINEAR,
 * a workspace of dust_block_workspace bytes (256-byte aligned).  A job's
 * own argument errors are returned as its entry point returns them; jobs
 * before it have been queued by then.  Device-side status: per job, at its
 * offset.
 */
dust_status dust_block_estimate(const dust_layer_job* jobs, int n, void* ws, size_t ws_bytes,
                                void* const* streams, int nstreams);

/*
 * Benchmark hook.  While set, every launch of an entry point's main kernels
 * (the head's draw kernel; the interior layer's two re-forward GEMMs, in the
 * order GEMM 1, GEMM 2 with the cross-entropy epilogue per chunk of draws,
 * then its credit and g pass; the embedding's piece sums; the attention
 * kernels; the optimiser step) is bracketed on its stream by
 * cudaEventRecord(start_events[n]) and cudaEventRecord(
 * stop_events[n]) for n = 0, 1, ... up to capacity - 1.  The events are the
 * caller's (created with timing enabled).  Passing NULL arrays turns the hook
 * off.  The hook is process-wide and not thread-safe: it is for timing runs.
 * dust_kernel_event_count returns how many pairs were recorded since the last
 * dust_set_kernel_events.
 */
dust_status dust_set_kernel_events(void* const* start_events, void* const* stop_events,
                                   int capacity);
int dust_kernel_event_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DUST_H */
