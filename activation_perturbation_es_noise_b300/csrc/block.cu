// block.cu -- one perturbed pass per layer type of a block, on the caller's
// streams.
//
// The pages perturb each layer type in a forward of its own, so that the
// noise of one type does not move the loss another type is credited with
// (Dust translation §2.3; laoyaoba.com, section 机制拆解).  Every estimator
// entry point is already such a pass from cached clean activations; this file
// is the host-side scheduler over them: it sizes and carves one workspace,
// checks that the passes use distinct noise layers, and queues them
// round-robin on the given streams, joined back onto the first stream.
// Nothing here launches a kernel of its own.
#include <cstring>
#include <mutex>
#include <vector>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {
namespace {

size_t job_workspace(const dust_layer_job& j) {
    const uint32_t K = j.nz.num_draws;
    switch (j.type) {
        case DUST_JOB_HEAD: return dust_head_workspace(j.T, j.n1, j.d_in, K);
        case DUST_JOB_LINEAR: return dust_linear_workspace(j.T, j.d_in, j.n1, j.n2, j.n3, K);
        case DUST_JOB_ATTN_VALUE: return dust_attn_value_workspace(j.T, j.seq_len, j.n1, 64, j.d_in, K);
        case DUST_JOB_ATTN_GATE: return dust_attn_gate_workspace(j.T, j.seq_len, j.n1, j.d_in, K);
        case DUST_JOB_ATTN_QUERY:
        case DUST_JOB_ATTN_KEY: return dust_attn_qk_workspace(j.T, j.seq_len, j.n1, 64, j.d_in, K);
        default: return 0;
    }
}

// Offsets of every job's slice; false if a job is invalid.
bool plan(const dust_layer_job* jobs, int n, std::vector<size_t>& off, size_t& total) {
    if (!jobs || n < 1) return false;
    off.assign(static_cast<size_t>(n), 0);
    size_t at = 0;
    for (int j = 0; j < n; ++j) {
        const size_t b = job_workspace(jobs[j]);
        if (b == 0) return false;
        off[j] = at;
        at += static_cast<size_t>(round_up(static_cast<int64_t>(b), 256));
    }
    total = at;
    return true;
}

// The job's own entry-point checks on its slice of the workspace, run for
// every job before anything is queued.
dust_status check_job(const dust_layer_job& j, const void* ws, size_t bytes) {
    const void* const* in = j.in;
    const float* f0 = static_cast<const float*>(in[0]);
    switch (j.type) {
        case DUST_JOB_HEAD:
            return head_estimate_check(f0, static_cast<const int32_t*>(in[1]), j.x, j.x_dtype, j.T,
                                       j.n1, j.d_in, j.nz, DUST_BASELINE_MEAN, j.g_hat, j.G_W,
                                       ws, bytes);
        case DUST_JOB_LINEAR:
            // the interior entry point reads x as bf16 only
            if (j.x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
            return linear_estimate_check(j.x, f0, in[1], j.ema_decay, in[2],
                                         static_cast<const float*>(in[3]),
                                         static_cast<const int32_t*>(in[4]), j.T, j.seq_len,
                                         j.d_in, j.n1, j.n2, j.n3, j.nz, j.g_hat, j.G_W, ws,
                                         bytes);
        case DUST_JOB_ATTN_VALUE:
            return attn_value_check(f0, static_cast<const float*>(in[1]), j.x, j.x_dtype, j.T,
                                    j.seq_len, j.n1, 64, j.d_in, j.nz, j.g_hat, j.G_W, ws, bytes);
        case DUST_JOB_ATTN_GATE:
            return attn_gate_check(f0, static_cast<const float*>(in[1]),
                                   static_cast<const float*>(in[2]), j.x, j.x_dtype, j.T,
                                   j.seq_len, j.n1, j.d_in, j.nz, j.g_hat, j.G_W, ws, bytes);
        case DUST_JOB_ATTN_QUERY:
        case DUST_JOB_ATTN_KEY:
            return attn_qk_check(j.type == DUST_JOB_ATTN_KEY ? 1 : 0, f0,
                                 static_cast<const float*>(in[1]),
                                 static_cast<const float*>(in[2]),
                                 static_cast<const float*>(in[3]),
                                 static_cast<const float*>(in[4]),
                                 static_cast<const float*>(in[5]), j.x, j.x_dtype, j.T,
                                 j.seq_len, j.n1, 64, j.d_in, j.nz, j.g_hat, j.G_W, ws, bytes);
        default: return DUST_ERR_INVALID_ARG;
    }
}

// Byte ranges of one job's buffers: its outputs (g_hat, G_W) and every input
// it reads, sized from the job's dimensions (all already validated).
struct Range {
    uintptr_t lo, hi;
};

int64_t out_width(const dust_layer_job& j) {  // channels of g_hat / rows of G_W
    switch (j.type) {
        case DUST_JOB_ATTN_VALUE:
        case DUST_JOB_ATTN_QUERY:
        case DUST_JOB_ATTN_KEY: return j.n1 * 64;
        default: return j.n1;
    }
}

void add_range(std::vector<Range>& v, const void* p, int64_t bytes) {
    if (p && bytes > 0) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        v.push_back({a, a + static_cast<uintptr_t>(bytes)});
    }
}

void job_outputs(const dust_layer_job& j, std::vector<Range>& v) {
    const int64_t C = out_width(j);
    add_range(v, j.g_hat, j.T * C * 4);
    add_range(v, j.G_W, C * j.d_in * 4);
}

void job_inputs(const dust_layer_job& j, std::vector<Range>& v) {
    const int64_t T = j.T, L = j.seq_len;
    add_range(v, j.x, T * j.d_in * (j.x_dtype == DUST_BF16 ? 2 : 4));
    switch (j.type) {
        case DUST_JOB_HEAD:
            add_range(v, j.in[0], T * j.n1 * 4);
            add_range(v, j.in[1], T * 4);
            break;
        case DUST_JOB_LINEAR:
            add_range(v, j.in[0], T * j.n1 * 4);        // y1
            add_range(v, j.in[1], j.n2 * j.n1 * 2);     // W2
            add_range(v, j.in[2], j.n3 * j.n2 * 2);     // W_head
            add_range(v, j.in[3], T * j.n3 * 4);        // z_clean
            add_range(v, j.in[4], T * 4);               // targets
            break;
        case DUST_JOB_ATTN_VALUE:
            add_range(v, j.in[0], (T / L) * j.n1 * L * L * 4);  // P
            add_range(v, j.in[1], T * j.n1 * 64 * 4);           // E
            break;
        case DUST_JOB_ATTN_GATE:
            for (int k = 0; k < 3; ++k) add_range(v, j.in[k], T * j.n1 * 4);
            break;
        case DUST_JOB_ATTN_QUERY:
        case DUST_JOB_ATTN_KEY:
            for (int k = 0; k < 4; ++k) add_range(v, j.in[k], T * j.n1 * 64 * 4);  // Q K V O
            add_range(v, j.in[4], (T / L) * j.n1 * L * L * 4);                  // P
            add_range(v, j.in[5], T * j.n1 * 64 * 4);                           // E
            break;
        default: break;
    }
}

bool overlap(const std::vector<Range>& a, const std::vector<Range>& b) {
    for (const Range& x : a)
        for (const Range& y : b)
            if (x.lo < y.hi && y.lo < x.hi) return true;
    return false;
}

// Every check of the block call, before any event or launch: the jobs'
// own argument checks on their workspace slices, distinct noise layers, and
// no job writing memory that another job reads or writes (with several
// streams that would race; on one stream a later job would clobber an
// earlier one's result).
dust_status check_block(const dust_layer_job* jobs, int n, const std::vector<size_t>& off,
                        size_t total, void* ws, size_t ws_bytes) {
    if (!ws || ws_bytes < total || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    const uint8_t* base = static_cast<const uint8_t*>(ws);
    std::vector<std::vector<Range>> outs(static_cast<size_t>(n)), ins(static_cast<size_t>(n));
    for (int j = 0; j < n; ++j) {
        const size_t bytes = (j + 1 < n ? off[j + 1] : total) - off[j];
        const dust_status st = check_job(jobs[j], base + off[j], bytes);
        if (st != DUST_OK) return st;
        for (int k = 0; k < j; ++k)  // separate noise per pass
            if (jobs[k].nz.layer == jobs[j].nz.layer) return DUST_ERR_INVALID_ARG;
        job_outputs(jobs[j], outs[j]);
        job_inputs(jobs[j], ins[j]);
        add_range(ins[j], base + off[j], static_cast<int64_t>(bytes));  // its workspace slice
        if (outs[j].size() == 2 &&  // g_hat and G_W of one job
            overlap({outs[j][0]}, {outs[j][1]}))
            return DUST_ERR_INVALID_ARG;
    }
    for (int j = 0; j < n; ++j)
        for (int k = 0; k < n; ++k) {
            if (k == j) continue;
            if (overlap(outs[j], outs[k]) || overlap(outs[j], ins[k])) return DUST_ERR_INVALID_ARG;
        }
    return DUST_OK;
}

dust_status run_job(const dust_layer_job& j, void* ws, size_t bytes, void* stream) {
    const void* const* in = j.in;
    const float* f0 = static_cast<const float*>(in[0]);
    switch (j.type) {
        case DUST_JOB_HEAD:
            return dust_head_estimate(f0, static_cast<const int32_t*>(in[1]), j.x, j.x_dtype, j.T,
                                      j.n1, j.d_in, j.nz, j.g_hat, j.G_W, ws, bytes, stream);
        case DUST_JOB_LINEAR:
            return dust_linear_estimate(j.x, f0, in[1], j.ema_decay, in[2],
                                        static_cast<const float*>(in[3]),
                                        static_cast<const int32_t*>(in[4]), j.T, j.seq_len, j.d_in,
                                        j.n1, j.n2, j.n3, j.nz, j.g_hat, j.G_W, ws, bytes, stream);
        case DUST_JOB_ATTN_VALUE:
            return dust_attn_value_estimate(f0, static_cast<const float*>(in[1]), j.x, j.x_dtype,
                                            j.T, j.seq_len, j.n1, 64, j.d_in, j.nz, j.g_hat, j.G_W,
                                            ws, bytes, stream);
        case DUST_JOB_ATTN_GATE:
            return dust_attn_gate_estimate(f0, static_cast<const float*>(in[1]),
                                           static_cast<const float*>(in[2]), j.x, j.x_dtype, j.T,
                                           j.seq_len, j.n1, j.d_in, j.nz, j.g_hat, j.G_W, ws,
                                           bytes, stream);
        case DUST_JOB_ATTN_QUERY:
        case DUST_JOB_ATTN_KEY:
            return dust_attn_qk_estimate(j.type == DUST_JOB_ATTN_KEY ? 1 : 0, f0,
                                         static_cast<const float*>(in[1]),
                                         static_cast<const float*>(in[2]),
                                         static_cast<const float*>(in[3]),
                                         static_cast<const float*>(in[4]),
                                         static_cast<const float*>(in[5]), j.x, j.x_dtype, j.T,
                                         j.seq_len, j.n1, 64, j.d_in, j.nz, j.g_hat, j.G_W, ws,
                                         bytes, stream);
        default: return DUST_ERR_INVALID_ARG;
    }
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" size_t dust_block_workspace(const dust_layer_job* jobs, int n) {
    std::vector<size_t> off;
    size_t total = 0;
    return plan(jobs, n, off, total) ? total : 0;
}

extern "C" size_t dust_block_job_offset(const dust_layer_job* jobs, int n, int j) {
    std::vector<size_t> off;
    size_t total = 0;
    if (j < 0 || j >= n || !plan(jobs, n, off, total)) return static_cast<size_t>(-1);
    return off[j];
}

namespace dust {
namespace {

// Fork/join events, created once per device and reused by every call made
// with that device current; the mutex is held for the whole call so that two
// host threads never record the same event at once.
struct BlockEvents {
    std::mutex mu;
    std::vector<cudaEvent_t> ev[64];
};
BlockEvents& block_events() {
    static BlockEvents* e = new BlockEvents();  // never destroyed: events live until exit
    return *e;
}

dust_status events_for_device(std::vector<cudaEvent_t>& ev, int need) {
    while (static_cast<int>(ev.size()) < need) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            return DUST_ERR_CUDA;
        }
        ev.push_back(e);
    }
    return DUST_OK;
}

}  // namespace
}  // namespace dust

extern "C" dust_status dust_block_estimate(const dust_layer_job* jobs, int n, void* ws,
                                           size_t ws_bytes, void* const* streams, int nstreams) {
    std::vector<size_t> off;
    size_t total = 0;
    if (!plan(jobs, n, off, total)) return DUST_ERR_INVALID_ARG;
    const dust_status chk = check_block(jobs, n, off, total, ws, ws_bytes);
    if (chk != DUST_OK) return chk;
    const int ns = (streams && nstreams > 0) ? nstreams : 1;
    auto stream_of = [&](int k) -> void* { return (streams && nstreams > 0) ? streams[k] : nullptr; };

    std::unique_lock<std::mutex> lock;
    std::vector<cudaEvent_t>* ev = nullptr;
    if (ns > 1) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return DUST_ERR_CUDA;
        }
        if (dev < 0 || dev >= 64) return DUST_ERR_UNSUPPORTED;
        BlockEvents& be = block_events();
        lock = std::unique_lock<std::mutex>(be.mu);
        ev = &be.ev[dev];
        if (events_for_device(*ev, ns) != DUST_OK) return DUST_ERR_CUDA;
        // Fork: every other stream waits for what is queued on the first.
        if (cudaEventRecord((*ev)[0], static_cast<cudaStream_t>(stream_of(0))) != cudaSuccess) {
            (void)cudaGetLastError();
            return DUST_ERR_CUDA;
        }
        for (int k = 1; k < ns; ++k)
            if (cudaStreamWaitEvent(static_cast<cudaStream_t>(stream_of(k)), (*ev)[0], 0) !=
                cudaSuccess) {
                (void)cudaGetLastError();
                return DUST_ERR_CUDA;
            }
    }
    dust_status st = DUST_OK;
    uint8_t* base = static_cast<uint8_t*>(ws);
    for (int j = 0; j < n && st == DUST_OK; ++j) {
        const size_t bytes = (j + 1 < n ? off[j + 1] : total) - off[j];
        st = run_job(jobs[j], base + off[j], bytes, stream_of(j % ns));
    }
    // Join: the first stream waits for every other one (also after an error,
    // so that nothing queued is left unordered with the caller's stream).
    if (ns > 1) {
        for (int k = 1; k < ns; ++k) {
            if (cudaEventRecord((*ev)[k], static_cast<cudaStream_t>(stream_of(k))) != cudaSuccess ||
                cudaStreamWaitEvent(static_cast<cudaStream_t>(stream_of(0)), (*ev)[k], 0) !=
                    cudaSuccess) {
                (void)cudaGetLastError();
                st = st == DUST_OK ? DUST_ERR_CUDA : st;
            }
        }
    }
    return st;
}
