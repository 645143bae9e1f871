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

extern "C" dust_status dust_block_estimate(const dust_layer_job* jobs, int n, void* ws,
                                           size_t ws_bytes, void* const* streams, int nstreams) {
    std::vector<size_t> off;
    size_t total = 0;
    if (!plan(jobs, n, off, total)) return DUST_ERR_INVALID_ARG;
    for (int j = 0; j < n; ++j) {
        if (!jobs[j].G_W) return DUST_ERR_INVALID_ARG;
        // the interior entry point reads x as bf16 only
        if (jobs[j].type == DUST_JOB_LINEAR && jobs[j].x_dtype != DUST_BF16) return DUST_ERR_INVALID_ARG;
        for (int k = 0; k < j; ++k)  // separate noise per pass
            if (jobs[k].nz.layer == jobs[j].nz.layer) return DUST_ERR_INVALID_ARG;
    }
    if (!ws || ws_bytes < total || !aligned(ws, 256)) return DUST_ERR_WORKSPACE;
    const int ns = (streams && nstreams > 0) ? nstreams : 1;
    auto stream_of = [&](int k) -> void* { return (streams && nstreams > 0) ? streams[k] : nullptr; };

    // Fork: every other stream waits for what is queued on the first.
    std::vector<cudaEvent_t> ev;
    auto release = [&]() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    };
    if (ns > 1) {
        ev.resize(static_cast<size_t>(ns), nullptr);
        for (int k = 0; k < ns; ++k) {
            if (cudaEventCreateWithFlags(&ev[k], cudaEventDisableTiming) != cudaSuccess) {
                ev.resize(static_cast<size_t>(k));
                release();
                return DUST_ERR_CUDA;
            }
        }
        if (cudaEventRecord(ev[0], static_cast<cudaStream_t>(stream_of(0))) != cudaSuccess) {
            release();
            return DUST_ERR_CUDA;
        }
        for (int k = 1; k < ns; ++k)
            if (cudaStreamWaitEvent(static_cast<cudaStream_t>(stream_of(k)), ev[0], 0) != cudaSuccess) {
                release();
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
            if (cudaEventRecord(ev[k], static_cast<cudaStream_t>(stream_of(k))) != cudaSuccess ||
                cudaStreamWaitEvent(static_cast<cudaStream_t>(stream_of(0)), ev[k], 0) != cudaSuccess)
                st = st == DUST_OK ? DUST_ERR_CUDA : st;
        }
        release();
    }
    return st;
}
