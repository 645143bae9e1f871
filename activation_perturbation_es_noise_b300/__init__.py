"""Python binding of the Dust estimator engine (libdust.so, C ABI in include/dust.h).

Argument marshalling only: every step of the estimator runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; outputs and workspaces are
allocated here with torch (device memory is the caller's, as the C ABI
requires) and their pointers are passed with the current CUDA stream.

There is no CPU path: if libdust.so is missing or cannot be loaded, every call
raises.  Build it with `python -m activation_perturbation_es_noise_b300.build`.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# DUST_LIBRARY=debug loads the bounds-checked build (libdust_debug.so) instead.
LIB_PATH = os.path.join(HERE, "libdust_debug.so" if os.environ.get("DUST_LIBRARY") == "debug"
                        else "libdust.so")

DUST_OK = 0
STATUS_NAMES = {0: "DUST_OK", 1: "DUST_ERR_INVALID_ARG", 2: "DUST_ERR_UNSUPPORTED",
                3: "DUST_ERR_WORKSPACE", 4: "DUST_ERR_CUDA", 5: "DUST_ERR_TIMEOUT",
                6: "DUST_ERR_DEVICE_RANGE"}
DUST_F32, DUST_BF16 = 0, 1

# Entry points declared in include/dust.h.
EXPORTS = ("dust_status_string", "dust_abi_version", "dust_workspace_status",
           "dust_head_workspace", "dust_head_estimate", "dust_linear_workspace",
           "dust_linear_estimate", "dust_embed_workspace", "dust_embed_scatter",
           "dust_embed_scatter_static", "dust_philox_fill", "dust_gemm_bf16", "dust_set_kernel_events",
           "dust_kernel_event_count", "dust_wait_selftest", "dust_sgd_step", "dust_adam_step",
           "dust_head_backprop_workspace", "dust_head_backprop", "dust_head_estimate_baseline",
           "dust_attn_value_workspace", "dust_attn_value_estimate", "dust_attn_gate_workspace",
           "dust_attn_gate_estimate", "dust_attn_qk_workspace", "dust_attn_qk_estimate",
           "dust_block_workspace", "dust_block_job_offset", "dust_block_estimate",
           "dust_issue_probe", "dust_head_chunked_workspace",
           "dust_head_estimate_chunked", "dust_es_perturb", "dust_es_estimate",
           "dust_box_muller_fast", "dust_debug_build", "dust_debug_fault",
           "dust_debug_check_index")
BASELINE_MEAN, BASELINE_LEAVE_ONE_OUT, BASELINE_ANTITHETIC = 0, 1, 2


class DustError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s returned %s (%s)" % (fn, STATUS_NAMES.get(status, status),
                                                    _status_string(status)))


class DustNoise(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("layer", ctypes.c_uint32),
                ("draw0", ctypes.c_uint32), ("num_draws", ctypes.c_uint32),
                ("token0", ctypes.c_uint32), ("sigma", ctypes.c_float),
                ("gamma", ctypes.c_float)]


JOB_HEAD, JOB_LINEAR, JOB_ATTN_VALUE, JOB_ATTN_GATE, JOB_ATTN_QUERY, JOB_ATTN_KEY = range(6)


class DustLayerJob(ctypes.Structure):
    _fields_ = [("type", ctypes.c_int), ("in_", ctypes.c_void_p * 6), ("x", ctypes.c_void_p),
                ("x_dtype", ctypes.c_int), ("T", ctypes.c_int64), ("seq_len", ctypes.c_int64),
                ("d_in", ctypes.c_int64), ("n1", ctypes.c_int64), ("n2", ctypes.c_int64),
                ("n3", ctypes.c_int64), ("ema_decay", ctypes.c_float), ("nz", DustNoise),
                ("g_hat", ctypes.c_void_p), ("G_W", ctypes.c_void_p)]


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U32 = ctypes.c_uint32
_SZ = ctypes.c_size_t


def lib():
    """The loaded libdust.so (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdust.so is not built: run "
                               "`python -m activation_perturbation_es_noise_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.dust_status_string.argtypes = [ctypes.c_int]
        L.dust_status_string.restype = ctypes.c_char_p
        L.dust_abi_version.restype = ctypes.c_int
        L.dust_workspace_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int)]
        L.dust_head_workspace.argtypes = [_I64, _I64, _I64, _U32]
        L.dust_head_workspace.restype = _SZ
        L.dust_head_estimate.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, DustNoise,
                                         _P, _P, _P, _SZ, _P]
        L.dust_linear_workspace.argtypes = [_I64, _I64, _I64, _I64, _I64, _U32]
        L.dust_linear_workspace.restype = _SZ
        L.dust_linear_estimate.argtypes = [_P, _P, _P, ctypes.c_float, _P, _P, _P, _I64, _I64,
                                           _I64, _I64, _I64, _I64, DustNoise, _P, _P, _P, _SZ,
                                           _P]
        L.dust_embed_workspace.argtypes = [_I64, _I64, _I64]
        L.dust_embed_workspace.restype = _SZ
        L.dust_embed_scatter.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]
        L.dust_embed_scatter_static.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P, _P]
        L.dust_philox_fill.argtypes = [ctypes.c_uint64, _U32, _U32, _I64, _I64, _I64, _P, _P, _P]
        L.dust_box_muller_fast.argtypes = [_P, _I64, _P, _P]
        L.dust_debug_build.restype = ctypes.c_int
        L.dust_debug_fault.restype = ctypes.c_uint64
        L.dust_debug_check_index.argtypes = [_I64, _I64, _P, _P]
        L.dust_gemm_bf16.argtypes = [_P, ctypes.c_int, _I64, _P, ctypes.c_int, _I64, _I64, _I64,
                                     _I64, _P, _I64, _P, _SZ, _P]
        L.dust_set_kernel_events.argtypes = [_P, _P, ctypes.c_int]
        L.dust_wait_selftest.argtypes = [_P, ctypes.c_uint64, _P]
        L.dust_kernel_event_count.restype = ctypes.c_int
        _F = ctypes.c_float
        L.dust_sgd_step.argtypes = [_P, _P, _P, _I64, _F, _F, _F, _P, _P]
        L.dust_adam_step.argtypes = [_P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _I64, _P, _P]
        L.dust_head_estimate_baseline.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                                  DustNoise, ctypes.c_int, _P, _P, _P, _SZ, _P]
        L.dust_attn_value_workspace.argtypes = [_I64, _I64, _I64, _I64, _I64, _U32]
        L.dust_attn_value_workspace.restype = _SZ
        L.dust_attn_value_estimate.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _I64,
                                               _I64, DustNoise, _P, _P, _P, _SZ, _P]
        JP = ctypes.POINTER(DustLayerJob)
        L.dust_block_workspace.argtypes = [JP, ctypes.c_int]
        L.dust_block_workspace.restype = _SZ
        L.dust_block_job_offset.argtypes = [JP, ctypes.c_int, ctypes.c_int]
        L.dust_block_job_offset.restype = _SZ
        L.dust_block_estimate.argtypes = [JP, ctypes.c_int, _P, _SZ, ctypes.POINTER(_P),
                                          ctypes.c_int]
        L.dust_attn_qk_workspace.argtypes = [_I64, _I64, _I64, _I64, _I64, _U32]
        L.dust_attn_qk_workspace.restype = _SZ
        L.dust_attn_qk_estimate.argtypes = [ctypes.c_int, _P, _P, _P, _P, _P, _P, _P,
                                            ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                            DustNoise, _P, _P, _P, _SZ, _P]
        L.dust_attn_gate_workspace.argtypes = [_I64, _I64, _I64, _I64, _U32]
        L.dust_attn_gate_workspace.restype = _SZ
        L.dust_attn_gate_estimate.argtypes = [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _I64,
                                              DustNoise, _P, _P, _P, _SZ, _P]
        L.dust_issue_probe.argtypes = [ctypes.c_int, _I64, ctypes.POINTER(_I64), _P, _P]
        L.dust_es_perturb.argtypes = [_P, _I64, DustNoise, _P, _P]
        L.dust_es_estimate.argtypes = [_P, _I64, DustNoise, _P, _P]
        L.dust_head_chunked_workspace.argtypes = [_I64, _I64, _I64, _U32, _I64]
        L.dust_head_chunked_workspace.restype = _SZ
        L.dust_head_estimate_chunked.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64,
                                                 DustNoise, _I64, _P, _P, _P, _SZ, _P]
        L.dust_head_backprop_workspace.argtypes = [_I64, _I64, _I64]
        L.dust_head_backprop_workspace.restype = _SZ
        L.dust_head_backprop.argtypes = [_P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P, _P, _P,
                                         _SZ, _P]
        for name in ("dust_set_kernel_events", "dust_wait_selftest", "dust_workspace_status",
                     "dust_head_estimate", "dust_linear_estimate", "dust_embed_scatter",
                     "dust_embed_scatter_static", "dust_philox_fill", "dust_gemm_bf16",
                     "dust_sgd_step", "dust_adam_step", "dust_head_backprop",
                     "dust_head_estimate_baseline", "dust_attn_value_estimate",
                     "dust_attn_gate_estimate", "dust_attn_qk_estimate", "dust_block_estimate",
                     "dust_issue_probe",
                     "dust_head_estimate_chunked", "dust_es_perturb", "dust_es_estimate",
                     "dust_box_muller_fast", "dust_debug_check_index"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _status_string(status):
    try:
        return lib().dust_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - only used to decorate an error message
        return "?"


def _check(fn, status):
    if status != DUST_OK:
        raise DustError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _workspace(nbytes, device):
    # 256-byte aligned by the caching allocator.
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def noise(seed, sigma, K, layer=0, draw0=0, token0=0, gamma=0.0):
    return DustNoise(seed, layer, draw0, K, token0, sigma, gamma)


def workspace_status(ws, stream=None):
    """Status word the kernels left in a workspace (and clear it)."""
    out = ctypes.c_int(0)
    _check("dust_workspace_status", lib().dust_workspace_status(_ptr(ws), _stream(stream),
                                                                ctypes.byref(out)))
    return out.value


# ----------------------------------------------------------------- head ----
def head_workspace_bytes(T, V, d, K):
    return lib().dust_head_workspace(T, V, d, K)


def head_estimate(logits, targets, x, sigma, K, seed, layer=0, draw0=0, token0=0,
                  want_g=True, out=None, ws=None, stream=None, baseline=BASELINE_MEAN):
    """LM-head estimator on cached logits.  Returns (g_hat or None, G_W, ws).
    baseline: BASELINE_MEAN (the pages'), BASELINE_LEAVE_ONE_OUT or
    BASELINE_ANTITHETIC (K noise draws, each evaluated as +a and -a)."""
    _need_cuda(logits, targets, x)
    T, V = logits.shape
    d = x.shape[1]
    dev = logits.device
    if out is None:
        g = torch.empty((T, V), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((V, d), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(head_workspace_bytes(T, V, d, K), dev)
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be bf16 or fp32")
    nz = noise(seed, sigma, K, layer, draw0, token0)
    if baseline == BASELINE_MEAN:
        st = lib().dust_head_estimate(_ptr(logits), _ptr(targets), _ptr(x), xdt, T, V, d, nz,
                                      _ptr(g), _ptr(G), _ptr(ws), ws.numel(), _stream(stream))
    else:
        st = lib().dust_head_estimate_baseline(_ptr(logits), _ptr(targets), _ptr(x), xdt, T, V,
                                               d, nz, int(baseline), _ptr(g), _ptr(G), _ptr(ws),
                                               ws.numel(), _stream(stream))
    _check("dust_head_estimate", st)
    return g, G, ws


# ------------------------------------------------------------- interior ----
def linear_workspace_bytes(T, d_in, C, d_model, V, K):
    return lib().dust_linear_workspace(T, d_in, C, d_model, V, K)


def linear_estimate(x, y1, W2, ema_decay, W_head, z_clean, targets, seq_len, sigma, gamma, K,
                    seed, layer=1, draw0=0, token0=0, want_g=True, out=None, ws=None,
                    stream=None):
    """Interior linear-layer estimator.  Returns (g_hat or None, G_W1, ws)."""
    _need_cuda(x, y1, W2, W_head, z_clean, targets)
    T, d_in = x.shape
    C = y1.shape[1]
    d_model = W2.shape[0]
    V = W_head.shape[0]
    dev = x.device
    if out is None:
        g = torch.empty((T, C), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((C, d_in), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(linear_workspace_bytes(T, d_in, C, d_model, V, K), dev)
    st = lib().dust_linear_estimate(_ptr(x), _ptr(y1), _ptr(W2), float(ema_decay), _ptr(W_head),
                                    _ptr(z_clean), _ptr(targets), T, seq_len, d_in, C, d_model,
                                    V, noise(seed, sigma, K, layer, draw0, token0, gamma),
                                    _ptr(g), _ptr(G), _ptr(ws), ws.numel(), _stream(stream))
    _check("dust_linear_estimate", st)
    return g, G, ws


# ------------------------------------------------------------ embedding ----
def embed_workspace_bytes(T, d, V):
    return lib().dust_embed_workspace(T, d, V)


def embed_scatter(g_hat, ids, V, want_perm=True, out=None, ws=None, stream=None):
    """Embedding gradient G_E (V x d) and the stable order of the ids."""
    _need_cuda(g_hat, ids)
    T, d = g_hat.shape
    dev = g_hat.device
    if out is None:
        G = torch.empty((V, d), dtype=torch.float32, device=dev)
        perm = torch.empty(T, dtype=torch.int32, device=dev) if want_perm else None
    else:
        G, perm = out
    if ws is None:
        ws = _workspace(embed_workspace_bytes(T, d, V), dev)
    st = lib().dust_embed_scatter(_ptr(g_hat), _ptr(ids), T, d, V, _ptr(G), _ptr(perm),
                                  _ptr(ws), ws.numel(), _stream(stream))
    _check("dust_embed_scatter", st)
    return G, perm, ws


# ---------------------------------------------------------- test hooks ----
def philox_fill(seed, layer, draw, token0, ntok, nchan, device="cuda", stream=None):
    """(words uint32 as int32 tensor, normals fp32) of one draw, ntok x nchan."""
    words = torch.empty((ntok, nchan), dtype=torch.int32, device=device)
    normals = torch.empty((ntok, nchan), dtype=torch.float32, device=device)
    st = lib().dust_philox_fill(seed, layer, draw, token0, ntok, nchan, _ptr(words),
                                _ptr(normals), _stream(stream))
    _check("dust_philox_fill", st)
    return words, normals


def box_muller_fast(words, stream=None):
    """Normals (fp32, same shape) of device words taken in pairs (int32 tensor
    holding the uint32 bits, an even number of elements) by the kernels' fast
    Box-Muller."""
    _need_cuda(words)
    if words.dtype != torch.int32 or not words.is_contiguous() or words.numel() % 2:
        raise ValueError("words: contiguous int32 tensor with an even number of elements")
    out = torch.empty(words.shape, dtype=torch.float32, device=words.device)
    _check("dust_box_muller_fast",
           lib().dust_box_muller_fast(_ptr(words), words.numel() // 2, _ptr(out), _stream(stream)))
    return out


def debug_build():
    """True when the loaded library is the bounds-checked build."""
    return bool(lib().dust_debug_build())


def debug_fault():
    """Synchronise the device and return the first out-of-range index the
    debug build's checks met since the last call, as (file id, source line),
    or None; always None for the release library."""
    v = int(lib().dust_debug_fault())
    if v == 0:
        return None
    if v == (1 << 64) - 1:
        raise DustError("dust_debug_fault", 4)  # DUST_ERR_CUDA: the read itself failed
    return (v >> 32, v & 0xFFFFFFFF)


def debug_check_index(i, n, stream=None):
    """The debug build's index check on its own (nothing is addressed with i):
    True when 0 <= i < n; in the debug build a False also records a fault."""
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check("dust_debug_check_index",
           lib().dust_debug_check_index(int(i), int(n), _ptr(out), _stream(stream)))
    return bool(out.item())


def wait_selftest(limit_ns, stream=None):
    """Run the bounded-wait check; returns the status word it left."""
    ws = _workspace(256, torch.device("cuda"))
    _check("dust_wait_selftest", lib().dust_wait_selftest(_ptr(ws), int(limit_ns), _stream(stream)))
    return workspace_status(ws, stream)


def gemm_bf16(A, a_mn, B, b_mn, M, N, K, stream=None):
    """G (M x N fp32) = sum_k A(m,k) B(n,k) on the tensor cores."""
    _need_cuda(A, B)
    G = torch.empty((M, N), dtype=torch.float32, device=A.device)
    ws = _workspace(256, A.device)
    st = lib().dust_gemm_bf16(_ptr(A), int(a_mn), A.shape[1], _ptr(B), int(b_mn), B.shape[1],
                              M, N, K, _ptr(G), N, _ptr(ws), ws.numel(), _stream(stream))
    _check("dust_gemm_bf16", st)
    return G


class KernelTimer:
    """Times the dominant kernel of the library's entry points with CUDA events
    recorded by the library on the kernel's own stream (dust_set_kernel_events).

    with KernelTimer(capacity) as kt:  ... calls ...
    kt.total_ms() sums the recorded launches (synchronises on the events).
    """

    def __init__(self, capacity):
        self.start = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        self.stop = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        s = torch.cuda.current_stream()
        for e in self.start + self.stop:  # create the underlying events
            e.record(s)
        torch.cuda.synchronize()
        self._a0 = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.start])
        self._a1 = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.stop])
        self.capacity = capacity
        self.count = 0

    def __enter__(self):
        _check("dust_set_kernel_events",
               lib().dust_set_kernel_events(self._a0, self._a1, self.capacity))
        return self

    def __exit__(self, *exc):
        self.count = lib().dust_kernel_event_count()
        lib().dust_set_kernel_events(None, None, 0)
        return False

    def times_ms(self):
        for e in self.stop[:self.count]:
            e.synchronize()
        return [a.elapsed_time(b) for a, b in zip(self.start[:self.count], self.stop[:self.count])]

    def total_ms(self):
        return float(sum(self.times_ms()))


# ------------------------------------------------------------ optimiser ----
def _f32_params(*ts):
    _need_cuda(*ts)
    for t in ts:
        if t.dtype != torch.float32:
            raise ValueError("parameters, gradients and moments are fp32")
    n = ts[0].numel()
    if any(t.numel() != n for t in ts):
        raise ValueError("parameter, gradient and moment sizes differ")
    return n


def sgd_step(W, G, momentum_buf, lr, momentum=0.9, weight_decay=0.0, W_bf16=None, stream=None):
    """b <- momentum b + (G + weight_decay W); W <- W - lr b (in place)."""
    n = _f32_params(W, G, momentum_buf)
    if W_bf16 is not None:
        _need_cuda(W_bf16)
    _check("dust_sgd_step", lib().dust_sgd_step(_ptr(W), _ptr(G), _ptr(momentum_buf), n, lr,
                                                momentum, weight_decay, _ptr(W_bf16),
                                                _stream(stream)))


def adam_step(W, G, m, v, step, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
              W_bf16=None, stream=None):
    """One Adam step (decoupled weight decay), step counted from 1 (in place)."""
    n = _f32_params(W, G, m, v)
    if W_bf16 is not None:
        _need_cuda(W_bf16)
    _check("dust_adam_step", lib().dust_adam_step(_ptr(W), _ptr(G), _ptr(m), _ptr(v), n, lr,
                                                  beta1, beta2, eps, weight_decay, step,
                                                  _ptr(W_bf16), _stream(stream)))


def head_backprop(logits, targets, x, want_g=False, out=None, ws=None, stream=None):
    """Exact head gradient: returns (g or None, G_W, ws) with
    g_t = softmax(z_t) - e_{y_t} and G_W = sum_t g_t x_t^T."""
    _need_cuda(logits, targets, x)
    T, V = logits.shape
    d = x.shape[1]
    dev = logits.device
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    if out is None:
        g = torch.empty((T, V), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((V, d), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(lib().dust_head_backprop_workspace(T, V, d), dev)
    _check("dust_head_backprop",
           lib().dust_head_backprop(_ptr(logits), _ptr(targets), _ptr(x), xdt, T, V, d, _ptr(g),
                                    _ptr(G), _ptr(ws), ws.numel(), _stream(stream)))
    return g, G, ws


# ------------------------------------------------------------ attention ----
def attn_value_estimate(P, E, x, seq_len, sigma, gamma, K, seed, layer=2, draw0=0, token0=0,
                        want_g=True, out=None, ws=None, stream=None):
    """Value projection of an attention layer, scored by the attention-output
    error E (T x H*64).  P: (T/seq_len, H, seq_len, seq_len) fp32 cached
    probabilities.  Returns (g_hat or None, G_W, ws)."""
    _need_cuda(P, E, x)
    nseq, H, L, L2 = P.shape
    T, C = E.shape
    if L != seq_len or L2 != seq_len or nseq * L != T or C != H * 64:
        raise ValueError("P must be (T/seq_len, H, seq_len, seq_len) and E T x H*64")
    d_in = x.shape[1]
    dev = P.device
    if out is None:
        g = torch.empty((T, C), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((C, d_in), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(lib().dust_attn_value_workspace(T, seq_len, H, 64, d_in, K), dev)
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    _check("dust_attn_value_estimate",
           lib().dust_attn_value_estimate(_ptr(P), _ptr(E), _ptr(x), xdt, T, seq_len, H, 64,
                                          d_in, noise(seed, sigma, K, layer, draw0, token0, gamma),
                                          _ptr(g), _ptr(G), _ptr(ws), ws.numel(),
                                          _stream(stream)))
    return g, G, ws


def attn_gate_estimate(z, o, E, x, seq_len, sigma, gamma, K, seed, layer=3, draw0=0, token0=0,
                       want_g=True, out=None, ws=None, stream=None):
    """Gate projection of a gated attention output sig(z) * o, scored by the
    error E of the gated output (all T x C fp32).  Returns (g_hat or None, G_W, ws)."""
    _need_cuda(z, o, E, x)
    T, C = z.shape
    d_in = x.shape[1]
    dev = z.device
    if out is None:
        g = torch.empty((T, C), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((C, d_in), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(lib().dust_attn_gate_workspace(T, seq_len, C, d_in, K), dev)
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    _check("dust_attn_gate_estimate",
           lib().dust_attn_gate_estimate(_ptr(z), _ptr(o), _ptr(E), _ptr(x), xdt, T, seq_len, C,
                                         d_in, noise(seed, sigma, K, layer, draw0, token0, gamma),
                                         _ptr(g), _ptr(G), _ptr(ws), ws.numel(), _stream(stream)))
    return g, G, ws


def attn_qk_estimate(which, Q, Kk, V, O, P, E, x, seq_len, sigma, gamma, K, seed, layer=None,
                     draw0=0, token0=0, want_g=True, out=None, ws=None, stream=None):
    """Query (which 0) or key (which 1) projection of a causal softmax
    attention layer, scored by the attention-output error E.  Q, Kk, V, O, E:
    T x H*64 fp32 (the clean forward and the error); P: (T/seq_len, H,
    seq_len, seq_len) fp32, the clean probabilities.  The noise layer defaults
    to 4 (queries) or 5 (keys).  Returns (g_hat or None, G_W, ws)."""
    _need_cuda(Q, Kk, V, O, P, E, x)
    if which not in (0, 1):
        raise ValueError("which is 0 (queries) or 1 (keys)")
    if layer is None:
        layer = 4 + which
    nseq, H, L, L2 = P.shape
    T, C = Q.shape
    if L != seq_len or L2 != seq_len or nseq * L != T or C != H * 64:
        raise ValueError("P must be (T/seq_len, H, seq_len, seq_len) and Q T x H*64")
    for t in (Kk, V, O, E):
        if tuple(t.shape) != (T, C):
            raise ValueError("Kk, V, O and E must have Q's shape")
    d_in = x.shape[1]
    dev = Q.device
    if out is None:
        g = torch.empty((T, C), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((C, d_in), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(lib().dust_attn_qk_workspace(T, seq_len, H, 64, d_in, K), dev)
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    _check("dust_attn_qk_estimate",
           lib().dust_attn_qk_estimate(which, _ptr(Q), _ptr(Kk), _ptr(V), _ptr(O), _ptr(P),
                                       _ptr(E), _ptr(x), xdt, T, seq_len, H, 64, d_in,
                                       noise(seed, sigma, K, layer, draw0, token0, gamma),
                                       _ptr(g), _ptr(G), _ptr(ws), ws.numel(), _stream(stream)))
    return g, G, ws


# ---------------------------------------------------------------- block ----
class LayerJob:
    """One layer type's perturbed pass for dust_block_estimate: the C job
    plus the tensors it points at (kept alive) and its outputs (g, G)."""

    def __init__(self, jtype, ins, x, T, seq_len, n, nz, want_g, C_out, ema_decay=0.0):
        _need_cuda(*ins, x)
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise ValueError("x must be bf16 or fp32")
        dev = x.device
        d_in = x.shape[1]
        self.tensors = list(ins) + [x]
        self.g = torch.empty((T, C_out), dtype=torch.float32, device=dev) if want_g else None
        self.G = torch.empty((C_out, d_in), dtype=torch.float32, device=dev)
        n = list(n) + [0] * (3 - len(n))
        self.c = DustLayerJob()
        self.c.type = jtype
        for k, t in enumerate(ins):
            self.c.in_[k] = t.data_ptr()
        self.c.x = x.data_ptr()
        self.c.x_dtype = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
        self.c.T, self.c.seq_len, self.c.d_in = T, seq_len, d_in
        self.c.n1, self.c.n2, self.c.n3 = n
        self.c.ema_decay = float(ema_decay)
        self.c.nz = nz
        self.c.g_hat = self.g.data_ptr() if self.g is not None else None
        self.c.G_W = self.G.data_ptr()


def job_head(logits, targets, x, sigma, K, seed, layer=0, draw0=0, token0=0, want_g=True):
    T, V = logits.shape
    return LayerJob(JOB_HEAD, [logits, targets], x, T, T, [V],
                    noise(seed, sigma, K, layer, draw0, token0), want_g, V)


def job_linear(x, y1, W2, ema_decay, W_head, z_clean, targets, seq_len, sigma, gamma, K, seed,
               layer=1, draw0=0, token0=0, want_g=True):
    T, C = y1.shape
    return LayerJob(JOB_LINEAR, [y1, W2, W_head, z_clean, targets], x, T, seq_len,
                    [C, W2.shape[0], W_head.shape[0]],
                    noise(seed, sigma, K, layer, draw0, token0, gamma), want_g, C, ema_decay)


def job_attn_value(P, E, x, seq_len, sigma, gamma, K, seed, layer=2, draw0=0, token0=0,
                   want_g=True):
    T, C = E.shape
    return LayerJob(JOB_ATTN_VALUE, [P, E], x, T, seq_len, [P.shape[1]],
                    noise(seed, sigma, K, layer, draw0, token0, gamma), want_g, C)


def job_attn_gate(z, o, E, x, seq_len, sigma, gamma, K, seed, layer=3, draw0=0, token0=0,
                  want_g=True):
    T, C = z.shape
    return LayerJob(JOB_ATTN_GATE, [z, o, E], x, T, seq_len, [C],
                    noise(seed, sigma, K, layer, draw0, token0, gamma), want_g, C)


def job_attn_qk(which, Q, Kk, V, O, P, E, x, seq_len, sigma, gamma, K, seed, layer=None,
                draw0=0, token0=0, want_g=True):
    if which not in (0, 1):
        raise ValueError("which is 0 (queries) or 1 (keys)")
    T, C = Q.shape
    return LayerJob(JOB_ATTN_KEY if which else JOB_ATTN_QUERY, [Q, Kk, V, O, P, E], x, T,
                    seq_len, [P.shape[1]],
                    noise(seed, sigma, K, 4 + which if layer is None else layer, draw0, token0,
                          gamma), want_g, C)


def _job_array(jobs):
    arr = (DustLayerJob * len(jobs))()
    for k, j in enumerate(jobs):
        arr[k] = j.c
    return arr


def block_workspace_bytes(jobs):
    return lib().dust_block_workspace(_job_array(jobs), len(jobs))


def block_job_offset(jobs, j):
    return lib().dust_block_job_offset(_job_array(jobs), len(jobs), j)


def block_estimate(jobs, streams=None, ws=None):
    """Runs the layer jobs (one perturbed pass each, distinct noise layers)
    through dust_block_estimate, job j on streams[j % len(streams)] (default:
    the current stream).  Returns ([(g or None, G) per job], ws)."""
    arr = _job_array(jobs)
    if ws is None:
        ws = _workspace(lib().dust_block_workspace(arr, len(jobs)), jobs[0].G.device)
    if streams is None:
        streams = [torch.cuda.current_stream()]
    sarr = (_P * len(streams))(*[s.cuda_stream for s in streams])
    _check("dust_block_estimate",
           lib().dust_block_estimate(arr, len(jobs), _ptr(ws), ws.numel(), sarr, len(streams)))
    return [(j.g, j.G) for j in jobs], ws


# ------------------------------------------------------------ data parallel ----
def sum_over_ranks(G, group=None):
    """The one exchange of a data-parallel estimator step: with the sequences of
    a batch sharded across ranks (each rank estimating its own tokens, noise
    keyed by the global token index), the weight gradient is the sum of the
    ranks' G_W, reduced in place by an all-reduce (NCCL between GPUs, gloo on
    CPU).  A no-op without an initialised process group of two or more ranks."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(G, op=dist.ReduceOp.SUM, group=group)
    return G


# ---------------------------------------------------------------- probes ----
PROBE_OPS_PER_ROUND = {0: 16, 1: 8, 2: 8, 3: 16, 4: 16, 5: 16}  # per thread and round


def issue_probe(kind, iters, stream=None):
    """Operations per second of one probe kind (0: Philox multiply/xor,
    1: ex2, 2: fp32 fma, 3 and 4: Philox with split multiplies, 5: packed fp32
    fma, two operations each), timed with events on the stream: (ops/s, ms)."""
    sink = torch.zeros(256, dtype=torch.int32, device="cuda")
    n = _I64(0)
    s = stream if stream is not None else torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    _check("dust_issue_probe", lib().dust_issue_probe(kind, iters, ctypes.byref(n), _ptr(sink),
                                                      ctypes.c_void_p(s.cuda_stream)))
    e1.record(s)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    return n.value * iters * PROBE_OPS_PER_ROUND[kind] / (ms * 1e-3), ms


def head_estimate_chunked(logits, targets, x, sigma, K, seed, chunk, layer=0, draw0=0, token0=0,
                          want_g=True, out=None, ws=None, stream=None):
    """The head with one vocabulary chunk of width `chunk` perturbed per draw
    (draw j perturbs chunk j mod V/chunk).  Returns (g_hat or None, G_W, ws)."""
    _need_cuda(logits, targets, x)
    T, V = logits.shape
    d = x.shape[1]
    dev = logits.device
    if out is None:
        g = torch.empty((T, V), dtype=torch.float32, device=dev) if want_g else None
        G = torch.empty((V, d), dtype=torch.float32, device=dev)
    else:
        g, G = out
    if ws is None:
        ws = _workspace(lib().dust_head_chunked_workspace(T, V, d, K, chunk), dev)
    xdt = DUST_BF16 if x.dtype == torch.bfloat16 else DUST_F32
    _check("dust_head_estimate_chunked",
           lib().dust_head_estimate_chunked(_ptr(logits), _ptr(targets), _ptr(x), xdt, T, V, d,
                                            noise(seed, sigma, K, layer, draw0, token0), chunk,
                                            _ptr(g), _ptr(G), _ptr(ws), ws.numel(),
                                            _stream(stream)))
    return g, G, ws


# ------------------------------------------------------- weight-space ES ----
def es_perturb(theta, sigma, K, seed, layer=9, draw0=0, token0=0, stream=None):
    """K perturbed copies theta + sigma eps_i (K x n) of a small fp32 vector."""
    _need_cuda(theta)
    out = torch.empty((K, theta.numel()), dtype=torch.float32, device=theta.device)
    _check("dust_es_perturb", lib().dust_es_perturb(_ptr(theta), theta.numel(),
                                                    noise(seed, sigma, K, layer, draw0, token0),
                                                    _ptr(out), _stream(stream)))
    return out


def es_estimate(losses, n, sigma, seed, layer=9, draw0=0, token0=0, stream=None):
    """(1/(K sigma)) sum_i (L_i - mean L) eps_i from the K losses of the copies."""
    _need_cuda(losses)
    g = torch.empty(n, dtype=torch.float32, device=losses.device)
    _check("dust_es_estimate", lib().dust_es_estimate(_ptr(losses), n,
                                                      noise(seed, sigma, losses.numel(), layer,
                                                            draw0, token0),
                                                      _ptr(g), _stream(stream)))
    return g

