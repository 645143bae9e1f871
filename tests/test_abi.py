"""The C-ABI library on the host (no GPU): it loads, exports every entry point
include/dust.h declares, sizes workspaces, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import activation_perturbation_es_noise_b300 as dust

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dust.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dust_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    from activation_perturbation_es_noise_b300 import build
    build.build()
    L = dust.lib()
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(dust.EXPORTS) == set(names)


def test_status_strings():
    L = dust.lib()
    for code in range(7):
        assert L.dust_status_string(code)
    assert L.dust_abi_version() == 100


def test_workspace_sizes_monotone():
    a = dust.head_workspace_bytes(256, 512, 64, 64)
    b = dust.head_workspace_bytes(16384, 4096, 512, 64)
    assert 0 < a < b
    assert dust.head_workspace_bytes(0, 512, 64, 64) == 0
    assert dust.head_workspace_bytes(16, 512, 64, 1) == 0
    assert dust.linear_workspace_bytes(16384, 512, 2048, 512, 4096, 256) > 0
    assert dust.embed_workspace_bytes(16384, 1536, 4096) > 0
    assert dust.embed_workspace_bytes(0, 1536, 4096) > 0


def test_bad_arguments_rejected_on_host():
    L = dust.lib()
    nz = dust.noise(1, 0.05, 4)
    fake = ctypes.c_void_p(256)
    # null logits
    assert L.dust_head_estimate(None, fake, fake, 0, 4, 4, 4, nz, None, fake, fake, 1 << 20,
                                None) == 1
    # K < 2
    assert L.dust_head_estimate(fake, fake, fake, 0, 4, 4, 4, dust.noise(1, 0.05, 1), None, fake,
                                fake, 1 << 20, None) == 1
    # workspace too small
    assert L.dust_head_estimate(fake, fake, fake, 0, 4, 4, 4, nz, None, fake, fake, 16,
                                None) == 3
    # V beyond the kernel's register budget
    assert L.dust_head_estimate(fake, fake, fake, 0, 4, 100000, 4, nz, None, fake, fake,
                                1 << 20, None) == 2
    # interior: seq_len must divide T; C must be a multiple of 64
    nzi = dust.noise(1, 0.02, 4, gamma=0.9)
    assert L.dust_linear_estimate(fake, fake, fake, 0.9, fake, fake, fake, 100, 30, 8, 64, 64,
                                  16, nzi, None, fake, fake, 1 << 30, None) == 1
    assert L.dust_linear_estimate(fake, fake, fake, 0.9, fake, fake, fake, 128, 64, 8, 96, 64,
                                  16, nzi, None, fake, fake, 1 << 30, None) == 2
    # gamma outside [0, 1]
    assert L.dust_linear_estimate(fake, fake, fake, 0.9, fake, fake, fake, 128, 64, 8, 64, 64,
                                  16, dust.noise(1, 0.02, 4, gamma=1.5), None, fake, fake,
                                  1 << 30, None) == 1
    # embedding: null output
    assert L.dust_embed_scatter(fake, fake, 4, 4, 4, None, None, fake, 1 << 20, None) == 1
    # philox: negative sizes
    assert L.dust_philox_fill(1, 0, 0, 0, -1, 4, fake, None, None) == 1
    # gemm: misaligned leading dimension
    assert L.dust_gemm_bf16(fake, 0, 7, fake, 0, 8, 4, 4, 4, fake, 4, fake, 256, None) == 1


def test_optimiser_and_backprop_reject_bad_arguments_on_host():
    L = dust.lib()
    f = ctypes.c_void_p(256)
    assert L.dust_sgd_step(None, f, f, 8, 0.1, 0.9, 0.0, None, None) == 1
    assert L.dust_sgd_step(f, f, f, -1, 0.1, 0.9, 0.0, None, None) == 1
    assert L.dust_sgd_step(f, f, f, 8, 0.1, 1.5, 0.0, None, None) == 1
    assert L.dust_sgd_step(f, f, f, 8, float("nan"), 0.9, 0.0, None, None) == 1
    assert L.dust_sgd_step(f, f, f, 8, 0.1, 0.9, -1.0, None, None) == 1
    assert L.dust_sgd_step(f, f, f, 0, 0.1, 0.9, 0.0, None, None) == 0  # n = 0: nothing to do
    adam = lambda **k: L.dust_adam_step(f, f, f, f, k.get("n", 8), 1e-3, k.get("b1", 0.9),
                                        k.get("b2", 0.999), k.get("eps", 1e-8), 0.0,
                                        k.get("step", 1), None, None)
    assert L.dust_sgd_step(None, None, None, 0, 0.1, 0.9, 0.0, None, None) == 0
    assert adam(step=0) == 1
    assert adam(b1=1.0) == 1
    assert adam(b2=-0.1) == 1
    assert adam(eps=0.0) == 1
    assert adam(n=0) == 0
    assert L.dust_head_backprop_workspace(0, 4, 4) == 0
    need = L.dust_head_backprop_workspace(4, 4, 4)
    assert need > 0
    assert L.dust_head_backprop(None, f, f, 0, 4, 4, 4, None, f, f, need, None) == 1
    assert L.dust_head_backprop(f, f, f, 0, 4, 4, 4, None, f, f, need - 1, None) == 3
    assert L.dust_head_backprop(f, f, f, 7, 4, 4, 4, None, f, f, need, None) == 1


def _host_job(jtype, layer, **kw):
    j = dust.DustLayerJob()
    j.type = jtype
    j.nz = dust.noise(1, 0.05, kw.pop("K", 8), layer)
    for k, v in kw.items():
        setattr(j, k, v)
    j.G_W = 256  # never dereferenced: the calls below fail before any launch
    return j


def test_block_workspace_is_the_jobs_slices_in_order():
    L = dust.lib()
    jobs = [_host_job(dust.JOB_HEAD, 0, T=256, seq_len=256, d_in=64, n1=512),
            _host_job(dust.JOB_ATTN_VALUE, 2, T=256, seq_len=128, d_in=32, n1=2),
            _host_job(dust.JOB_ATTN_QUERY, 4, T=256, seq_len=128, d_in=32, n1=2, K=5)]
    arr = (dust.DustLayerJob * 3)(*jobs)
    sizes = [L.dust_head_workspace(256, 512, 64, 8),
             L.dust_attn_value_workspace(256, 128, 2, 64, 32, 8),
             L.dust_attn_qk_workspace(256, 128, 2, 64, 32, 5)]
    assert all(b > 0 for b in sizes)
    up = [(b + 255) // 256 * 256 for b in sizes]
    assert L.dust_block_workspace(arr, 3) == sum(up)
    assert [L.dust_block_job_offset(arr, 3, j) for j in range(3)] == [0, up[0], up[0] + up[1]]
    assert L.dust_block_job_offset(arr, 3, 3) == ctypes.c_size_t(-1).value


def test_block_rejects_bad_jobs_before_any_launch():
    L = dust.lib()
    good = _host_job(dust.JOB_ATTN_GATE, 3, T=256, seq_len=128, d_in=16, n1=64)
    bad_type = _host_job(17, 5, T=256, seq_len=128, d_in=16, n1=64)
    one_draw = _host_job(dust.JOB_ATTN_GATE, 6, T=256, seq_len=128, d_in=16, n1=64, K=1)
    assert L.dust_block_workspace((dust.DustLayerJob * 2)(good, bad_type), 2) == 0
    assert L.dust_block_workspace((dust.DustLayerJob * 1)(one_draw), 1) == 0
    assert L.dust_block_workspace((dust.DustLayerJob * 1)(good), 0) == 0
    ws = ctypes.c_void_p(4096)  # never touched: every case fails on the host
    same_layer = _host_job(dust.JOB_ATTN_VALUE, 3, T=256, seq_len=128, d_in=16, n1=1)
    arr = (dust.DustLayerJob * 2)(good, same_layer)
    assert L.dust_block_estimate(arr, 2, ws, 1 << 30, None, 0) == 1  # INVALID_ARG
    no_out = _host_job(dust.JOB_ATTN_GATE, 3, T=256, seq_len=128, d_in=16, n1=64)
    no_out.G_W = None
    assert L.dust_block_estimate((dust.DustLayerJob * 1)(no_out), 1, ws, 1 << 30, None, 0) == 1
    lin = _host_job(dust.JOB_LINEAR, 8, T=256, seq_len=128, d_in=64, n1=128, n2=64, n3=256)
    assert L.dust_block_workspace((dust.DustLayerJob * 1)(lin), 1) > 0
    lin.x_dtype = dust.DUST_F32  # the interior layer reads x as bf16 only
    assert L.dust_block_estimate((dust.DustLayerJob * 1)(lin), 1, ws, 1 << 30, None, 0) == 1
    assert L.dust_block_estimate((dust.DustLayerJob * 1)(good), 1, None, 0, None, 0) == 3  # WORKSPACE
    assert L.dust_block_estimate((dust.DustLayerJob * 1)(good), 1, ctypes.c_void_p(4100),
                                 1 << 30, None, 0) == 3  # unaligned workspace



def _gate_job(layer, base, sigma=0.05, K=8):
    """A gate job on fake, 16-byte-aligned addresses starting at `base` (never
    dereferenced: every call below must fail on the host)."""
    T, C, d = 256, 64, 16
    j = dust.DustLayerJob()
    j.type = dust.JOB_ATTN_GATE
    j.nz = dust.noise(1, sigma, K, layer)
    j.T, j.seq_len, j.d_in, j.n1 = T, 128, d, C
    step = T * C * 4
    for k in range(3):
        j.in_[k] = base + k * step
    j.x = base + 3 * step
    j.x_dtype = dust.DUST_F32
    j.g_hat = base + 4 * step
    j.G_W = base + 5 * step
    return j


def test_block_checks_every_job_before_queueing_anything():
    """A bad sigma, gamma or missing input in the LAST job is reported as that
    entry point's INVALID_ARG.  Job 0 is valid; had it been queued first, the
    call on this GPU-less host would have failed with DUST_ERR_CUDA instead."""
    L = dust.lib()
    ws = ctypes.c_void_p(1 << 40)
    good = _gate_job(3, 1 << 32)
    for mutate in (lambda j: setattr(j.nz, "sigma", -1.0),
                   lambda j: setattr(j.nz, "gamma", 2.0),
                   lambda j: j.in_.__setitem__(1, None)):
        last = _gate_job(4, 1 << 33)
        mutate(last)
        arr = (dust.DustLayerJob * 2)(good, last)
        assert L.dust_block_estimate(arr, 2, ws, 1 << 30, None, 0) == 1
    # the same two valid jobs get past every check and only then need the GPU
    arr = (dust.DustLayerJob * 2)(good, _gate_job(4, 1 << 33))
    assert L.dust_block_estimate(arr, 2, ws, 1 << 30, None, 0) == 4


def test_block_rejects_jobs_whose_buffers_overlap():
    L = dust.lib()
    ws = ctypes.c_void_p(1 << 40)
    a = _gate_job(3, 1 << 32)
    b = _gate_job(4, 1 << 33)
    b.G_W = a.G_W  # two passes writing one weight gradient
    assert L.dust_block_estimate((dust.DustLayerJob * 2)(a, b), 2, ws, 1 << 30, None, 0) == 1
    b = _gate_job(4, 1 << 33)
    b.g_hat = a.in_[2]  # one pass writing what another reads
    assert L.dust_block_estimate((dust.DustLayerJob * 2)(a, b), 2, ws, 1 << 30, None, 0) == 1
    b = _gate_job(4, 1 << 33)
    b.G_W = (1 << 40) + 512  # an output inside the workspace
    assert L.dust_block_estimate((dust.DustLayerJob * 2)(a, b), 2, ws, 1 << 30, None, 0) == 1
    c = _gate_job(3, 1 << 32)
    c.g_hat = c.G_W  # one pass's two outputs on top of each other
    assert L.dust_block_estimate((dust.DustLayerJob * 1)(c), 1, ws, 1 << 30, None, 0) == 1
