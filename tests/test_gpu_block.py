"""dust_block_estimate on the GPU: one perturbed pass per layer type of a block
(head, interior linear layer, attention values, gate, queries, keys), spread
over two streams.  Every pass must match the oracle's estimator for its layer
type (g rel-L2 <= 1e-4, G_W <= 5e-3), give exactly what the single entry
point gives for the same inputs and noise (each pass is one of those calls on
its own workspace slice), and leave its status word clean.  A bad job anywhere
in the list stops the call before anything is queued."""
import numpy as np
import pytest
import torch

from conftest import parity, rel_l2
from test_gpu_interior import _inputs as _linear_inputs

pytestmark = pytest.mark.gpu


def _block_inputs(orc, seed=0):
    rng = np.random.default_rng(seed)
    L, nseq, H = 128, 2, 2
    T, C = nseq * L, H * 64
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    Q, Kk, V = (rng.standard_normal((T, C)) for _ in range(3))
    P, O = orc.attn_forward(Q, Kk, V, L, H)
    d = {"L": L, "T": T, "C": C, "H": H,
         "Q": f(Q), "Kk": f(Kk), "V": f(V), "P": f(P), "O": f(O),
         "E": f(0.1 * rng.standard_normal((T, C))),
         "z": f(rng.standard_normal((T, C))), "o": f(rng.standard_normal((T, C))),
         "x": f(rng.standard_normal((T, 40))),
         "logits": f(rng.standard_normal((T, 300))),
         "targets": torch.from_numpy(rng.integers(0, 300, T).astype(np.int32)).cuda(),
         "xh": f(rng.standard_normal((T, 48)))}
    return d


def _linear(d):
    li = _linear_inputs(256, 64, 128, 64, 256, 128, seed=5)
    bf = torch.bfloat16
    return {"x": torch.from_numpy(li["x"]).cuda().to(bf), "y1": torch.from_numpy(li["y1"]).cuda(),
            "W2": torch.from_numpy(li["W2"]).cuda().to(bf), "lam": li["lam"],
            "WH": torch.from_numpy(li["WH"]).cuda().to(bf), "z": torch.from_numpy(li["z"]).cuda(),
            "y": torch.from_numpy(li["y"]).cuda(), "seq_len": li["seq_len"], "host": li}


def test_block_matches_single_calls_on_two_streams(dust, orc):
    d = _block_inputs(orc)
    li = _linear(d)
    L, sig, K, seed = d["L"], 0.02, 6, 99
    jobs = [
        dust.job_head(d["logits"], d["targets"], d["xh"], 0.05, K, seed, layer=0),
        dust.job_linear(li["x"], li["y1"], li["W2"], li["lam"], li["WH"], li["z"], li["y"],
                        li["seq_len"], sig, 0.95, K, seed, layer=1),
        dust.job_attn_value(d["P"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=2),
        dust.job_attn_gate(d["z"], d["o"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=3),
        dust.job_attn_qk(0, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                         0.99, K, seed),
        dust.job_attn_qk(1, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                         0.99, K, seed),
    ]
    side = torch.cuda.Stream()
    outs, ws = dust.block_estimate(jobs, streams=[torch.cuda.current_stream(), side])
    torch.cuda.synchronize()
    for j in range(len(jobs)):
        off = dust.block_job_offset(jobs, j)
        assert dust.workspace_status(ws[off:]) == 0, j

    singles = [
        dust.head_estimate(d["logits"], d["targets"], d["xh"], 0.05, K, seed, layer=0),
        dust.linear_estimate(li["x"], li["y1"], li["W2"], li["lam"], li["WH"], li["z"], li["y"],
                             li["seq_len"], sig, 0.95, K, seed, layer=1),
        dust.attn_value_estimate(d["P"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=2),
        dust.attn_gate_estimate(d["z"], d["o"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=3),
        dust.attn_qk_estimate(0, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                              0.99, K, seed),
        dust.attn_qk_estimate(1, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                              0.99, K, seed),
    ]
    torch.cuda.synchronize()
    for j, ((g, G), (g1, G1, _)) in enumerate(zip(outs, singles)):
        assert torch.equal(g, g1), j
        assert torch.equal(G, G1), j


def test_block_rejects_shared_noise_layers(dust, orc):
    d = _block_inputs(orc, seed=1)
    L = d["L"]
    jobs = [dust.job_attn_value(d["P"], d["E"], d["x"], L, 0.02, 0.9, 4, 1, layer=7),
            dust.job_attn_gate(d["z"], d["o"], d["E"], d["x"], L, 0.02, 0.9, 4, 1, layer=7)]
    with pytest.raises(dust.DustError):
        dust.block_estimate(jobs)


def _block_jobs(dust, d, li, K, seed, sig):
    L = d["L"]
    return [
        dust.job_head(d["logits"], d["targets"], d["xh"], 0.05, K, seed, layer=0),
        dust.job_linear(li["x"], li["y1"], li["W2"], li["lam"], li["WH"], li["z"], li["y"],
                        li["seq_len"], sig, 0.95, K, seed, layer=1),
        dust.job_attn_value(d["P"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=2),
        dust.job_attn_gate(d["z"], d["o"], d["E"], d["x"], L, sig, 0.99, K, seed, layer=3),
        dust.job_attn_qk(0, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                         0.99, K, seed),
        dust.job_attn_qk(1, d["Q"], d["Kk"], d["V"], d["O"], d["P"], d["E"], d["x"], L, sig,
                         0.99, K, seed),
    ]


def test_block_jobs_match_the_oracle(dust, orc):
    """Each pass of a block run on two streams against the oracle's estimator
    of its layer type on the block's own inputs and noise layer."""
    d = _block_inputs(orc, seed=2)
    li = _linear(d)
    L, H, sig, K, seed = d["L"], d["H"], 0.02, 6, 31
    jobs = _block_jobs(dust, d, li, K, seed, sig)
    side = torch.cuda.Stream()
    outs, ws = dust.block_estimate(jobs, streams=[torch.cuda.current_stream(), side])
    torch.cuda.synchronize()
    h = lambda t: t.cpu().numpy()
    hl = li["host"]
    refs = [
        orc.head_estimate(h(d["logits"]), h(d["targets"]), h(d["xh"]), 0.05, K, seed, 0),
        orc.linear_estimate(hl["x"], hl["y1"], hl["W2"], hl["lam"], hl["WH"], hl["z"], hl["y"],
                            hl["seq_len"], sig, 0.95, K, seed, 1),
        orc.attn_value_estimate(h(d["P"]), h(d["E"]), h(d["x"]), L, sig, 0.99, K, seed, 2),
        orc.attn_gate_estimate(h(d["z"]), h(d["o"]), h(d["E"]), h(d["x"]), L, sig, 0.99, K, seed,
                               3),
        orc.attn_qk_estimate(0, h(d["Q"]), h(d["Kk"]), h(d["V"]), h(d["E"]), h(d["x"]), L, H, sig,
                             0.99, K, seed, 4),
        orc.attn_qk_estimate(1, h(d["Q"]), h(d["Kk"]), h(d["V"]), h(d["E"]), h(d["x"]), L, H, sig,
                             0.99, K, seed, 5),
    ]
    names = ["head", "linear", "value", "gate", "query", "key"]
    errs = {}
    for j, ((g, G), ref) in enumerate(zip(outs, refs)):
        assert dust.workspace_status(ws[dust.block_job_offset(jobs, j):]) == 0, j
        eg, eG = rel_l2(h(g), ref["g"]), rel_l2(h(G), ref["G"])
        assert eg <= 1e-4, (names[j], eg)
        assert eG <= 5e-3, (names[j], eG)
        errs["g_" + names[j]] = eg
        errs["G_" + names[j]] = eG
    parity(**errs)


def test_block_bad_last_job_queues_nothing(dust, orc):
    """An invalid sigma in the last job is reported before any pass is queued:
    every output keeps the sentinel it held before the call."""
    d = _block_inputs(orc, seed=4)
    li = _linear(d)
    jobs = _block_jobs(dust, d, li, 4, 8, 0.02)
    for j in jobs:
        j.G.fill_(float("nan"))
        if j.g is not None:
            j.g.fill_(float("nan"))
    jobs[-1].c.nz.sigma = -1.0
    side = torch.cuda.Stream()
    with pytest.raises(dust.DustError):
        dust.block_estimate(jobs, streams=[torch.cuda.current_stream(), side])
    torch.cuda.synchronize()
    for j in jobs:
        assert torch.isnan(j.G).all()
        assert j.g is None or torch.isnan(j.g).all()
