"""dust_block_estimate on the GPU: one perturbed pass per layer type of a block
(head, interior linear layer, attention values, gate, queries, keys), spread
over two streams, must give exactly what the single entry points give for the
same inputs and noise (each pass is one of those calls on its own workspace
slice), and every pass must leave its status word clean."""
import numpy as np
import pytest
import torch

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
            "y": torch.from_numpy(li["y"]).cuda(), "seq_len": li["seq_len"]}


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
