"""The query and key estimators inside attention on the GPU against the fp64
oracle (oracle/attention.py), which re-runs the perturbed softmax attention."""
import numpy as np
import pytest
import torch

from conftest import parity, rel_l2

pytestmark = pytest.mark.gpu

G_TOL, GW_TOL = 1e-4, 5e-3


def _case(orc, nseq, H, L, d_in, seed):
    rng = np.random.default_rng(seed)
    T, C = nseq * L, H * 64
    Q, Kk, V = (rng.standard_normal((T, C)) for _ in range(3))
    E = 0.1 * rng.standard_normal((T, C))
    x = rng.standard_normal((T, d_in))
    P, O = orc.attn_forward(Q, Kk, V, L, H)
    return Q, Kk, V, E, x, P, O


def _dev(*arrays):
    return [torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda() for a in arrays]


# several query tiles and sequences, three heads, the smallest population
# (K = 2), a sequence of three query tiles; queries and keys each.
@pytest.mark.parametrize("which", [0, 1])
@pytest.mark.parametrize("nseq,H,L,d_in,K,gamma", [(2, 2, 128, 32, 8, 0.95),
                                                   (1, 3, 256, 40, 2, 0.99),
                                                   (2, 1, 384, 16, 5, 1.0)])
def test_attn_qk_matches_oracle(dust, orc, which, nseq, H, L, d_in, K, gamma):
    Q, Kk, V, E, x, P, O = _case(orc, nseq, H, L, d_in, seed=L + H + which)
    dQ, dK, dV, dE, dx, dP, dO = _dev(Q, Kk, V, E, x, P, O)
    g, G, ws = dust.attn_qk_estimate(which, dQ, dK, dV, dO, dP, dE, dx, L, 0.02, gamma, K, 77,
                                     draw0=3, token0=50)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_qk_estimate(which, Q, Kk, V, E, x, L, H, 0.02, gamma, K, 77, 4 + which, 3, 50)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


@pytest.mark.parametrize("which", [0, 1])
def test_attn_qk_large_score_shifts(dust, orc, which):
    """sigma 0.6: most score shifts are beyond the short e^x - 1 series'
    range (|x| >= 1/8), so the warps take the expm1f fallback, and the
    perturbed softmax is far from linear in the noise."""
    nseq, H, L, d_in, K = 1, 2, 256, 24, 6
    Q, Kk, V, E, x, P, O = _case(orc, nseq, H, L, d_in, seed=91 + which)
    dQ, dK, dV, dE, dx, dP, dO = _dev(Q, Kk, V, E, x, P, O)
    g, G, ws = dust.attn_qk_estimate(which, dQ, dK, dV, dO, dP, dE, dx, L, 0.6, 0.97, K, 5)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_qk_estimate(which, Q, Kk, V, E, x, L, H, 0.6, 0.97, K, 5, 4 + which)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


@pytest.mark.parametrize("which", [0, 1])
def test_attn_qk_repeats_bit_for_bit(dust, which):
    """The same call four times gives the same bits: 4 sequences of 1024,
    4 heads, K = 16, sigma 0.3 (some warps take the expm1f fallback and some
    do not, so the epilogue warps drift apart in time), the workspace reused."""
    nseq, H, L, d_in, K = 4, 4, 1024, 64, 16
    T, C = nseq * L, H * 64
    gen = torch.Generator(device="cuda").manual_seed(17 + which)
    Q, Kk, V = (torch.randn((T, C), generator=gen, device="cuda") for _ in range(3))
    E = torch.randn((T, C), generator=gen, device="cuda") * 0.1
    x = torch.randn((T, d_in), generator=gen, device="cuda")
    q4, k4, v4 = (t.view(nseq, L, H, 64).transpose(1, 2) for t in (Q, Kk, V))
    s = (q4 @ k4.transpose(-1, -2)) / 8.0
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool, device="cuda"), 1),
                      float("-inf"))
    P = torch.softmax(s, dim=-1).contiguous()
    O = (P @ v4).transpose(1, 2).reshape(T, C).contiguous()
    ws = dust._workspace(dust.lib().dust_attn_qk_workspace(T, L, H, 64, d_in, K), Q.device)
    outs = []
    for _ in range(4):
        g, G, _ = dust.attn_qk_estimate(which, Q, Kk, V, O, P, E, x, L, 0.3, 0.99, K, 99,
                                        ws=ws)
        torch.cuda.synchronize()
        assert dust.workspace_status(ws) == 0
        outs.append((g.clone(), G.clone()))
    for g, G in outs[1:]:
        assert torch.equal(g, outs[0][0]) and torch.equal(G, outs[0][1])


@pytest.mark.parametrize("which", [0, 1])
def test_attn_qk_full_size_first_sequence(dust, orc, which):
    """8 x 2048 tokens, 8 heads of 64, d_in 512 (the bench's shapes) with 4
    draws: sequence 0's rows of g against the oracle run on that sequence
    alone (sequences never exchange credit; the noise is keyed by global
    token), G_W against g^T x in bf16."""
    nseq, H, L, d_in, K = 8, 8, 2048, 512, 4
    T, C = nseq * L, H * 64
    gen = torch.Generator(device="cuda").manual_seed(5 + which)
    Q, Kk, V = (torch.randn((T, C), generator=gen, device="cuda", dtype=torch.float64)
                for _ in range(3))
    E = torch.randn((T, C), generator=gen, device="cuda") * 0.1
    x = torch.randn((T, d_in), generator=gen, device="cuda").to(torch.bfloat16)
    q4, k4, v4 = (t.view(nseq, L, H, 64).transpose(1, 2) for t in (Q, Kk, V))
    s = (q4 @ k4.transpose(-1, -2)) / 8.0
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool, device="cuda"), 1),
                      float("-inf"))
    P = torch.softmax(s, dim=-1)
    del s
    O = (P @ v4).transpose(1, 2).reshape(T, C)
    P = P.float().contiguous()
    O = O.float().contiguous()
    Qf, Kf, Vf = (t.float().contiguous() for t in (Q, Kk, V))
    g, G, ws = dust.attn_qk_estimate(which, Qf, Kf, Vf, O, P, E, x, L, 0.02, 0.99, K, 1234)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_qk_estimate(which, Q[:L].cpu().numpy(), Kk[:L].cpu().numpy(),
                               V[:L].cpu().numpy(), E[:L].cpu().numpy(),
                               x[:L].float().cpu().numpy(), L, H, 0.02, 0.99, K, 1234, 4 + which)
    eg = rel_l2(g[:L].cpu().numpy(), ref["g"])
    assert eg <= G_TOL, eg
    gb = g.to(torch.bfloat16).double()
    eG = rel_l2(G.cpu().numpy(), (gb.T @ x.double()).cpu().numpy())
    assert eG <= 1e-4, eG
    parity(g_seq0=eg, G_W_vs_g_x=eG)


def test_attn_qk_rejects_bad_arguments(dust):
    L = dust.lib()
    assert L.dust_attn_qk_workspace(256, 100, 2, 64, 8, 4) == 0  # seq_len does not divide T
    assert L.dust_attn_qk_workspace(256, 128, 2, 32, 8, 4) == 0  # dv != 64
    assert L.dust_attn_qk_workspace(256, 128, 2, 64, 8, 1) == 0  # one draw
    z = torch.zeros((128, 64), device="cuda")
    P = torch.zeros((1, 1, 128, 128), device="cuda")
    x = torch.zeros((128, 8), device="cuda")
    with pytest.raises(ValueError):
        dust.attn_qk_estimate(2, z, z, z, z, P, z, x, 128, 0.02, 0.9, 4, 1)
    P64 = torch.zeros((2, 1, 64, 64), device="cuda")
    with pytest.raises(dust.DustError):  # seq_len not a multiple of 128
        dust.attn_qk_estimate(0, z, z, z, z, P64, z, x, 64, 0.02, 0.9, 4, 1)
    ws = torch.zeros(L.dust_attn_qk_workspace(128, 128, 1, 64, 8, 4), dtype=torch.uint8,
                     device="cuda")
    from activation_perturbation_es_noise_b300 import DUST_F32, noise, _ptr
    G = torch.zeros((64, 8), device="cuda")
    st = L.dust_attn_qk_estimate(3, _ptr(z), _ptr(z), _ptr(z), _ptr(z), _ptr(P), _ptr(z), _ptr(x),
                                 DUST_F32, 128, 128, 1, 64, 8, noise(1, 0.02, 4, 4), None,
                                 _ptr(G), _ptr(ws), ws.numel(), None)
    assert st != 0  # which must be 0 or 1
