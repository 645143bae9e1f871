"""The value-projection estimator inside attention on the GPU against the fp64
oracle (oracle/attention.py)."""
import numpy as np
import pytest
import torch

from conftest import parity, rel_l2, to_dev

pytestmark = pytest.mark.gpu

G_TOL, GW_TOL = 1e-4, 5e-3


def _probs(nseq, H, L, gen, device):
    """Causal softmax of random scores (fp32, rows sum to 1 over keys <= query)."""
    s = torch.randn((nseq, H, L, L), generator=gen, device=device) * 2.0
    s = s.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool, device=device), 1), -1e30)
    return torch.softmax(s, dim=-1).contiguous()


def _case(nseq, H, L, d_in, seed):
    gen = torch.Generator().manual_seed(seed)
    P = _probs(nseq, H, L, gen, "cpu")
    T = nseq * L
    E = torch.randn((T, H * 64), generator=gen) * 0.1
    x = torch.randn((T, d_in), generator=gen)
    return P, E, x


# several query tiles and sequences; a ragged last group of draws (6 = 4 + 2)
# and three heads; a sequence of three query tiles with a 5-draw population.
@pytest.mark.parametrize("nseq,H,L,d_in,K,gamma", [(2, 2, 128, 32, 8, 0.95),
                                                   (1, 3, 256, 40, 6, 0.99),
                                                   (2, 1, 384, 16, 5, 1.0)])
def test_attn_value_matches_oracle(dust, orc, nseq, H, L, d_in, K, gamma):
    P, E, x = _case(nseq, H, L, d_in, seed=L + H)
    g, G, ws = dust.attn_value_estimate(P.cuda(), E.cuda(), x.cuda(), L, 0.02, gamma, K, 1234,
                                        layer=2, draw0=5, token0=40)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_value_estimate(P.numpy(), E.numpy(), x.numpy(), L, 0.02, gamma, K, 1234, 2,
                                  5, 40)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


def test_attn_value_full_size_first_sequence(dust, orc):
    """8 x 2048 tokens, 8 heads of 64, d_in 512 (the bench's shapes) with 4
    draws: sequence 0's rows of g against the oracle run on that sequence
    alone (sequences never exchange credit and the noise is keyed by global
    token)."""
    nseq, H, L, d_in, K = 8, 8, 2048, 512, 4
    gen = torch.Generator(device="cuda").manual_seed(3)
    P = _probs(nseq, H, L, gen, "cuda")
    E = torch.randn((nseq * L, H * 64), generator=gen, device="cuda") * 0.1
    x = torch.randn((nseq * L, d_in), generator=gen, device="cuda").to(torch.bfloat16)
    g, G, ws = dust.attn_value_estimate(P, E, x, L, 0.02, 0.99, K, 1234)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_value_estimate(P[:1].cpu().numpy(), E[:L].cpu().numpy(),
                                  x[:L].float().cpu().numpy(), L, 0.02, 0.99, K, 1234, 2)
    eg = rel_l2(g[:L].cpu().numpy(), ref["g"])
    assert eg <= G_TOL, eg
    gb = g.to(torch.bfloat16).double()
    eG = rel_l2(G.cpu().numpy(), (gb.T @ x.double()).cpu().numpy())
    assert eG <= 1e-4, eG
    parity(g_seq0=eg, G_W_vs_g_x=eG)


def test_attn_value_rejects_unsupported_shapes(dust):
    L = dust.lib()
    assert L.dust_attn_value_workspace(256, 100, 2, 64, 8, 4) == 0  # seq_len does not divide T
    assert L.dust_attn_value_workspace(256, 128, 2, 32, 8, 4) == 0  # dv != 64
    P = torch.zeros((2, 1, 64, 64), device="cuda")
    with pytest.raises(dust.DustError):  # seq_len not a multiple of 128
        dust.attn_value_estimate(P, torch.zeros((128, 64), device="cuda"),
                                 torch.zeros((128, 8), device="cuda"), 64, 0.02, 0.9, 4, 1)


@pytest.mark.parametrize("T,L,C,d_in,K,gamma", [(256, 128, 64, 16, 8, 0.95),
                                                (300, 100, 520, 24, 5, 0.0),
                                                (2048, 1024, 512, 64, 12, 0.99)])
def test_attn_gate_matches_oracle(dust, orc, T, L, C, d_in, K, gamma):
    gen = torch.Generator().manual_seed(T + C)
    z, o, E = (torch.randn((T, C), generator=gen) for _ in range(3))
    x = torch.randn((T, d_in), generator=gen)
    g, G, ws = dust.attn_gate_estimate(z.cuda(), o.cuda(), E.cuda(), x.cuda(), L, 0.05, gamma, K,
                                       1234, layer=3, draw0=2, token0=9)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_gate_estimate(z.numpy(), o.numpy(), E.numpy(), x.numpy(), L, 0.05, gamma, K,
                                 1234, 3, 2, 9)
    eg, eG = rel_l2(g.cpu().numpy(), ref["g"]), rel_l2(G.cpu().numpy(), ref["G"])
    assert eg <= G_TOL and eG <= GW_TOL, (eg, eG)
    parity(g=eg, G_W=eG)


def test_value_embedding_gradient_is_the_value_estimate_scattered(dust, orc):
    """Value embeddings add to the values (v_t = W_v x_t + ve[id_t]), so their
    estimated gradient is the value estimate g scattered into the table by
    token id: the library's two entry points chained, against the oracle's."""
    P, E, x = _case(2, 2, 128, 16, seed=77)
    ids = torch.randint(0, 50, (256,), generator=torch.Generator().manual_seed(1),
                        dtype=torch.int32)
    g, _, _ = dust.attn_value_estimate(P.cuda(), E.cuda(), x.cuda(), 128, 0.02, 0.99, 6, 1234)
    GE, _, ws = dust.embed_scatter(g, ids.cuda(), 50)
    torch.cuda.synchronize()
    assert dust.workspace_status(ws) == 0
    ref = orc.attn_value_estimate(P.numpy(), E.numpy(), x.numpy(), 128, 0.02, 0.99, 6, 1234, 2)
    _, ref_GE = orc.embed_scatter(ref["g"], ids.numpy(), 50)
    e = rel_l2(GE.cpu().numpy(), ref_GE)
    assert e <= G_TOL, e
    parity(G_ve=e)
