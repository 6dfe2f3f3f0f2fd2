"""The seeded input recipe, checked on the CPU: the configs have the stated
shapes, every unit regenerates alone and repeats bit for bit, and the drawn
values follow the stated distributions (N(0,1) keys and values, a unit
direction planted with +α·u, α ∈ [2, 4], in 3 % of the blocks, queries
N(0,1) + γu).  The generators hold no arithmetic of the method."""
from __future__ import annotations

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import workloads as W  # noqa: E402


def test_configs_have_the_stated_shapes():
    shape = lambda c: (c.L, c.H, c.Hq, c.D, c.n_tok, c.nb_total, c.W, c.budget,  # noqa: E731
                       c.n_sink, c.n_recent, c.lp)
    assert shape(W.config_tiny()) == (1, 2, 4, 64, 4096, 128, 16, 16, 1, 2, 1)
    c8 = W.config_8b()
    assert shape(c8) == (36, 8, 32, 128, 131072, 4096, 32, 256, 1, 4, 36)
    assert c8.view_tokens == 8192 and c8.n_sess == 1
    assert shape(W.config_27b()) == (64, 8, 48, 128, 1048576, 32768, 32, 2048, 1, 8, 16)
    rg = W.config_ragged()
    assert (rg.n_sess, rg.L, rg.lp, rg.budget, rg.n_sink, rg.n_recent) == (128, 36, 2, 512, 1, 4)
    assert all(h % 32 == 0 and 16384 <= h <= 262144 for h in rg.hist)
    assert rg.n_tok == 18286048
    sm = W.config_slotmap()
    assert (sm.n_sess, sm.N, sm.prefix, sm.page, sm.T, sm.turns, sm.budget) == \
        (64, 32768, 4096, 16, 32, 4, 8192)
    assert sm.n_slots - sm.page == 1839104  # unique slots besides the dead slot's page
    for n in (1, 4, 16, 64):
        p = W.config_paged(n)
        assert (p.n_req, p.BS, p.H, p.D, p.L, p.Hq, p.seq, p.keep) == \
            (n, 16, 8, 128, 36, 32, 6144, 4096)


def test_units_regenerate_alone_and_repeat_bit_for_bit():
    c = W.scaled(W.config_ragged(n_sess=3, L_pack=1), L=2, H=2, Hq=8,
                 hist=[64 * 32, 96 * 32, 32 * 32])
    q = c.q()
    assert torch.equal(q[1, 2, 5], c.q_unit(2, 1, 5))
    assert torch.equal(c.q(), q)
    assert not torch.equal(c.q_unit(0, 0, 0), c.q_unit(0, 0, 1))
    k, v = c.kv_raw()
    off = c.tok_off()
    assert torch.equal(k[0, 1, off[1]:off[2]], c.kraw_unit(0, 1, 1))
    assert torch.equal(v[0, 0, off[2]:off[3]], c.vraw_unit(0, 0, 2))
    mk = c.meank_direct()
    boff = c.blk_off()
    assert torch.equal(mk[1, 1, boff[1]:boff[2]], c.meank_direct_unit(1, 1, 1))
    assert torch.all(mk[0] == 0)  # resident layers are built from raw K, not drawn
    sm = W.config_slotmap()
    assert np.array_equal(sm.block_tables(), sm.block_tables())


def test_planted_blocks_and_value_distributions():
    c = W.config_8b()
    blocks, alpha = c.planted(3, 5, 0)
    assert len(blocks) == round(0.03 * 4096)
    assert np.all(np.diff(blocks) > 0) and blocks[0] >= 0 and blocks[-1] < 4096
    assert np.all((alpha >= 2.0) & (alpha <= 4.0))
    u = c.direction(3, 5)
    assert abs(float(np.linalg.norm(u)) - 1.0) < 1e-6
    k = c.kraw_unit(3, 5, 0).float().numpy()
    # per block, the mean key projected on u is α (planted) or 0 (not), with
    # N(0, 1/32) noise from the 32 N(0,1) tokens
    proj = k.reshape(4096, 32, 128).mean(axis=1) @ u
    planted = np.zeros(4096, bool)
    planted[blocks] = True
    assert np.max(np.abs(proj[planted] - alpha)) < 1.0
    assert np.max(np.abs(proj[~planted])) < 1.0
    rest = k.reshape(4096, 32, 128)[~planted]
    assert abs(float(rest.mean())) < 0.01 and abs(float(rest.std()) - 1.0) < 0.01
    # queries: N(0,1) + γu per token, γ the calibrated strength
    qh = c.q_unit(0, 3, 5 * c.G + 2).float().numpy()
    assert abs(float((qh @ u).mean()) - W.GAMMA_PLANTED) < 1.0
    qr = qh - np.outer(qh @ u, u)
    assert abs(float(qr.std()) - 1.0) < 0.05
    # Mean-K drawn directly: N(0, 1/32) off the planted blocks
    mk = c.meank_direct_unit(3, 5, 0).float().numpy()
    assert abs(float(mk[~planted].std()) - 1.0 / math.sqrt(32)) < 0.005
