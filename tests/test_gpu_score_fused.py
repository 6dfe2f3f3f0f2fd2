"""The single-read tensor-core scorer (4 query heads per KV head, W = 32,
D = 128) against the oracle, over the cluster sizes its heuristic picks
(about four 256-block tiles of a mean-length session per CTA: 1, 2, 4 and 8
CTAs), sessions long enough that a CTA multiplies tiles twice, sessions too
short to give every CTA of the cluster a tile, partial tiles, and several
sessions of very different lengths in one launch.  Scores follow KVMem
"Query-conditioned retrieval" with ActKV §7.1's aggregation; the tolerance is
1e-3 relative (the same bound as every other scorer)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402
from helpers import assert_scores_close  # noqa: E402

DEV = "cuda"


def _cfg(name, hist_blocks, L=1, seed=0):
    return W.MeanKConfig(name=name, L=L, H=2, Hq=8, D=128, W=32,
                         hist=[32 * n for n in hist_blocks], budget=16, n_sink=1,
                         n_recent=2, gamma=W.GAMMA_PLANTED, L_pack=0, seed=seed)


# mean session length in 256-block tiles → CTAs per cluster (4 tiles per CTA;
# 8 when the longest session is 1.5× the mean or more)
CASES = {
    "c1_partial": _cfg("c1", [700 + 37], L=2, seed=21),       # 3 tiles → 1 CTA
    "c2_rec": _cfg("c2", [2048 + 200], seed=22),             # 9 tiles → 2 CTAs, 3 reloads
    "c4": _cfg("c4", [4096 + 300], seed=23),                 # 18 tiles → 4 CTAs, 3 reloads
    "c8_long": _cfg("c8", [16384 + 129], seed=24),           # 65 tiles → 8 CTAs, 7 reloads
    "mixed": _cfg("mx", [12000, 40, 3000, 256, 9000], seed=25),  # spread lengths: 8 tiles/CTA → 2 CTAs
    "c1_long": _cfg("c1l", [1000, 900], seed=26),             # mean 4 tiles → 1 CTA, 2 reloads
    # tile boundaries: 1 block, one short of a tile, exactly one, one over
    "edges": _cfg("ed", [1, 255, 256, 257], L=2, seed=27),   # mean 1 tile → 1 CTA
    # eight CTAs over several sessions; the 300-block one leaves six idle
    "c8_multi": _cfg("c8m", [16384, 16384, 300], seed=28),   # mean 44 tiles → 8 CTAs
}


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


_CACHE = {}


def _case(orc, name):
    if name not in _CACHE:
        cfg = CASES[name]
        q = cfg.q(DEV)
        mk = cfg.meank_direct(DEV)
        boff = cfg.blk_off()
        ref = orc.score_meank(W.bf16_bits(q), W.bf16_bits(mk), cfg.H, boff)
        _CACHE[name] = (cfg, q, mk, torch.from_numpy(np.asarray(boff, np.int64)).to(DEV), ref)
    return _CACHE[name]


def _score(kvc, cfg, q, mk, boff, kernel="auto"):
    nb_max = max(cfg.nb)
    ws_bytes = kvc.kvc_score_workspace_size(cfg.L, cfg.H, cfg.Hq, cfg.W, cfg.n_sess, nb_max,
                                           cfg.nb_total)
    ws = torch.empty(max(1, ws_bytes), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((cfg.L, cfg.H, cfg.nb_total), -1.0, dtype=torch.float32, device=DEV)
    kvc.kvc_score_ex(q, mk, out, cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, boff, cfg.n_sess,
                     cfg.nb_total, nb_max, ws, kernel, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_fused_scores_match_oracle(kvc, orc, name):
    cfg, q, mk, boff, ref = _case(orc, name)
    out = _score(kvc, cfg, q, mk, boff, "score_fused")
    assert_scores_close(out.cpu().numpy().reshape(-1), ref.reshape(-1))


@pytest.mark.parametrize("name", ["c2_rec", "mixed"])
def test_fused_is_the_default_and_deterministic(kvc, orc, name):
    """Without a named kernel the library picks the single-read kernel for
    this shape; two runs give the same bits."""
    cfg, q, mk, boff, _ = _case(orc, name)
    a = _score(kvc, cfg, q, mk, boff)
    b = _score(kvc, cfg, q, mk, boff, "score_fused")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
