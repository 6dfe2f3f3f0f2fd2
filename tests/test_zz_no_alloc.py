"""kvc_score_static: the scoring entry point for callers that cannot allocate
device memory (a runtime that owns all of HBM after start-up, or a plugin
inside one that gets tensors but no allocator).  It must give the scores of
kvc_score — the entry point that takes a caller workspace — on the same
inputs, bit for bit (kvc_score is repeatable to the bit), call after call,
while its scratch lives in the library's one fixed array.

The shapes cover a scorer that keeps its partial sums in the scratch (the
CUDA-core scorer, W = 24) and the default tensor-core scorer of the 8B-class
heads; a call that needs more scratch runs before one that needs less, so
leftovers of the first would show in the second.  Self-contained: it builds
its own inputs, so it passes alone in a fresh process as well as after the
rest of the suite."""
from __future__ import annotations

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import workloads as W  # noqa: E402

DEV = "cuda"


def _inputs(cfg):
    q = cfg.q(DEV)
    meank = cfg.meank_direct(DEV)
    blk_off = torch.tensor(cfg.blk_off(), dtype=torch.int64, device=DEV)
    nb_max = max(cfg.nb)
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, blk_off, cfg.n_sess, cfg.nb_total, nb_max)
    return q, meank, args


def _workspace_scores(kvc, cfg, q, meank, args):
    need = kvc.kvc_score_workspace_size(cfg.L, cfg.H, cfg.Hq, cfg.W, cfg.n_sess, args[-1],
                                        cfg.nb_total)
    assert 0 < need <= kvc.SCORE_STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ref = torch.empty(cfg.L, cfg.H, cfg.nb_total, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_score(q, meank, ref, *args, ws, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    return ref, need


# W = 24 is not a tensor-core window, so these run the CUDA-core scorer,
# whose per-split row partials live in the scratch; the first needs more
# scratch than the second
CC_LARGE = W.MeanKConfig(name="static_cc_large", L=2, H=4, Hq=16, D=128, W=24,
                         hist=[32 * 1500, 32 * 700], budget=16, n_sink=1, n_recent=2,
                         L_pack=0, seed=41)
CC_SMALL = W.MeanKConfig(name="static_cc_small", L=1, H=2, Hq=4, D=64, W=24,
                         hist=[32 * 300], budget=16, n_sink=1, n_recent=2, L_pack=0, seed=42)


def test_static_scratch_scores_equal_workspace_scores():
    import query_conditioned_kv_gb300 as kvc

    cases = [CC_LARGE, CC_SMALL, W.scaled(W.config_8b(), L=4)]
    for cfg in cases:
        q, meank, args = _inputs(cfg)
        ref, need = _workspace_scores(kvc, cfg, q, meank, args)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        for call in range(2):  # two calls in a row share the one scratch array
            out = torch.full_like(ref, -1.0)
            st.zero_()
            kvc.kvc_score_static(q, meank, out, *args, st)
            torch.cuda.synchronize()
            assert kvc.kvc_device_status(st) == 0, f"{cfg.name} call {call}"
            assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), \
                f"{cfg.name} call {call}: static-scratch scores differ from kvc_score's"
        del q, meank, ref


def test_static_scratch_rejects_sizes_beyond_its_array():
    import query_conditioned_kv_gb300 as kvc

    # 27B-class 1M-token scoring needs far more scratch than the fixed array;
    # the call is refused on the host, before any launch
    L, H, Hq, D, Wn, nb = 64, 8, 48, 128, 32, 32768
    need = kvc.kvc_score_workspace_size(L, H, Hq, Wn, 1, nb, nb)
    assert need > kvc.SCORE_STATIC_SCRATCH_BYTES
    q = torch.zeros(16, dtype=torch.uint8, device=DEV)
    blk_off = torch.tensor([0, nb], dtype=torch.int64, device=DEV)
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_score_static(q, q, q, L, H, Hq, D, Wn, blk_off, 1, nb, nb)
    assert ei.value.code == 5  # KVC_ERR_WORKSPACE
    # a shape kvc_score refuses is refused with kvc_score's own status first
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_score_static(q, q, q, L, H, Hq, 96, Wn, blk_off, 1, nb, nb)
    assert ei.value.code == 2  # KVC_ERR_SHAPE (head dim)
