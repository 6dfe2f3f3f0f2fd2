"""kvc_score_static: the scoring entry point for callers that cannot allocate
device memory (a runtime that owns all of HBM after start-up, or a plugin
inside one that gets tensors but no allocator).  It must give the scores of
kvc_score — the entry point that takes a caller workspace — on the same
inputs, call after call, while its scratch lives in the library's fixed
array.  Self-contained: it builds its own inputs, so it passes alone in a
fresh process as well as after the rest of the suite."""
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


def test_static_scratch_scores_match_workspace_scores():
    import query_conditioned_kv_gb300 as kvc

    # the 8B-class head layout and history, on 4 of its layers
    cfg = W.scaled(W.config_8b(), L=4)
    q = cfg.q(DEV)
    meank = torch.empty(cfg.L, cfg.H, cfg.nb_total, cfg.D, dtype=torch.bfloat16, device=DEV)
    for l in range(cfg.L):
        for h in range(cfg.H):
            meank[l, h] = cfg.meank_direct_unit(l, h, 0, DEV)
    blk_off = torch.tensor(cfg.blk_off(), dtype=torch.int64, device=DEV)
    nb_max = max(cfg.nb)
    args = (cfg.L, cfg.H, cfg.Hq, cfg.D, cfg.W, blk_off, cfg.n_sess, cfg.nb_total, nb_max)
    need = kvc.kvc_score_workspace_size(cfg.L, cfg.H, cfg.Hq, cfg.W, cfg.n_sess, nb_max,
                                        cfg.nb_total)
    assert 0 < need <= kvc.SCORE_STATIC_SCRATCH_BYTES

    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ref = torch.empty(cfg.L, cfg.H, cfg.nb_total, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_score(q, meank, ref, *args, ws, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    ref_np = ref.cpu().numpy().reshape(-1)

    for call in range(2):  # two calls in a row share the one scratch array
        out = torch.full_like(ref, -1.0)
        st.zero_()
        kvc.kvc_score_static(q, meank, out, *args, st)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(st) == 0, f"call {call}"
        assert_scores_close(out.cpu().numpy().reshape(-1), ref_np, f"static call {call}")


def test_static_scratch_rejects_sizes_beyond_its_array():
    import query_conditioned_kv_gb300 as kvc

    # 27B-class 1M-token scoring needs far more scratch than the fixed array;
    # the call is refused on the host, before any launch
    L, H, Hq, D, Wn, nb = 64, 8, 48, 128, 32, 32768
    need = kvc.kvc_score_workspace_size(L, H, Hq, Wn, 1, nb, nb)
    assert need > kvc.SCORE_STATIC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.uint8, device=DEV)
    blk_off = torch.tensor([0, nb], dtype=torch.int64, device=DEV)
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_score_static(dummy, dummy, dummy, L, H, Hq, D, Wn, blk_off, 1, nb, nb)
    assert ei.value.code == 5  # KVC_ERR_WORKSPACE
