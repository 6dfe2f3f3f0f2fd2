"""Device-side error reporting: bad indices, bad offsets and NaN scores are
recorded in the caller's status word; nothing out of range is dereferenced
and the context stays usable.  Every case here is bounds-checked by the
kernels before any access (no fault is provoked)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

DEV = "cuda"


@pytest.fixture(scope="module")
def kvc():
    import query_conditioned_kv_gb300 as k
    return k


def test_pack_out_of_range_kept_index(kvc):
    D, n_tok, budget = 128, 32 * 10, 3
    kraw = torch.randn(1, 1, n_tok, D, device=DEV).to(torch.bfloat16)
    vraw = torch.randn(1, 1, n_tok, D, device=DEV).to(torch.bfloat16)
    kept = torch.tensor([[2, 99, 5]], dtype=torch.int32, device=DEV)  # 99 ≥ 10 blocks
    cnt = torch.tensor([3], dtype=torch.int32, device=DEV)
    tok_off = torch.tensor([0, n_tok], dtype=torch.int64, device=DEV)
    tab = torch.empty(32 * budget, D // 2, 2, dtype=torch.float32, device=DEV)
    kvc.kvc_rope_table(tab, 32 * budget, 0, D, 1e6)
    kv = torch.full((1, 1, 1, 32 * budget, D), 7.0, device=DEV).to(torch.bfloat16)
    vv = kv.clone()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_pack_rerope(kraw, vraw, kept, cnt, 1, 1, D, tok_off, 1, n_tok, budget, tab,
                        kv, vv, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 7
    assert torch.all(vv[0, 0, 0, 32:64] == 0) and torch.all(kv[0, 0, 0, 32:64] == 0)
    assert torch.equal(vv[0, 0, 0, 0:32], vraw[0, 0, 64:96])
    assert torch.equal(vv[0, 0, 0, 64:96], vraw[0, 0, 160:192])


def test_select_nan_is_reported_and_ranked_last(kvc):
    s = torch.tensor([0.5, float("nan"), 0.1, 0.2, 0.9, 0.3], device=DEV)
    off = torch.tensor([0, 6], dtype=torch.int64, device=DEV)
    kept = torch.empty(1, 3, dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_select(s, off, 1, 6, 3, 0, 0, kept, cnt, None, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 8
    assert kept.cpu().tolist() == [[0, 4, 5]]


def test_select_bad_segment_offsets(kvc):
    s = torch.rand(100, device=DEV)
    off = torch.tensor([0, 60, 40], dtype=torch.int64, device=DEV)  # decreasing
    kept = torch.empty(2, 4, dtype=torch.int32, device=DEV)
    cnt = torch.empty(2, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_select(s, off, 2, 64, 4, 1, 1, kept, cnt, None, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 7
    assert cnt.cpu().tolist()[1] == 0 and kept.cpu().tolist()[1] == [-1] * 4


@pytest.mark.parametrize("W", [4, 8])  # CUDA-core and tensor-core scorers
def test_score_bad_block_offsets(kvc, W):
    L, H, Hq, D, nb = 1, 1, 2, 64, 8
    q = torch.randn(1, L, Hq, W, D, device=DEV).to(torch.bfloat16)
    mk = torch.randn(L, H, nb, D, device=DEV).to(torch.bfloat16)
    sc = torch.full((L, H, nb), -5.0, device=DEV)
    off = torch.tensor([0, nb + 4], dtype=torch.int64, device=DEV)  # past nb_total
    ws = torch.empty(kvc.kvc_score_workspace_size(L, H, Hq, W, 1, nb, nb) + 256,
                     dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_score(q, mk, sc, L, H, Hq, D, W, off, 1, nb, nb, ws, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 7
    assert torch.all(sc == -5.0)


def test_host_validation_raises_before_launch(kvc):
    s = torch.rand(10, device=DEV)
    off = torch.tensor([0, 10], dtype=torch.int64, device=DEV)
    kept = torch.empty(1, 2, dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_select(s, off, 1, 10, 2, 2, 1, kept, cnt)
    assert ei.value.code == 3
