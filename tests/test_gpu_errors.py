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


# CUDA-core scorer (W = 4), two-pass tensor-core scorer (W = 8) and the
# single-read one (4 query heads per KV head, W = 32, D = 128)
@pytest.mark.parametrize("W,Hq,D", [(4, 2, 64), (8, 2, 64), (32, 4, 128)])
def test_score_bad_block_offsets(kvc, W, Hq, D):
    L, H, nb = 1, 1, 8
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


def test_score_bad_session_leaves_the_others_scored(kvc):
    """Single-read scorer: a session whose offsets run past the index is
    reported (KVC_ERR_BOUNDS) and left unwritten; the other session of the
    same launch is scored as usual."""
    L, H, Hq, D, W, nb = 2, 2, 8, 128, 32, 600
    q = torch.randn(L, 2, Hq, W, D, device=DEV).to(torch.bfloat16)
    mk = (torch.randn(L, H, nb, D, device=DEV) * 0.2).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(kvc.kvc_score_workspace_size(L, H, Hq, W, 2, 500, nb) + 256,
                     dtype=torch.uint8, device=DEV)
    good = torch.tensor([0, 400, 600], dtype=torch.int64, device=DEV)
    ref = torch.full((L, H, nb), -5.0, device=DEV)
    kvc.kvc_score(q, mk, ref, L, H, Hq, D, W, good, 2, nb, 400, ws, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    bad = torch.tensor([0, 400, 900], dtype=torch.int64, device=DEV)  # session 1 past nb_total
    sc = torch.full((L, H, nb), -5.0, device=DEV)
    kvc.kvc_score(q, mk, sc, L, H, Hq, D, W, bad, 2, nb, 500, ws, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 7
    assert torch.all(sc[:, :, 400:] == -5.0)
    # same mean session length, so the same cluster size: session 0 has the same bits
    assert torch.equal(sc[:, :, :400].view(torch.int32), ref[:, :, :400].view(torch.int32))


def test_host_validation_raises_before_launch(kvc):
    s = torch.rand(10, device=DEV)
    off = torch.tensor([0, 10], dtype=torch.int64, device=DEV)
    kept = torch.empty(1, 2, dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    with pytest.raises(kvc.KvcError) as ei:
        kvc.kvc_select(s, off, 1, 10, 2, 2, 1, kept, cnt)
    assert ei.value.code == 3


def test_bounded_wait_gives_up_and_the_context_stays_usable(kvc):
    """A wait that nothing completes ends after about a second with
    KVC_ERR_TIMEOUT in the status word (no fault, no trap), and the next
    kernels run normally."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvc.kvc_selftest_bounded_wait(st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert kvc.kvc_device_status(st) == 9  # KVC_ERR_TIMEOUT
    assert 0.9 < dt < 30.0
    s = torch.tensor([0.5, 0.1, 0.2, 0.9, 0.3], device=DEV)
    off = torch.tensor([0, 5], dtype=torch.int64, device=DEV)
    kept = torch.empty(1, 3, dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_select(s, off, 1, 5, 3, 0, 0, kept, cnt, None, st2)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st2) == 0
    assert kept.cpu().tolist() == [[0, 3, 4]] and cnt.cpu().tolist() == [3]
