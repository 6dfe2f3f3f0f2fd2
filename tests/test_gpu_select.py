"""GPU select against the oracle on segments built to stress the selection
rule: many equal scores (ties broken by index), signed zeros, forced sink
and recent items, ragged lengths from below the budget up to the longest
segment the call accepts, and the keep mask.  Indices, counts and masks are
compared bit for bit."""
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


def _run(kvc, scores, lens, budget, n_sink, n_recent):
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    n_seg, max_len = len(lens), int(max(lens))
    words = (max_len + 31) // 32
    kept = torch.empty(n_seg, budget, dtype=torch.int32, device=DEV)
    cnt = torch.empty(n_seg, dtype=torch.int32, device=DEV)
    mask = torch.empty(n_seg, words, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_select(torch.from_numpy(scores).to(DEV), torch.from_numpy(off).to(DEV), n_seg,
                   max_len, budget, n_sink, n_recent, kept, cnt, mask, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 0
    return off, kept.cpu().numpy(), cnt.cpu().numpy(), mask.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("budget,n_sink,n_recent", [(256, 1, 4), (64, 0, 0), (512, 3, 9),
                                                     (8192, 0, 0), (20, 10, 10)])
def test_select_ties_ragged_bit_exact(kvc, orc, budget, n_sink, n_recent):
    rng = np.random.default_rng(budget + 7 * n_sink + n_recent)
    lens = [1, budget, budget + 1, 300, 4096, 4097, 9000, 33, 32768, 49152]
    lens = [n for n in lens if n >= 1]
    parts = []
    for j, n in enumerate(lens):
        if j % 3 == 0:   # few distinct values: ties everywhere
            s = rng.integers(0, 6, n).astype(np.float32)
        elif j % 3 == 1:  # signed zeros among a few values
            s = rng.choice(np.array([0.0, -0.0, 1.0, 0.5], np.float32), n)
        else:             # continuous scores with a block of equal ones
            s = rng.random(n).astype(np.float32)
            s[n // 3: n // 3 + min(n, 50)] = s[n // 2]
        parts.append(s)
    scores = np.concatenate(parts)
    off, kept, cnt, mask = _run(kvc, scores, lens, budget, n_sink, n_recent)
    kref, cref, mref = orc.select_segments(scores, off, budget, n_sink, n_recent,
                                           mask_words=mask.shape[1])
    assert np.array_equal(cnt, cref)
    assert np.array_equal(kept, kref)
    assert np.array_equal(mask, mref)


def test_select_all_equal_and_monotone(kvc, orc):
    """All scores equal (the lowest indices win) and strictly increasing
    scores (the latest items win), on 4096-item segments."""
    n, budget = 4096, 256
    scores = np.concatenate([np.full(n, 0.25, np.float32),
                             np.arange(n, dtype=np.float32),
                             -np.arange(n, dtype=np.float32)])
    lens = [n, n, n]
    off, kept, cnt, mask = _run(kvc, scores, lens, budget, 1, 4)
    kref, cref, mref = orc.select_segments(scores, off, budget, 1, 4, mask_words=mask.shape[1])
    assert np.array_equal(kept, kref) and np.array_equal(cnt, cref)
    assert np.array_equal(mask, mref)
    assert kept[0, :5].tolist() == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("n_seg", [3000, 7000])
def test_select_many_segments_bit_exact(kvc, orc, n_seg):
    """Launches with tens of millions of items: the kernel then runs fewer
    threads per segment (32 or 64 items each) to keep more segments in
    flight; the result is the same bits."""
    rng = np.random.default_rng(n_seg)
    lens = rng.integers(1, 8193, n_seg)
    lens[:3] = [8192, 1, 300]
    scores = rng.random(int(lens.sum())).astype(np.float32)
    scores[::7] = 0.5  # ties
    budget, n_sink, n_recent = 256, 1, 4
    off, kept, cnt, mask = _run(kvc, scores, [int(n) for n in lens], budget, n_sink, n_recent)
    kref, cref, mref = orc.select_segments(scores, off, budget, n_sink, n_recent,
                                           mask_words=mask.shape[1])
    assert np.array_equal(cnt, cref)
    assert np.array_equal(kept, kref)
    assert np.array_equal(mask, mref)


@pytest.mark.parametrize("budget,n_sink,n_recent", [(2048, 1, 8), (8192, 0, 0), (512, 3, 9)])
def test_select_long_segments_bit_exact(kvc, orc, budget, n_sink, n_recent):
    """Segments longer than shared memory can stage (the KVMem 10M-token
    workspace is 312,500 blocks per layer and KV head; a 1M-token session at
    token granularity is 1,048,576 items), mixed with short ones in the same
    launch: the streaming path, with ties, signed zeros and blocks of equal
    scores, bit-exact against the oracle (indices, counts, keep masks)."""
    rng = np.random.default_rng(budget + n_sink)
    lens = [312_500, 1_048_576, kvc.SELECT_STAGED_SEG + 1, 300, budget, 70]
    parts = []
    for j, n in enumerate(lens):
        if j == 0:    # continuous scores with blocks of equal values
            s = rng.random(n).astype(np.float32)
            s[1000:1700] = s[5]
            s[n // 2:n // 2 + 4000] = s[n // 3]
        elif j == 1:  # a few values only: ties everywhere, signed zeros
            s = rng.choice(np.array([0.0, -0.0, 1.0, 0.5, 0.25], np.float32), n)
        else:
            s = rng.standard_normal(n).astype(np.float32)
            s[::11] = 0.0
            s[1::11] = -0.0
        parts.append(s)
    scores = np.concatenate(parts)
    off, kept, cnt, mask = _run(kvc, scores, lens, budget, n_sink, n_recent)
    kref, cref, mref = orc.select_segments(scores, off, budget, n_sink, n_recent,
                                           mask_words=mask.shape[1])
    assert np.array_equal(cnt, cref)
    assert np.array_equal(kept, kref)
    assert np.array_equal(mask, mref)


def test_select_streaming_path_equals_staged_path(kvc):
    """The same segments selected through the staged kernel (a launch whose
    longest segment fits shared memory) and the streaming one (the same
    segments plus one longer segment in the launch) give the same bits."""
    rng = np.random.default_rng(5)
    lens = [4096, 30000, 9000, 49152]
    scores = rng.random(sum(lens)).astype(np.float32)
    scores[::13] = 0.75
    _, k1, c1, m1 = _run(kvc, scores, lens, 256, 1, 4)
    long_seg = rng.random(200_000).astype(np.float32)
    _, k2, c2, m2 = _run(kvc, np.concatenate([scores, long_seg]), lens + [200_000], 256, 1, 4)
    assert np.array_equal(k1, k2[:4]) and np.array_equal(c1, c2[:4])
    assert np.array_equal(m1, m2[:4, :m1.shape[1]])
    assert not m2[:4, m1.shape[1]:].any()
