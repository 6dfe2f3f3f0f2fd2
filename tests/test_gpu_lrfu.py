"""GPU LRFU keep score (ActKV §5.2) against the oracle: hit sets bit for
bit, keep scores within one fp32 rounding, over ragged segments, ties,
zero and dominant scores, several p (0 included) and λ, and a chain of
steps.  The kernel's masses carry about 48 significant bits (fp32 pairs
with their rounding errors), so a segment whose top-p boundary lies within
1e-10 of the total from a prefix mass is counted rather than failed."""
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


def _boundary_margin(s: np.ndarray, p: float) -> float:
    """Distance, relative to the total, between the target p·Σ and the
    nearest prefix mass of the ordered scores (how near the hit/miss
    decision is to a tie)."""
    m = np.where(np.isfinite(s) & (s > 0), s, 0).astype(np.float64)
    tot = m.sum()
    if tot == 0 or p <= 0.0:
        return np.inf  # nothing is asked for: no hits, exactly
    order = np.lexsort((np.arange(len(m)), -m))
    cum = np.concatenate([[0.0], np.cumsum(m[order])])
    if p >= 1.0:
        # the target is the total itself, which both sides form by the same
        # sum as the full prefix: only the prefixes short of it can be near
        cum = cum[:int(np.count_nonzero(m))]
    return float(np.min(np.abs(cum - p * tot)) / tot)


def _segments(rng):
    lens = [1, 7, 32, 33, 500, 6144, 4097, 49152]
    parts = []
    for j, n in enumerate(lens):
        kind = j % 4
        if kind == 0:
            s = rng.random(n).astype(np.float32)
        elif kind == 1:  # few distinct values: ties at the boundary
            s = rng.choice(np.array([0.0, 0.25, 0.5, 1.0], np.float32), n)
        elif kind == 2:  # heavy tail with zeros
            s = (rng.pareto(1.5, n) * (rng.random(n) < 0.7)).astype(np.float32)
        else:            # one dominant entry among small ones
            s = (rng.random(n) * 1e-3).astype(np.float32)
            s[n // 2] = 5.0
        parts.append(s)
    return lens, parts


@pytest.mark.parametrize("p,lam", [(0.9, 0.5), (0.5, 0.0), (1.0, 1.0), (0.9, 0.9), (0.0, 0.5)])
def test_lrfu_matches_oracle(kvc, orc, p, lam):
    p32, lam32 = float(np.float32(p)), float(np.float32(lam))
    rng = np.random.default_rng(int(p * 100) + int(lam * 10))
    lens, parts = _segments(rng)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    n_seg, max_len = len(lens), max(lens)
    words = (max_len + 31) // 32
    ks_ref = [np.zeros(n, np.float32) for n in lens]
    ks_d = torch.zeros(int(off[-1]), dtype=torch.float32, device=DEV)
    off_d = torch.from_numpy(off).to(DEV)
    near = 0
    for step in range(3):
        if step:
            parts = [np.roll(s, 17 * step) * np.float32(1 + step) for s in parts]
        sc = torch.from_numpy(np.concatenate(parts)).to(DEV)
        mask = torch.empty(n_seg, words, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        kvc.kvc_lrfu_update(sc, off_d, n_seg, max_len, p32, lam32, ks_d, mask, st)
        torch.cuda.synchronize()
        assert kvc.kvc_device_status(st) == 0
        got_ks = ks_d.cpu().numpy()
        got_mask = mask.cpu().numpy().view(np.uint32)
        for s_i, n in enumerate(lens):
            ks_ref[s_i], hits = orc.lrfu_update(parts[s_i], ks_ref[s_i], p32, lam32)
            bits = np.array([(got_mask[s_i, i // 32] >> (i % 32)) & 1 for i in range(n)], bool)
            assert not np.any(got_mask[s_i] & ~_pack(np.ones(n, bool), words))  # no bit ≥ n
            if _boundary_margin(parts[s_i], p32) < 1e-10:
                near += 1
                ks_ref[s_i] = got_ks[off[s_i]:off[s_i + 1]].copy()  # follow the GPU on a tie
                continue
            assert np.array_equal(bits, hits), f"segment {s_i} step {step}"
            np.testing.assert_allclose(got_ks[off[s_i]:off[s_i + 1]], ks_ref[s_i],
                                       rtol=2.0 ** -23, atol=0)
            ks_ref[s_i] = got_ks[off[s_i]:off[s_i + 1]].copy()
    print(f"near-tie segments: {near}")


def _pack(b: np.ndarray, words: int) -> np.ndarray:
    out = np.zeros(words, np.uint32)
    for i in np.nonzero(b)[0]:
        out[i // 32] |= np.uint32(1 << (i % 32))
    return out


def test_lrfu_nan_recorded_and_ignored(kvc, orc):
    s = np.array([1.0, np.nan, 2.0, 0.5], np.float32)
    off = torch.tensor([0, 4], dtype=torch.int64, device=DEV)
    ks = torch.zeros(4, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvc.kvc_lrfu_update(torch.from_numpy(s).to(DEV), off, 1, 4, 0.9, 0.5, ks, None, st)
    torch.cuda.synchronize()
    assert kvc.kvc_device_status(st) == 8  # KVC_ERR_NAN
    ref, _ = orc.lrfu_update(s, np.zeros(4), float(np.float32(0.9)), 0.5)
    assert np.array_equal(ks.cpu().numpy(), ref)
