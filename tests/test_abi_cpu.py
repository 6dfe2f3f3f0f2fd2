"""The C-ABI library loads and exports every entry point of include/kvc.h;
host-side validation rejects bad arguments before any launch.  CPU only:
no call here reaches a kernel (every call below fails validation first)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        src = f.read()
    for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(kvc_\w+)\s*\(", src, re.M):
        names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def kvc():
    import __graft_entry__
    __graft_entry__.build()
    import query_conditioned_kv_gb300 as k
    return k


def test_header_declares_the_event_calls():
    names = _declared()
    for n in ("kvc_build_meank", "kvc_score", "kvc_select", "kvc_pack_rerope",
              "kvc_redirect_free", "kvc_qmem_update", "kvc_score_qmem",
              "kvc_rope_table", "kvc_init_sentinel", "kvc_status_string",
              "kvc_device_status", "kvc_recover_score", "kvc_tail_plan",
              "kvc_tail_compact"):
        assert n in names


def test_library_exports_every_declared_symbol(kvc):
    lib = ctypes.CDLL(kvc.LIB_PATH)
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(kvc):
    for code in range(0, 13):
        s = kvc.kvc_status_string(code)
        assert s and s != "unknown status"
    assert kvc.kvc_status_string(99) == "unknown status"


def test_workspace_queries(kvc):
    assert kvc.kvc_score_workspace_size(36, 8, 32, 32, 1, 4096, 4096) > 0
    assert kvc.kvc_score_workspace_size(1, 3, 4, 1, 1, 1, 1) == 0  # Hq % H
    assert kvc.kvc_score_qmem_workspace_size(64, 36, 32, 32768) >= 64 * 36 * 32 * 32768 * 4
    assert kvc.kvc_redirect_free_workspace_size(64, 32768, 1839120) >= 1839120 * 4


FAKE = 1 << 20  # a 16-byte-aligned non-NULL address; never dereferenced


def _call(kvc, name, *args):
    return getattr(kvc.lib, name)(*args)


def test_selftest_rejects_a_null_status_word(kvc):
    assert _call(kvc, "kvc_selftest_bounded_wait", None, None) == 1


def test_validation_rejects_before_launch(kvc):
    P, U = FAKE, FAKE + 2  # U: misaligned
    # build_meank: shape (n_tok % 32), head dim, alignment, NULL
    assert _call(kvc, "kvc_build_meank", P, P, 1, 1, 128, 33, None, None) == 2
    assert _call(kvc, "kvc_build_meank", P, P, 1, 1, 96, 64, None, None) == 2
    assert _call(kvc, "kvc_build_meank", U, P, 1, 1, 128, 64, None, None) == 4
    assert _call(kvc, "kvc_build_meank", None, P, 1, 1, 128, 64, None, None) == 1
    # score: Hq % H, too many rows, workspace too small
    assert _call(kvc, "kvc_score", P, P, P, 1, 3, 4, 128, 16, P, 1, 128, 128, P,
                 1 << 20, None, None) == 2
    assert _call(kvc, "kvc_score", P, P, P, 1, 1, 16, 128, 32, P, 1, 128, 128, P,
                 1 << 20, None, None) == 2
    assert _call(kvc, "kvc_score", P, P, P, 1, 2, 4, 64, 16, P, 1, 128, 128, P,
                 8, None, None) == 5
    # select: budget rules and the segment cap
    assert _call(kvc, "kvc_select", P, P, 1, 100, 0, 0, 0, P, P, None, None, None) == 3
    assert _call(kvc, "kvc_select", P, P, 1, 100, 4, 3, 2, P, P, None, None, None) == 3
    assert _call(kvc, "kvc_select", P, P, 1, 100, 4, -1, 0, P, P, None, None, None) == 3
    assert _call(kvc, "kvc_select", P, P, 1, (1 << 30) + 1, 4, 1, 1, P, P, None, None,
                 None) == 2
    # pack: shape, alignment, budget
    assert _call(kvc, "kvc_pack_rerope", P, P, P, P, 1, 1, 128, P, 1, 100, 4, P, P, P,
                 None, None) == 2
    assert _call(kvc, "kvc_pack_rerope", P, U, P, P, 1, 1, 128, P, 1, 128, 4, P, P, P,
                 None, None) == 4
    assert _call(kvc, "kvc_pack_rerope", P, P, P, P, 1, 1, 128, P, 1, 128, 0, P, P, P,
                 None, None) == 3
    # rope table: theta must be > 1
    assert _call(kvc, "kvc_rope_table", P, 16, 0, 128, 0.5, None) == 1
    # sentinel outside the pool
    assert _call(kvc, "kvc_init_sentinel", P, None, 1, 8, 128, 10, 10, None) == 1
    # score_qmem: a GQA group of more than 8 query heads; H not dividing 32
    assert _call(kvc, "kvc_score_qmem", P, P, P, 0, P, 1, 1, 1, 16, 64, 16, 10, P, 1 << 30,
                 None, None) == 2
    assert _call(kvc, "kvc_score_qmem", P, P, P, 0, P, 1, 1, 3, 6, 64, 16, 10, P, 1 << 30,
                 None, None) == 2
    # redirect: workspace too small
    assert _call(kvc, "kvc_redirect_free", P, P, 1, 64, P, 100, 0, 0, P, 100, P, P, 16,
                 None, None) == 5
    # recover: D, Hq % H, a NULL state, misaligned pool
    assert _call(kvc, "kvc_recover_score", P, P, P, 1 << 12, P, 8, P, P, 1, 1, 8, 32, 96, 16,
                 P, None, 0, None, None) == 2
    assert _call(kvc, "kvc_recover_score", P, P, P, 1 << 12, P, 8, P, P, 1, 1, 8, 30, 128, 16,
                 P, None, 0, None, None) == 2
    assert _call(kvc, "kvc_recover_score", P, P, P, 1 << 12, P, 8, P, P, 1, 1, 8, 32, 128, 16,
                 None, None, 0, None, None) == 1
    assert _call(kvc, "kvc_recover_score", P, P, U, 1 << 12, P, 8, P, P, 1, 1, 8, 32, 128, 16,
                 P, None, 0, None, None) == 4
    assert _call(kvc, "kvc_recover_score", P, P, P, 1 << 12, P, 8, P, P, 1, 1, 8, 32, 128, 16,
                 P, U, 1 << 20, None, None) == 4  # misaligned workspace
    # tail plan: a request longer than the plan accepts; no mask
    assert _call(kvc, "kvc_tail_plan", P, 4, P, P, 1 << 17, 1, 16, 1 << 22, P, P, P, P, P, P,
                 P, P, None, None) == 2
    assert _call(kvc, "kvc_tail_plan", None, 4, P, P, 8, 1, 16, 1 << 12, P, P, P, P, P, P,
                 P, P, None, None) == 1
    # compaction: D, misaligned pool, no pair capacity
    assert _call(kvc, "kvc_tail_compact", P, P, 1 << 12, 2, 8, 96, P, P, P, 16, 1, None,
                 None) == 2
    assert _call(kvc, "kvc_tail_compact", P, U, 1 << 12, 2, 8, 128, P, P, P, 16, 1, None,
                 None) == 4
    assert _call(kvc, "kvc_tail_compact", P, P, 1 << 12, 2, 8, 128, P, P, P, 0, 1, None,
                 None) == 1
    # tiered pack: prev lists without their buffers; misaligned history
    assert _call(kvc, "kvc_pack_tiered", P, P, P, None, None, None, P, P, 1, 1, 128, P, 1, 128,
                 4, P, P, P, P, None, None, None) == 1
    assert _call(kvc, "kvc_pack_tiered", U, P, None, None, None, None, P, P, 1, 1, 128, P, 1,
                 128, 4, P, P, P, P, None, None, None) == 4
    # tiered pack from repository slots: no slot table, slots smaller than a
    # block, no slots, a slot stride that breaks 16-byte alignment
    def slots(slot_elems, n_slots, table):
        return _call(kvc, "kvc_pack_tiered_slots", P, P, slot_elems, n_slots, table, None, None,
                     None, None, P, P, 1, 1, 128, P, 1, 128, 4, P, P, P, P, None, None, None)
    assert slots(2 * 32 * 128, 4, None) == 1
    assert slots(32 * 128 - 8, 4, P) == 1
    assert slots(2 * 32 * 128, 0, P) == 1
    assert slots(2 * 32 * 128 + 4, 4, P) == 4
    # LRFU: p or lambda outside [0, 1]; a segment longer than the staging allows
    assert _call(kvc, "kvc_lrfu_update", P, P, 1, 64, ctypes.c_float(1.5), ctypes.c_float(0.5),
                 P, None, None, None) == 1
    assert _call(kvc, "kvc_lrfu_update", P, P, 1, 64, ctypes.c_float(0.9), ctypes.c_float(-0.1),
                 P, None, None, None) == 1
    assert _call(kvc, "kvc_lrfu_update", P, P, 1, 49153, ctypes.c_float(0.9),
                 ctypes.c_float(0.5), P, None, None, None) == 2
    # confidence: top_k beyond the vocabulary; too many windows; misaligned slope
    assert _call(kvc, "kvc_token_confidence", P, 4, 10, 11, P, None, None) == 1
    assert _call(kvc, "kvc_conf_trend_budget", P, P, 1, 100000, 1, 1, ctypes.c_float(10.0),
                 256, 8192, P, P, P, None, None) == 2
    assert _call(kvc, "kvc_conf_trend_budget", P, P, 1, 1000, 16, 4, ctypes.c_float(10.0),
                 256, 8192, FAKE + 4, P, P, None, None) == 4
    assert _call(kvc, "kvc_device_status", None, None) == 1


def test_kernel_choice_is_validated_before_launch(kvc):
    """The _ex entry points take only their own kvc_kernel values; the rest of
    their validation is that of the plain call (no kernel is reached here)."""
    P = FAKE
    # a rule-score kernel named for the Mean-K scorer, an unknown value
    assert _call(kvc, "kvc_score_ex", P, P, P, 1, 2, 4, 64, 16, P, 1, 128, 128, P, 1 << 20,
                 None, kvc.KERNELS["qmem_tc"], None) == 1
    assert _call(kvc, "kvc_score_ex", P, P, P, 1, 2, 4, 64, 16, P, 1, 128, 128, P, 1 << 20,
                 None, 99, None) == 1
    # a valid kernel, but the plain call's shape rule (Hq % H) still applies
    assert _call(kvc, "kvc_score_ex", P, P, P, 1, 3, 4, 128, 16, P, 1, 128, 128, P, 1 << 20,
                 None, kvc.KERNELS["score_ring"], None) == 2
    assert _call(kvc, "kvc_score_qmem_ex", P, P, P, 0, P, 1, 1, 1, 8, 64, 16, 10, P, 1 << 30,
                 None, kvc.KERNELS["score_cc"], None) == 1
    # every rule-score kernel is accepted (the shape rule then answers)
    for name in ("qmem_tc", "qmem_tc_spill", "qmem_cc"):
        assert _call(kvc, "kvc_score_qmem_ex", P, P, P, 0, P, 1, 1, 2, 9, 64, 16, 10, P,
                     1 << 30, None, kvc.KERNELS[name], None) == 2
    assert _call(kvc, "kvc_score_qmem_ex", P, P, P, 0, P, 1, 1, 2, 9, 64, 16, 10, P, 1 << 30,
                 None, 19, None) == 1
    assert _call(kvc, "kvc_recover_score_ex", P, P, P, 1 << 12, P, 8, P, P, 1, 1, 8, 32, 128,
                 16, P, None, 0, None, kvc.KERNELS["qmem_cc"], None) == 1
    with pytest.raises(ValueError):
        kvc._kernel("no_such_kernel")


def test_static_scratch_limit_matches_the_header(kvc):
    """The binding reads the fixed scratch array's size from the library; it
    must be the header's KVC_SCORE_STATIC_SCRATCH_BYTES."""
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        m = re.search(r"#define\s+KVC_SCORE_STATIC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)",
                      f.read())
    assert m, "KVC_SCORE_STATIC_SCRATCH_BYTES not found in kvc.h"
    header = int(m.group(1)) << int(m.group(2))
    assert kvc.kvc_score_static_scratch_bytes() == header == kvc.SCORE_STATIC_SCRATCH_BYTES
    # kvc_score's own checks come before the scratch limit: Hq % H is a shape
    # error even for sizes far beyond the array
    P = FAKE
    assert _call(kvc, "kvc_score_static", P, P, P, 64, 3, 4, 128, 32, P, 1, 32768, 32768,
                 None, None) == 2


def test_recover_tensor_core_coverage(kvc):
    """The page tile of ActKV's Table 1 shapes (block 16, 8 KV heads, d 128)
    runs on the tensor cores; other page shapes take the CUDA-core kernel."""
    assert kvc.kvc_recover_tensor_core(8, 32, 128, 16)
    assert kvc.kvc_recover_tensor_core(8, 64, 64, 16)
    assert not kvc.kvc_recover_tensor_core(4, 16, 128, 16)
    assert not kvc.kvc_recover_tensor_core(8, 24, 128, 16)
    assert not kvc.kvc_recover_tensor_core(8, 32, 128, 32)


def test_binding_raises_on_error(kvc):
    with pytest.raises(kvc.KvcError) as ei:
        kvc._ok(3, "kvc_select")
    assert ei.value.code == 3 and "budget" in str(ei.value)


def test_binding_refuses_strided_tensors(kvc):
    """Every buffer crosses the boundary as a packed row-major pointer, so a
    transposed view must be refused, not read in storage order."""
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="contiguous"):
        kvc._ptr(torch.zeros(4, 6).t())
    # a column-major numpy array keeps its strides through from_numpy
    import numpy as np
    with pytest.raises(ValueError, match="contiguous"):
        kvc._ptr(torch.from_numpy(np.asfortranarray(np.zeros((3, 5), np.int32))))


def test_slot_map_generator_is_row_major():
    import workloads as W
    cfg = W.SlotMapConfig(name="t", n_sess=3, N=1008, prefix=256, page=16, L=1, H=8,
                          Hq=32, D=128, T=4, turns=1, budget=300)
    assert cfg.slot_maps().flags["C_CONTIGUOUS"]
