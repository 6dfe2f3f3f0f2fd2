"""query_conditioned_kv_gb300 — Python binding of libkvc (sm_103a).

A thin ctypes layer over the C ABI declared in ``include/kvc.h``: every
function here has the name of the C entry point it calls and only marshals
arguments (tensor → device pointer, current torch stream → cudaStream_t).
Every step of the compression event runs in the library's CUDA kernels;
there is no Python or CPU fallback.  PyTorch is used for device memory and
streams only.

Importing this package loads ``libkvc.so`` and fails loudly if it has not
been built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "KvcError", "lib", "BLOCK_TOKENS", "SENTINEL_K_BITS", "SELECT_MAX_SEG", "SELECT_STAGED_SEG",
    "LRFU_MAX_SEG",
    "kvc_status_string", "kvc_version", "kvc_device_status", "kvc_selftest_bounded_wait",
    "kvc_build_meank", "kvc_score_workspace_size", "kvc_score_launches", "kvc_score",
    "kvc_score_ex", "kvc_score_static", "kvc_score_static_scratch_bytes",
    "SCORE_STATIC_SCRATCH_BYTES", "KERNELS",
    "kvc_qmem_update", "kvc_score_qmem_workspace_size", "kvc_score_qmem", "kvc_score_qmem_ex",
    "kvc_select", "kvc_rope_table", "kvc_pack_rerope", "kvc_pack_tiered", "kvc_init_sentinel",
    "kvc_redirect_free_workspace_size", "kvc_redirect_free",
    "kvc_recover_score", "kvc_recover_score_ex", "kvc_recover_score_workspace_size",
    "kvc_recover_tensor_core", "kvc_tail_plan", "kvc_tail_compact",
    "kvc_lrfu_update", "kvc_token_confidence", "kvc_conf_trend_budget",
    "TAIL_MAX_TOKENS",
    "kvc_pack_tiered_slots", "kvc_repo_plan", "KvcRepo",
]

BLOCK_TOKENS = 32
SENTINEL_K_BITS = 0xC61C
SELECT_STAGED_SEG = 49152
SELECT_MAX_SEG = 1 << 30
LRFU_MAX_SEG = 49152
SCORE_MAX_ROWS = 256
TAIL_MAX_TOKENS = 1 << 20

# kvc_kernel values (include/kvc.h): the kernel an _ex entry point runs
KERNELS = {
    "auto": 0,
    "score_fused": 1, "score_ring": 2, "score_persist": 3, "score_split": 4, "score_cc": 5,
    "score_group": 6,
    "qmem_tc": 16, "qmem_cc": 17, "qmem_tc_spill": 18,
    "recover_tc": 32, "recover_cc": 33,
}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: the CUDA library must be built first "
        "(python -c 'import __graft_entry__ as g; g.build()'); there is no "
        "fallback path")

_c = ctypes
_P = _c.c_void_p
_I32 = _c.c_int32
_I64 = _c.c_int64
_SZ = _c.c_size_t

lib = _c.CDLL(LIB_PATH)

_SIGS = {
    "kvc_status_string": (_c.c_char_p, [_c.c_int]),
    "kvc_version": (_c.c_char_p, []),
    "kvc_device_status": (_c.c_int, [_P, _P]),
    "kvc_selftest_bounded_wait": (_c.c_int, [_P, _P]),
    "kvc_build_meank": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I64, _P, _P]),
    "kvc_score_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I64]),
    "kvc_score_launches": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "kvc_score_static": (_c.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P,
                                    _I32, _I64, _I32, _P, _P]),
    "kvc_score": (_c.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P,
                             _I32, _I64, _I32, _P, _SZ, _P, _P]),
    "kvc_score_ex": (_c.c_int, [_P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P,
                                _I32, _I64, _I32, _P, _SZ, _P, _c.c_int, _P]),
    "kvc_score_static_scratch_bytes": (_SZ, []),
    "kvc_qmem_update": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32,
                                   _c.c_float, _c.c_float, _I32, _P]),
    "kvc_score_qmem_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "kvc_score_qmem": (_c.c_int, [_P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                  _I32, _I32, _I32, _I64, _P, _SZ, _P, _P]),
    "kvc_score_qmem_ex": (_c.c_int, [_P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                     _I32, _I32, _I32, _I64, _P, _SZ, _P, _c.c_int, _P]),
    "kvc_select": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P,
                              _P, _P, _P]),
    "kvc_rope_table": (_c.c_int, [_P, _I32, _I32, _I32, _c.c_double, _P]),
    "kvc_pack_rerope": (_c.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _P, _I32,
                                   _I64, _I32, _P, _P, _P, _P, _P]),
    "kvc_pack_tiered": (_c.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P,
                                   _I32, _I64, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "kvc_pack_tiered_slots": (_c.c_int, [_P, _P, _I64, _I32, _P, _P, _P, _P, _P, _P, _P,
                                         _I32, _I32, _I32, _P, _I32, _I64, _I32, _P, _P, _P,
                                         _P, _P, _P, _P]),
    "kvc_repo_create": (_c.c_int, [_c.c_char_p, _I64, _I32, _I32, _I32, _I32, _P, _I32, _I32,
                                   _c.POINTER(_c.c_void_p)]),
    "kvc_repo_put": (_c.c_int, [_P, _I64, _I64, _P, _P, _I64]),
    "kvc_repo_plan": (_c.c_int, [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _I64, _P, _P,
                                 _P, _P]),
    "kvc_repo_step": (_c.c_int, [_P, _P, _I64, _P, _I64, _P]),
    "kvc_repo_where": (_I32, [_P, _I64]),
    "kvc_repo_slots": (_c.c_int, [_P, _P]),
    "kvc_repo_changes": (_I64, [_P, _P, _P, _I64]),
    "kvc_repo_get_stats": (_c.c_int, [_P, _P]),
    "kvc_repo_destroy": (None, [_P]),
    "kvc_init_sentinel": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I64, _I32,
                                     _P]),
    "kvc_redirect_free_workspace_size": (_SZ, [_I32, _I32, _I64]),
    "kvc_redirect_free": (_c.c_int, [_P, _P, _I32, _I32, _P, _I64, _I32, _I32,
                                     _P, _I32, _P, _P, _SZ, _P, _P]),
    "kvc_recover_score_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "kvc_recover_score": (_c.c_int, [_P, _P, _P, _I64, _P, _I32, _P, _P, _I32,
                                     _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "kvc_recover_score_ex": (_c.c_int, [_P, _P, _P, _I64, _P, _I32, _P, _P, _I32,
                                        _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P,
                                        _c.c_int, _P]),
    "kvc_recover_tensor_core": (_I32, [_I32, _I32, _I32, _I32]),
    "kvc_token_confidence": (_c.c_int, [_P, _I32, _I32, _I32, _P, _P, _P]),
    "kvc_conf_trend_budget": (_c.c_int, [_P, _P, _I32, _I32, _I32, _I32, _c.c_float, _I32,
                                         _I32, _P, _P, _P, _P, _P]),
    "kvc_lrfu_update": (_c.c_int, [_P, _P, _I32, _I32, _c.c_float, _c.c_float, _P, _P, _P,
                                   _P]),
    "kvc_tail_plan": (_c.c_int, [_P, _I32, _P, _P, _I32, _I32, _I32, _I64, _P, _P,
                                 _P, _P, _P, _P, _P, _P, _P, _P]),
    "kvc_tail_compact": (_c.c_int, [_P, _P, _I64, _I32, _I32, _I32, _P, _P, _P,
                                    _I32, _I32, _P, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


SCORE_STATIC_SCRATCH_BYTES = int(lib.kvc_score_static_scratch_bytes())


def _kernel(name) -> int:
    if isinstance(name, int):
        return name
    try:
        return KERNELS[name]
    except KeyError:
        raise ValueError(f"unknown kernel {name!r}; one of {sorted(KERNELS)}") from None


class KvcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {kvc_status_string(code)} (status {code})")


def kvc_status_string(code: int) -> str:
    return lib.kvc_status_string(int(code)).decode()


def kvc_version() -> str:
    return lib.kvc_version().decode()


def _ptr(t):
    """Device pointer of a dense row-major CUDA tensor (None → NULL).  The
    library indexes every buffer as packed row-major, so a strided view
    (a transpose, a Fortran-ordered array brought over from numpy) is
    refused rather than read in the wrong order."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous row-major tensors only "
                         f"(got shape {tuple(t.shape)}, strides {t.stride()})")
    if not t.is_cuda:
        raise ValueError("libkvc takes device tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ok(code: int, where: str) -> None:
    if code != 0:
        raise KvcError(code, where)


def kvc_device_status(dev_status) -> int:
    """Synchronously reads the device status word (0 = no device error)."""
    out = _c.c_int32(0)
    _ok(lib.kvc_device_status(_ptr(dev_status), _c.addressof(out)),
        "kvc_device_status")
    return int(out.value)


def kvc_selftest_bounded_wait(dev_status, stream=None):
    _ok(lib.kvc_selftest_bounded_wait(_ptr(dev_status), _stream(stream)),
        "kvc_selftest_bounded_wait")


def kvc_build_meank(kraw, meank, L, H, D, n_tok, dev_status=None, stream=None):
    _ok(lib.kvc_build_meank(_ptr(kraw), _ptr(meank), L, H, D, n_tok,
                            _ptr(dev_status), _stream(stream)), "kvc_build_meank")


def kvc_score_workspace_size(L, H, Hq, W, n_sess, nb_max, nb_total) -> int:
    return int(lib.kvc_score_workspace_size(L, H, Hq, W, n_sess, nb_max, nb_total))


def kvc_score_launches(L, H, Hq, D, W, n_sess, nb_max) -> int:
    return int(lib.kvc_score_launches(L, H, Hq, D, W, n_sess, nb_max))


def kvc_score(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total,
              nb_max, ws, dev_status=None, stream=None):
    _ok(lib.kvc_score(_ptr(q), _ptr(meank), _ptr(scores), L, H, Hq, D, W,
                      _ptr(blk_off), n_sess, nb_total, nb_max, _ptr(ws),
                      ws.numel() * ws.element_size(), _ptr(dev_status),
                      _stream(stream)), "kvc_score")


def kvc_score_ex(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total,
                 nb_max, ws, kernel="auto", dev_status=None, stream=None):
    """kvc_score with a named kernel (a KERNELS key or value)."""
    _ok(lib.kvc_score_ex(_ptr(q), _ptr(meank), _ptr(scores), L, H, Hq, D, W,
                         _ptr(blk_off), n_sess, nb_total, nb_max, _ptr(ws),
                         ws.numel() * ws.element_size(), _ptr(dev_status), _kernel(kernel),
                         _stream(stream)), "kvc_score_ex")


def kvc_score_static_scratch_bytes() -> int:
    return int(lib.kvc_score_static_scratch_bytes())


def kvc_score_static(q, meank, scores, L, H, Hq, D, W, blk_off, n_sess, nb_total,
                     nb_max, dev_status=None, stream=None):
    """kvc_score with the library's fixed scratch array instead of a caller
    workspace, for callers that cannot allocate device memory."""
    _ok(lib.kvc_score_static(_ptr(q), _ptr(meank), _ptr(scores), L, H, Hq, D, W,
                             _ptr(blk_off), n_sess, nb_total, nb_max, _ptr(dev_status),
                             _stream(stream)), "kvc_score_static")


def kvc_qmem_update(M, q_turn, n_sess, L, Hq, D, T, decay=0.9, gain=0.1,
                    renorm=1, stream=None):
    _ok(lib.kvc_qmem_update(_ptr(M), _ptr(q_turn), n_sess, L, Hq, D, T,
                            float(decay), float(gain), int(renorm),
                            _stream(stream)), "kvc_qmem_update")


def kvc_score_qmem_workspace_size(n_sess, L, Hq, N) -> int:
    return int(lib.kvc_score_qmem_workspace_size(n_sess, L, Hq, N))


def kvc_score_qmem(M, kpool, slot_map, sentinel, rule, n_sess, L, H, Hq, D, N,
                   n_slots, ws, dev_status=None, stream=None):
    _ok(lib.kvc_score_qmem(_ptr(M), _ptr(kpool), _ptr(slot_map), sentinel,
                           _ptr(rule), n_sess, L, H, Hq, D, N, n_slots,
                           _ptr(ws), ws.numel() * ws.element_size(),
                           _ptr(dev_status), _stream(stream)), "kvc_score_qmem")


def kvc_score_qmem_ex(M, kpool, slot_map, sentinel, rule, n_sess, L, H, Hq, D, N,
                      n_slots, ws, kernel="auto", dev_status=None, stream=None):
    """kvc_score_qmem with a named logits kernel (a KERNELS key or value)."""
    _ok(lib.kvc_score_qmem_ex(_ptr(M), _ptr(kpool), _ptr(slot_map), sentinel,
                              _ptr(rule), n_sess, L, H, Hq, D, N, n_slots,
                              _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(dev_status), _kernel(kernel), _stream(stream)),
        "kvc_score_qmem_ex")


def kvc_select(scores, seg_off, n_seg, max_seg_len, budget, n_sink, n_recent,
               kept, kept_count, keepmask=None, dev_status=None, stream=None):
    _ok(lib.kvc_select(_ptr(scores), _ptr(seg_off), n_seg, max_seg_len, budget,
                       n_sink, n_recent, _ptr(kept), _ptr(kept_count),
                       _ptr(keepmask), _ptr(dev_status), _stream(stream)),
        "kvc_select")


def kvc_rope_table(tab, n_pos, pos0, D, theta, stream=None):
    _ok(lib.kvc_rope_table(_ptr(tab), n_pos, pos0, D, float(theta),
                           _stream(stream)), "kvc_rope_table")


def kvc_pack_rerope(kraw, vraw, kept, kept_count, L, H, D, tok_off, n_sess,
                    n_tok, budget, rope_tab, kview, vview, dev_status=None,
                    stream=None):
    _ok(lib.kvc_pack_rerope(_ptr(kraw), _ptr(vraw), _ptr(kept),
                            _ptr(kept_count), L, H, D, _ptr(tok_off), n_sess,
                            n_tok, budget, _ptr(rope_tab), _ptr(kview),
                            _ptr(vview), _ptr(dev_status), _stream(stream)),
        "kvc_pack_rerope")


def _host_ptr(t):
    """Address of a pinned host tensor (device-accessible at the same address
    under unified addressing)."""
    if not t.is_contiguous():
        raise ValueError("libkvc takes contiguous row-major tensors only")
    if t.is_cuda or not t.is_pinned():
        raise ValueError("the host-resident history must be a pinned CPU tensor")
    return t.data_ptr()


def kvc_pack_tiered(kraw_host, vraw_host, kept_prev, kept_count_prev, kcache_prev,
                    vview_prev, kept, kept_count, L, H, D, tok_off, n_sess, n_tok, budget,
                    rope_tab, kcache, kview, vview, n_hits=None, dev_status=None, stream=None):
    _ok(lib.kvc_pack_tiered(_host_ptr(kraw_host), _host_ptr(vraw_host), _ptr(kept_prev),
                            _ptr(kept_count_prev), _ptr(kcache_prev), _ptr(vview_prev),
                            _ptr(kept), _ptr(kept_count), L, H, D, _ptr(tok_off), n_sess,
                            n_tok, budget, _ptr(rope_tab), _ptr(kcache), _ptr(kview),
                            _ptr(vview), _ptr(n_hits), _ptr(dev_status), _stream(stream)),
        "kvc_pack_tiered")


def kvc_pack_tiered_slots(kslots_host, vslots_host, slot_elems, n_slots, host_slot, kept_prev,
                          kept_count_prev, kcache_prev, vview_prev, kept, kept_count, L, H, D,
                          tok_off, n_sess, n_tok, budget, rope_tab, kcache, kview, vview,
                          n_hits=None, dev_status=None, stream=None):
    _ok(lib.kvc_pack_tiered_slots(_host_ptr(kslots_host), _host_ptr(vslots_host), slot_elems,
                                  n_slots, _ptr(host_slot), _ptr(kept_prev),
                                  _ptr(kept_count_prev), _ptr(kcache_prev), _ptr(vview_prev),
                                  _ptr(kept), _ptr(kept_count), L, H, D, _ptr(tok_off), n_sess,
                                  n_tok, budget, _ptr(rope_tab), _ptr(kcache), _ptr(kview),
                                  _ptr(vview), _ptr(n_hits), _ptr(dev_status), _stream(stream)),
        "kvc_pack_tiered_slots")


def _np_ptr(a, dtype, count=None):
    """Address of a C-contiguous host array of the given dtype (None → NULL);
    with `count`, the array must hold at least that many elements (the C side
    reads that many)."""
    import numpy as np
    if a is None:
        return None
    if hasattr(a, "is_cuda"):  # a CPU torch tensor: elements of the same size
        if a.is_cuda or not a.is_contiguous():
            raise ValueError("expected a contiguous host tensor")
        if a.element_size() != np.dtype(dtype).itemsize:
            raise ValueError(f"expected {np.dtype(dtype).itemsize}-byte elements")
        n, ptr = a.numel(), a.data_ptr()
    else:
        if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
            raise ValueError(f"expected a C-contiguous numpy array of {np.dtype(dtype).name}")
        n, ptr = a.size, a.ctypes.data
    if count is not None and n < count:
        raise ValueError(f"expected at least {count} elements, got {n}")
    return ptr


def kvc_repo_plan(kept, kept_count, kept_prev, kept_count_prev, L, H, n_sess, budget, tok_off,
                  n_blocks):
    """(used, need): sorted int64 unit indices (l·H + h)·n_blocks + g of one
    step (host arrays in)."""
    import numpy as np
    used = np.empty(L * H * n_blocks, np.int64)
    need = np.empty(L * H * n_blocks, np.int64)
    nu, nn = _c.c_int64(0), _c.c_int64(0)
    segs = L * H * n_sess
    _ok(lib.kvc_repo_plan(_np_ptr(kept, np.int32, segs * budget),
                          _np_ptr(kept_count, np.int32, segs),
                          _np_ptr(kept_prev, np.int32, segs * budget),
                          _np_ptr(kept_count_prev, np.int32, segs),
                          L, H, n_sess, budget, _np_ptr(tok_off, np.int64, n_sess + 1), n_blocks,
                          used.ctypes.data, _c.addressof(nu), need.ctypes.data,
                          _c.addressof(nn)), "kvc_repo_plan")
    return used[:nu.value].copy(), need[:nn.value].copy()


class _RepoStats(_c.Structure):
    _fields_ = [(n, _c.c_int64) for n in ("steps", "needed", "host_hits", "fetched",
                                          "read_calls", "bytes_read", "evictions",
                                          "bytes_written")]


class KvcRepo:
    """The repository view (kvc_repo_*): units (layer, KV head, 32-token
    block) of raw K/V in a backing file, up to n_slots of them in a host arena
    [n_slots][2][32][D] (pinned when a GPU is present, so
    kvc_pack_tiered_slots can read it)."""

    def __init__(self, path, n_blocks, L, H, D, n_slots, io_threads=4, direct=False):
        import numpy as np
        import torch
        self.n_blocks, self.L, self.H, self.D, self.n_slots = n_blocks, L, H, D, n_slots
        self.n_units = L * H * n_blocks
        self.half = 32 * D
        self.slot_elems = 2 * self.half
        if torch.cuda.is_available():
            # 4096-byte aligned (direct I/O needs it; the pinned allocator
            # does not promise it)
            raw = torch.empty(n_slots * self.slot_elems + 2048, dtype=torch.bfloat16,
                              pin_memory=True)
            off = (-raw.data_ptr() % 4096) // 2
            self._raw = raw
            self.arena = raw[off:off + n_slots * self.slot_elems]
            base = self.arena.data_ptr()
        else:  # host-only use: a 4096-byte-aligned numpy buffer
            raw = np.empty(n_slots * self.slot_elems + 2048, np.uint16)
            off = (-raw.ctypes.data % 4096) // 2
            self._raw = raw
            self.arena = raw[off:off + n_slots * self.slot_elems]
            base = self.arena.ctypes.data
        self._h = _c.c_void_p()
        _ok(lib.kvc_repo_create(str(path).encode(), n_blocks, L, H, D, n_slots, base,
                                io_threads, 1 if direct else 0, _c.byref(self._h)),
            "kvc_repo_create")
        self.host_slot = np.full(self.n_units, -1, np.int32)

    def put(self, b0, nb, kraw, vraw, n_tok):
        """Blocks b0 … b0+nb−1 from host [L][H][n_tok][D] bf16 arrays."""
        import numpy as np
        n = self.L * self.H * n_tok * self.D
        _ok(lib.kvc_repo_put(self._h, b0, nb, _np_ptr(kraw, np.uint16, n),
                             _np_ptr(vraw, np.uint16, n), n_tok), "kvc_repo_put")

    def step(self, used, need, table=True):
        """Brings `need` into host slots.  With `table`, returns the slot of
        every unit (−1: file only); otherwise None (see changes())."""
        import numpy as np
        used = np.ascontiguousarray(used, np.int64)
        need = np.ascontiguousarray(need, np.int64)
        _ok(lib.kvc_repo_step(self._h, used.ctypes.data, len(used), need.ctypes.data,
                              len(need), self.host_slot.ctypes.data if table else None),
            "kvc_repo_step")
        return self.host_slot if table else None

    def slot_table(self):
        """The slot of every unit now (without taking a step)."""
        _ok(lib.kvc_repo_slots(self._h, self.host_slot.ctypes.data), "kvc_repo_slots")
        return self.host_slot

    def changes(self):
        """(units, slots) whose slot the last step changed (−1: evicted)."""
        import numpy as np
        n = int(lib.kvc_repo_changes(self._h, None, None, 0))
        units = np.empty(n, np.int64)
        slots = np.empty(n, np.int32)
        if n:
            lib.kvc_repo_changes(self._h, units.ctypes.data, slots.ctypes.data, n)
        return units, slots

    def where(self, g) -> int:
        return int(lib.kvc_repo_where(self._h, g))

    def stats(self) -> dict:
        st = _RepoStats()
        _ok(lib.kvc_repo_get_stats(self._h, _c.addressof(st)), "kvc_repo_get_stats")
        return {n: int(getattr(st, n)) for n, _ in _RepoStats._fields_}

    def slots(self):
        """(kslots, vslots): the arena's K and V bases for kvc_pack_tiered_slots."""
        return self.arena, self.arena[self.half:]

    def close(self):
        if self._h:
            lib.kvc_repo_destroy(self._h)
            self._h = _c.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kvc_init_sentinel(kpool, vpool, L, H, D, n_slots, sentinel, stream=None):
    _ok(lib.kvc_init_sentinel(_ptr(kpool), _ptr(vpool), L, H, D, n_slots,
                              sentinel, _stream(stream)), "kvc_init_sentinel")


def kvc_redirect_free_workspace_size(n_sess, N, n_slots) -> int:
    return int(lib.kvc_redirect_free_workspace_size(n_sess, N, n_slots))


def kvc_redirect_free(slot_map, keepmask, n_sess, N, refcnt, n_slots,
                      prefix_len, sentinel, freed, freed_cap, n_freed, ws,
                      dev_status=None, stream=None):
    _ok(lib.kvc_redirect_free(_ptr(slot_map), _ptr(keepmask), n_sess, N,
                              _ptr(refcnt), n_slots, prefix_len, sentinel,
                              _ptr(freed), freed_cap, _ptr(n_freed), _ptr(ws),
                              ws.numel() * ws.element_size(), _ptr(dev_status),
                              _stream(stream)), "kvc_redirect_free")


def kvc_recover_score_workspace_size(n_req, max_blocks, L, H, Hq, D, block_size) -> int:
    return int(lib.kvc_recover_score_workspace_size(n_req, max_blocks, L, H, Hq, D, block_size))


def kvc_recover_score(q, lse, kpool, n_slots, block_table, max_blocks, seqused_k, count,
                      n_req, L, H, Hq, D, block_size, state, ws=None, dev_status=None,
                      stream=None):
    _ok(lib.kvc_recover_score(_ptr(q), _ptr(lse), _ptr(kpool), n_slots, _ptr(block_table),
                              max_blocks, _ptr(seqused_k), _ptr(count), n_req, L, H, Hq, D,
                              block_size, _ptr(state), _ptr(ws),
                              0 if ws is None else ws.numel() * ws.element_size(),
                              _ptr(dev_status), _stream(stream)), "kvc_recover_score")


def kvc_recover_score_ex(q, lse, kpool, n_slots, block_table, max_blocks, seqused_k, count,
                         n_req, L, H, Hq, D, block_size, state, ws=None, kernel="auto",
                         dev_status=None, stream=None):
    """kvc_recover_score with a named kernel (a KERNELS key or value)."""
    _ok(lib.kvc_recover_score_ex(_ptr(q), _ptr(lse), _ptr(kpool), n_slots, _ptr(block_table),
                                 max_blocks, _ptr(seqused_k), _ptr(count), n_req, L, H, Hq, D,
                                 block_size, _ptr(state), _ptr(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(),
                                 _ptr(dev_status), _kernel(kernel), _stream(stream)),
        "kvc_recover_score_ex")


def kvc_recover_tensor_core(H, Hq, D, block_size) -> bool:
    return bool(lib.kvc_recover_tensor_core(H, Hq, D, block_size))


def kvc_tail_plan(keepmask, mask_words, seqused_k, block_table, max_blocks, n_req,
                  block_size, n_slots, src_slot, dst_slot, n_pairs, n_tail_blocks,
                  freed_blocks, n_freed, new_table, tail_mask, dev_status=None, stream=None):
    _ok(lib.kvc_tail_plan(_ptr(keepmask), mask_words, _ptr(seqused_k), _ptr(block_table),
                          max_blocks, n_req, block_size, n_slots, _ptr(src_slot),
                          _ptr(dst_slot), _ptr(n_pairs), _ptr(n_tail_blocks),
                          _ptr(freed_blocks), _ptr(n_freed), _ptr(new_table),
                          _ptr(tail_mask), _ptr(dev_status), _stream(stream)),
        "kvc_tail_plan")


def kvc_tail_compact(kpool, vpool, n_slots, L, H, D, src_slot, dst_slot, n_pairs, pair_cap,
                     n_req, dev_status=None, stream=None):
    _ok(lib.kvc_tail_compact(_ptr(kpool), _ptr(vpool), n_slots, L, H, D, _ptr(src_slot),
                             _ptr(dst_slot), _ptr(n_pairs), pair_cap, n_req,
                             _ptr(dev_status), _stream(stream)), "kvc_tail_compact")


def kvc_lrfu_update(scores, seg_off, n_seg, max_seg_len, top_p, lam, keep_score,
                    hitmask=None, dev_status=None, stream=None):
    _ok(lib.kvc_lrfu_update(_ptr(scores), _ptr(seg_off), n_seg, max_seg_len, float(top_p),
                            float(lam), _ptr(keep_score), _ptr(hitmask), _ptr(dev_status),
                            _stream(stream)), "kvc_lrfu_update")


def kvc_token_confidence(logits, n_tok, V, top_k, conf, dev_status=None, stream=None):
    _ok(lib.kvc_token_confidence(_ptr(logits), n_tok, V, top_k, _ptr(conf), _ptr(dev_status),
                                 _stream(stream)), "kvc_token_confidence")


def kvc_conf_trend_budget(conf, trace_off, n_trace, max_trace_len, window, stride, bottom_pct,
                          budget_step, max_budget, slope, budget, n_kept, dev_status=None,
                          stream=None):
    _ok(lib.kvc_conf_trend_budget(_ptr(conf), _ptr(trace_off), n_trace, max_trace_len, window,
                                  stride, float(bottom_pct), budget_step, max_budget,
                                  _ptr(slope), _ptr(budget), _ptr(n_kept), _ptr(dev_status),
                                  _stream(stream)), "kvc_conf_trend_budget")
