"""Thin ctypes binding of libforkkv (include/forkkv.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
computation of its own: tensors are passed as device pointers, host arrays as
host pointers, and a non-zero status raises ``ForkKVError``.  PyTorch only
provides device memory and streams.  Importing this module does not load the
library; the first call does, and raises if ``libforkkv.so`` has not been
built (``__graft_entry__.build()``).  There is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libforkkv.so")
_lib = None

PAGE_SIZE = 16
HEAD_DIM = 128
RANK = 16
BASE_TILE_BYTES = 4096
RES_TILE_BYTES = 512
ROPE_ROW_BYTES = 256
PLAN_ITEM_INTS = 16
PLAN_UNIT_INTS = 16
JOB_BASE = 0
JOB_RES = 1
JOB_BASE_ZERO = 2
JOB_RES_ZERO = 3
FORK_SHARE_RES = 1
FORK_FREEZE_TAIL = 2
DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_ARG = 1, 2, 4


class ForkKVError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({strerror(code)})")
        self.code = code


class forkkv_cow_job(ctypes.Structure):
    _fields_ = [("src_page", ctypes.c_int32), ("dst_page", ctypes.c_int32), ("n_valid", ctypes.c_int32),
                ("kind", ctypes.c_int32)]


class forkkv_stats(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int32), ("base_live", ctypes.c_int32), ("res_live", ctypes.c_int32),
                ("base_free", ctypes.c_int32), ("res_free", ctypes.c_int32), ("base_shared", ctypes.c_int32),
                ("res_shared", ctypes.c_int32), ("base_refsum", ctypes.c_int64), ("res_refsum", ctypes.c_int64)]


class forkkv_pool_desc(ctypes.Structure):
    _fields_ = [("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p), ("k_res", ctypes.c_void_p),
                ("v_res", ctypes.c_void_p), ("num_base_pages", ctypes.c_int32), ("num_res_pages", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("n_layers", ctypes.c_int32)]


class forkkv_plan_info(ctypes.Structure):
    _fields_ = [("n_items", ctypes.c_int32), ("n_slots", ctypes.c_int32), ("n_ctas", ctypes.c_int32),
                ("n_units", ctypes.c_int32), ("plan_ints", ctypes.c_int32)]


class forkkv_attn_params(ctypes.Structure):
    _fields_ = [
        ("n_agents", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("rank", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("layer", ctypes.c_int32), ("pools", forkkv_pool_desc),
        ("q", ctypes.c_void_p), ("out", ctypes.c_void_p), ("bpt", ctypes.c_void_p), ("rpt", ctypes.c_void_p),
        ("pt_stride", ctypes.c_int32), ("seq_lens", ctypes.c_void_p), ("positions", ctypes.c_void_p),
        ("max_seq_len", ctypes.c_int32), ("B_k", ctypes.c_void_p), ("B_v", ctypes.c_void_p),
        ("adapter_ids", ctypes.c_void_p), ("n_adapters", ctypes.c_int32), ("rope_table", ctypes.c_void_p),
        ("rope_table_positions", ctypes.c_int32), ("rope_theta", ctypes.c_double), ("sm_scale", ctypes.c_float),
        ("plan", ctypes.c_void_p), ("plan_items", ctypes.c_int32), ("plan_slots", ctypes.c_int32),
        ("plan_ctas", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("holes", ctypes.c_void_p),
    ]


_P = ctypes.POINTER
_i32, _u32, _vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p
_SIGNATURES = {
    "forkkv_strerror": ([_i32], ctypes.c_char_p),
    "forkkv_version": ([], _i32),
    "forkkv_alloc_create": ([_i32, _i32, _i32, _P(_vp)], _i32),
    "forkkv_alloc_destroy": ([_vp], _i32),
    "forkkv_seq_create": ([_vp, _i32, _P(_i32)], _i32),
    "forkkv_fork": ([_vp, _i32, _i32, _u32, _P(_i32), _P(forkkv_cow_job), _i32, _P(_i32)], _i32),
    "forkkv_append": ([_vp, _i32, _i32, _P(forkkv_cow_job), _i32, _P(_i32)], _i32),
    "forkkv_free": ([_vp, _i32], _i32),
    "forkkv_abort": ([_vp, _i32, _P(_i32), _P(_i32)], _i32),
    "forkkv_commit": ([_vp, _i32, _i32, _vp, _i32, _P(forkkv_cow_job), _i32, _P(_i32)], _i32),
    "forkkv_lcp_len": ([_vp, _i32, _vp, _i32, _P(_i32)], _i32),
    "forkkv_seq_len": ([_vp, _i32, _P(_i32)], _i32),
    "forkkv_slot_maps": ([_vp, _vp, _i32, _vp], _i32),
    "forkkv_page_tables": ([_vp, _vp, _i32, _i32, _vp, _vp, _vp], _i32),
    "forkkv_refcount": ([_vp, _i32, _i32, _P(_i32)], _i32),
    "forkkv_stats_get": ([_vp, _P(forkkv_stats)], _i32),
    "forkkv_write_rows": ([_P(forkkv_pool_desc), _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp], _i32),
    "forkkv_residual_fill": ([_P(forkkv_pool_desc), _i32, _vp, _i32, _i32, _vp, _i32, _vp, _vp], _i32),
    "forkkv_append_rows": ([_P(forkkv_pool_desc), _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp],
                           _i32),
    "forkkv_cow_copy_rows": ([_P(forkkv_pool_desc), _P(forkkv_cow_job), _i32, _vp], _i32),
    "forkkv_rope_table_bytes": ([_i32, _P(ctypes.c_size_t)], _i32),
    "forkkv_rope_table_build": ([ctypes.c_double, _i32, _vp, _vp], _i32),
    "forkkv_plan_build": ([_vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _P(forkkv_plan_info)], _i32),
    "forkkv_decode_workspace_size": ([_P(forkkv_attn_params), _P(ctypes.c_size_t)], _i32),
    "forkkv_residual_attn_decode": ([_P(forkkv_attn_params), _vp], _i32),
    "forkkv_step_graph_create": ([_P(forkkv_attn_params), _vp, _i32, _P(_vp)], _i32),
    "forkkv_step_graph_launch": ([_vp, _vp], _i32),
    "forkkv_step_graph_destroy": ([_vp], _i32),
    "forkkv_prefill_workspace_size": ([_P(forkkv_attn_params), _P(ctypes.c_size_t)], _i32),
    "forkkv_residual_attn_prefill_chunk": ([_P(forkkv_attn_params), _vp], _i32),
    "forkkv_get_device_status": ([_P(_u32), _vp], _i32),
    "forkkv_wait_selftest": ([_u32, _vp], _i32),
    "forkkv_residual_attn_decode_static": ([_P(forkkv_attn_params), _vp], _i32),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build(); "
                               "there is no CPU or PyTorch fallback for this library")
        l = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def strerror(code: int) -> str:
    return lib().forkkv_strerror(code).decode()


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ForkKVError(rc, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---- allocator -------------------------------------------------------------

def forkkv_alloc_create(num_base_pages: int, num_res_pages: int, page_size: int = PAGE_SIZE) -> int:
    h = ctypes.c_void_p()
    _check(lib().forkkv_alloc_create(num_base_pages, num_res_pages, page_size, ctypes.byref(h)), "alloc_create")
    return h.value


def forkkv_alloc_destroy(alloc: int) -> None:
    _check(lib().forkkv_alloc_destroy(alloc), "alloc_destroy")


def forkkv_seq_create(alloc: int, n_tokens: int) -> int:
    sid = ctypes.c_int32()
    _check(lib().forkkv_seq_create(alloc, n_tokens, ctypes.byref(sid)), "seq_create")
    return sid.value


def _jobs_out(buf, n) -> List[Tuple[int, int, int, int]]:
    return [(buf[i].src_page, buf[i].dst_page, buf[i].n_valid, buf[i].kind) for i in range(n)]


def forkkv_fork(alloc: int, parent: int, prefix_len: int, flags: int = 0) -> Tuple[int, list]:
    child, n = ctypes.c_int32(), ctypes.c_int32()
    buf = (forkkv_cow_job * 2)()
    _check(lib().forkkv_fork(alloc, parent, prefix_len, flags, ctypes.byref(child), buf, 2, ctypes.byref(n)), "fork")
    return child.value, _jobs_out(buf, n.value)


def forkkv_append(alloc: int, seq: int, n_tokens: int) -> list:
    n = ctypes.c_int32()
    buf = (forkkv_cow_job * 2)()
    _check(lib().forkkv_append(alloc, seq, n_tokens, buf, 2, ctypes.byref(n)), "append")
    return _jobs_out(buf, n.value)


def forkkv_free(alloc: int, seq: int) -> None:
    _check(lib().forkkv_free(alloc, seq), "free")


def forkkv_abort(alloc: int, seq: int) -> Tuple[int, int]:
    """Free a speculative branch; returns (base pages, residual pages) released."""
    nb, nr = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().forkkv_abort(alloc, seq, ctypes.byref(nb), ctypes.byref(nr)), "abort")
    return nb.value, nr.value


def forkkv_commit(alloc: int, seq: int, lcp_len: int, siblings: Sequence[int] = ()) -> list:
    """LCP commit: abort the siblings, truncate seq to lcp_len, split a shared boundary page."""
    sib = np.ascontiguousarray(np.asarray(list(siblings), dtype=np.int32))
    n = ctypes.c_int32()
    buf = (forkkv_cow_job * 2)()
    _check(lib().forkkv_commit(alloc, seq, lcp_len, sib.ctypes.data if len(sib) else None, len(sib), buf, 2,
                               ctypes.byref(n)), "commit")
    return _jobs_out(buf, n.value)


def forkkv_lcp_len(spec: Sequence[int], observed: Sequence[int]) -> int:
    a = np.ascontiguousarray(np.asarray(list(spec), dtype=np.int32))
    b = np.ascontiguousarray(np.asarray(list(observed), dtype=np.int32))
    n = ctypes.c_int32()
    _check(lib().forkkv_lcp_len(a.ctypes.data if len(a) else None, len(a), b.ctypes.data if len(b) else None, len(b),
                                ctypes.byref(n)), "lcp_len")
    return n.value


def forkkv_seq_len(alloc: int, seq: int) -> int:
    n = ctypes.c_int32()
    _check(lib().forkkv_seq_len(alloc, seq, ctypes.byref(n)), "seq_len")
    return n.value


def forkkv_page_tables(alloc: int, seqs: Sequence[int], stride: int):
    """(bpt, rpt, seq_lens) as int32 numpy arrays [n, stride], [n, stride], [n]."""
    n = len(seqs)
    s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
    bpt = np.empty((n, stride), np.int32)
    rpt = np.empty((n, stride), np.int32)
    lens = np.empty((n,), np.int32)
    _check(lib().forkkv_page_tables(alloc, s.ctypes.data, n, stride, bpt.ctypes.data, rpt.ctypes.data,
                                    lens.ctypes.data), "page_tables")
    return bpt, rpt, lens


def forkkv_slot_maps(alloc: int, seqs: Sequence[int]) -> np.ndarray:
    """[n, 2] int32: each sequence's hole (first slot, length), (0, 0) without one."""
    n = len(seqs)
    s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
    holes = np.zeros((n, 2), np.int32)
    _check(lib().forkkv_slot_maps(alloc, s.ctypes.data, n, holes.ctypes.data), "slot_maps")
    return holes


def forkkv_refcount(alloc: int, kind: int, page: int) -> int:
    out = ctypes.c_int32()
    _check(lib().forkkv_refcount(alloc, kind, page, ctypes.byref(out)), "refcount")
    return out.value


def forkkv_stats_get(alloc: int) -> dict:
    st = forkkv_stats()
    _check(lib().forkkv_stats_get(alloc, ctypes.byref(st)), "stats")
    return {f: getattr(st, f) for f, _ in forkkv_stats._fields_}


# ---- pools -----------------------------------------------------------------

class Pools:
    """Device pools owned by PyTorch, described to the library by a forkkv_pool_desc."""

    def __init__(self, num_base_pages: int, num_res_pages: int, num_kv_heads: int, n_layers: int = 1,
                 device="cuda", fill: Optional[int] = None):
        mk = (lambda shape: torch.full(shape, fill, dtype=torch.uint8, device=device)) if fill is not None else \
            (lambda shape: torch.empty(shape, dtype=torch.uint8, device=device))
        self.k_base = mk((n_layers, num_kv_heads, num_base_pages, BASE_TILE_BYTES))
        self.v_base = mk((n_layers, num_kv_heads, num_base_pages, BASE_TILE_BYTES))
        self.k_res = mk((n_layers, num_res_pages, RES_TILE_BYTES))
        self.v_res = mk((n_layers, num_res_pages, RES_TILE_BYTES))
        self.desc = forkkv_pool_desc(self.k_base.data_ptr(), self.v_base.data_ptr(), self.k_res.data_ptr(),
                                     self.v_res.data_ptr(), num_base_pages, num_res_pages, num_kv_heads, n_layers)

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in (self.k_base, self.v_base, self.k_res, self.v_res))


def forkkv_write_rows(pools: Pools, layer: int, slot_base: Optional[torch.Tensor], slot_res: Optional[torch.Tensor],
                      k_base_rows=None, v_base_rows=None, k_res_rows=None, v_res_rows=None, stream=None) -> None:
    n = int((slot_base if slot_base is not None else slot_res).numel())
    _check(lib().forkkv_write_rows(ctypes.byref(pools.desc), layer, n, _ptr(slot_base), _ptr(slot_res),
                                   _ptr(k_base_rows), _ptr(v_base_rows), _ptr(k_res_rows), _ptr(v_res_rows),
                                   _stream(stream)), "write_rows")


def forkkv_residual_fill(pools: Pools, layer: int, x: torch.Tensor, A: torch.Tensor, slot_res: torch.Tensor,
                         stream=None) -> None:
    """x [n_tok, hidden], A [n_agents, 2, 16, hidden] bf16, slot_res [n_agents, n_tok] int32 (device)."""
    n_tok, hidden = x.shape
    n_ag = A.shape[0]
    _check(lib().forkkv_residual_fill(ctypes.byref(pools.desc), layer, _ptr(x), n_tok, hidden, _ptr(A), n_ag,
                                      _ptr(slot_res), _stream(stream)), "residual_fill")


def forkkv_append_rows(pools: Pools, layer: int, slot_base: Optional[torch.Tensor], slot_res: Optional[torch.Tensor],
                       k_base_rows=None, v_base_rows=None, x=None, A=None, adapter_ids=None, stream=None) -> None:
    """New tokens' base rows and residual rows from their hidden states x [n, hidden] with adapters
    A [n_adapters, 2, 16, hidden] (adapter_ids [n] or None: row index)."""
    n = int((slot_base if slot_base is not None else slot_res).numel())
    hidden = 0 if x is None else x.shape[1]
    n_ad = 0 if A is None else A.shape[0]
    _check(lib().forkkv_append_rows(ctypes.byref(pools.desc), layer, n, _ptr(slot_base), _ptr(slot_res),
                                    _ptr(k_base_rows), _ptr(v_base_rows), _ptr(x), hidden, _ptr(A), n_ad,
                                    _ptr(adapter_ids), _stream(stream)), "append_rows")


def forkkv_cow_copy_rows(pools: Pools, jobs: Sequence[Tuple[int, int, int, int]], stream=None) -> None:
    buf = (forkkv_cow_job * max(1, len(jobs)))(*[forkkv_cow_job(*j) for j in jobs])
    _check(lib().forkkv_cow_copy_rows(ctypes.byref(pools.desc), buf, len(jobs), _stream(stream)), "cow_copy_rows")


def forkkv_rope_table_build(rope_theta: float, n_positions: int, table: torch.Tensor, stream=None) -> None:
    assert table.numel() * table.element_size() >= n_positions * ROPE_ROW_BYTES
    _check(lib().forkkv_rope_table_build(float(rope_theta), n_positions, table.data_ptr(), _stream(stream)),
           "rope_table_build")


def rope_table(rope_theta: float, n_positions: int, device="cuda", stream=None) -> torch.Tensor:
    n = (n_positions + PAGE_SIZE - 1) // PAGE_SIZE * PAGE_SIZE
    t = torch.empty((n, ROPE_ROW_BYTES), dtype=torch.uint8, device=device)
    forkkv_rope_table_build(rope_theta, n, t, stream)
    return t


def forkkv_plan_build(bpt: np.ndarray, seq_lens: np.ndarray, num_kv_heads: int, target_ctas: int = 0):
    """Host plan: (int32 numpy array, forkkv_plan_info)."""
    bpt = np.ascontiguousarray(bpt, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    A, stride = bpt.shape
    info = forkkv_plan_info()
    _check(lib().forkkv_plan_build(bpt.ctypes.data, lens.ctypes.data, A, stride, num_kv_heads, target_ctas, None, 0,
                                   ctypes.byref(info)), "plan_build(size)")
    plan = np.empty((info.plan_ints,), np.int32)
    _check(lib().forkkv_plan_build(bpt.ctypes.data, lens.ctypes.data, A, stride, num_kv_heads, target_ctas,
                                   plan.ctypes.data, info.plan_ints, ctypes.byref(info)), "plan_build")
    return plan, info


# ---- attention -------------------------------------------------------------

def attn_params(pools: Pools, layer: int, q: torch.Tensor, out: torch.Tensor, bpt: torch.Tensor, rpt: torch.Tensor,
                seq_lens: torch.Tensor, positions: torch.Tensor, max_seq_len: int, B_k: torch.Tensor,
                B_v: torch.Tensor, adapter_ids: Optional[torch.Tensor] = None, rope: Optional[torch.Tensor] = None,
                rope_theta: float = 0.0, sm_scale: float = 0.0, plan: Optional[torch.Tensor] = None,
                plan_info: Optional[forkkv_plan_info] = None,
                holes: Optional[torch.Tensor] = None) -> forkkv_attn_params:
    """Fill a forkkv_attn_params from tensors (q/out [A, q_len, Hq, 128], tables [A, stride])."""
    A, q_len, Hq, D = q.shape
    p = forkkv_attn_params()
    p.n_agents, p.q_len, p.num_q_heads = A, q_len, Hq
    p.num_kv_heads = pools.desc.num_kv_heads
    p.head_dim, p.rank, p.page_size, p.layer = D, RANK, PAGE_SIZE, layer
    p.pools = pools.desc
    p.q, p.out = q.data_ptr(), out.data_ptr()
    p.bpt, p.rpt, p.pt_stride = bpt.data_ptr(), rpt.data_ptr(), bpt.shape[1]
    p.seq_lens, p.positions, p.max_seq_len = seq_lens.data_ptr(), positions.data_ptr(), max_seq_len
    p.B_k, p.B_v = B_k.data_ptr(), B_v.data_ptr()
    p.adapter_ids = _ptr(adapter_ids)
    p.n_adapters = B_k.shape[0]
    p.rope_table = _ptr(rope)
    p.rope_table_positions = 0 if rope is None else rope.shape[0]
    p.rope_theta = rope_theta
    p.sm_scale = sm_scale
    p.holes = _ptr(holes)
    if plan is not None:
        p.plan, p.plan_items, p.plan_slots = plan.data_ptr(), plan_info.n_items, plan_info.n_slots
        p.plan_ctas = plan_info.n_ctas
    return p


def forkkv_decode_workspace_size(p: forkkv_attn_params) -> int:
    n = ctypes.c_size_t()
    _check(lib().forkkv_decode_workspace_size(ctypes.byref(p), ctypes.byref(n)), "decode_workspace_size")
    return n.value


def forkkv_prefill_workspace_size(p: forkkv_attn_params) -> int:
    n = ctypes.c_size_t()
    _check(lib().forkkv_prefill_workspace_size(ctypes.byref(p), ctypes.byref(n)), "prefill_workspace_size")
    return n.value


def set_workspace(p: forkkv_attn_params, ws: Optional[torch.Tensor]) -> None:
    p.workspace = _ptr(ws)
    p.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()


def workspace_for(p: forkkv_attn_params, prefill: bool = False, device="cuda") -> Optional[torch.Tensor]:
    n = forkkv_prefill_workspace_size(p) if prefill else forkkv_decode_workspace_size(p)
    ws = torch.empty((max(n, 256) + 255) // 256 * 256, dtype=torch.uint8, device=device) if n else None
    set_workspace(p, ws)
    return ws


def forkkv_residual_attn_decode(p: forkkv_attn_params, stream=None) -> None:
    _check(lib().forkkv_residual_attn_decode(ctypes.byref(p), _stream(stream)), "residual_attn_decode")


class forkkv_step_rows(ctypes.Structure):
    _fields_ = [("n_rows", _i32), ("slot_base", _vp), ("slot_res", _vp), ("k_base_rows", _vp),
                ("v_base_rows", _vp), ("k_res_rows", _vp), ("v_res_rows", _vp)]


def forkkv_step_graph_create(params: Sequence[forkkv_attn_params], rows=None) -> int:
    """One decode step of len(params) layers as one CUDA graph.  rows: None, or per layer a tuple
    (slot_base, slot_res, k_base_rows, v_base_rows, k_res_rows, v_res_rows) of device tensors (or None)."""
    n = len(params)
    parr = (forkkv_attn_params * n)(*params)
    rarr = None
    if rows is not None:
        rarr = (forkkv_step_rows * n)()
        for l, (sb, sr, kb, vb, kr, vr) in enumerate(rows):
            rarr[l].n_rows = int((sb if sb is not None else sr).numel())
            rarr[l].slot_base, rarr[l].slot_res = _ptr(sb), _ptr(sr)
            rarr[l].k_base_rows, rarr[l].v_base_rows = _ptr(kb), _ptr(vb)
            rarr[l].k_res_rows, rarr[l].v_res_rows = _ptr(kr), _ptr(vr)
    out = _vp()
    _check(lib().forkkv_step_graph_create(parr, ctypes.cast(rarr, _vp) if rarr is not None else None, n,
                                          ctypes.byref(out)), "step_graph_create")
    return out.value


def forkkv_step_graph_launch(graph: int, stream=None) -> None:
    _check(lib().forkkv_step_graph_launch(graph, _stream(stream)), "step_graph_launch")


def forkkv_step_graph_destroy(graph: int) -> None:
    _check(lib().forkkv_step_graph_destroy(graph), "step_graph_destroy")


def forkkv_residual_attn_prefill_chunk(p: forkkv_attn_params, stream=None) -> None:
    _check(lib().forkkv_residual_attn_prefill_chunk(ctypes.byref(p), _stream(stream)), "residual_attn_prefill_chunk")


STATIC_SCRATCH_BYTES = 8 << 20
ERR_SCRATCH = -7


def forkkv_residual_attn_decode_static(p: forkkv_attn_params, stream=None) -> None:
    """Decode with the library's own static scratch, for callers that cannot allocate device
    memory (the workspace fields of ``p`` are ignored; see include/forkkv.h)."""
    _check(lib().forkkv_residual_attn_decode_static(ctypes.byref(p), _stream(stream)),
           "residual_attn_decode_static")


def forkkv_wait_selftest(polls: int, stream=None) -> None:
    _check(lib().forkkv_wait_selftest(int(polls), _stream(stream)), "wait_selftest")


def forkkv_get_device_status(stream=None) -> int:
    v = ctypes.c_uint32()
    _check(lib().forkkv_get_device_status(ctypes.byref(v), _stream(stream)), "get_device_status")
    return v.value
