"""fp64 CPU oracle for Windowed-MTP decode attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA
library (``speculative_decoding_attention_gb300``) and never imports it.

The arithmetic lives in ``wm_oracle.c`` (plain C, fp64, OpenMP over rows); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
What each function computes, and the page passage it follows, is stated in
the C file's header:

* ``verify``  -- full-context causal attention of the k+1 proposed positions
  ("Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
  Context", Abstract: full-attention verification left intact);
* ``draft``   -- attention over the sink + sliding-window key set (same
  Abstract: StreamingLLM-style sliding window plus attention sink, draft only);
* ``attend_subset`` -- attention over an explicit key subset;
* ``lse_merge`` -- the log-sum-exp merge identity.

Inputs are bf16 tensors (torch, CPU) or uint16 numpy arrays holding bf16 bit
patterns; outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(plant: int = 0) -> str:
    name = "libwm_oracle.so" if plant == 0 else f"libwm_oracle_plant{plant}.so"
    return os.path.join(_BUILD, name)


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant used by the pin tests)."""
    out = lib_path(plant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           f"-DWMO_PLANT={plant}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _KV(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("n_cap", ctypes.c_int64), ("n_pages", ctypes.c_int64),
        ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
    ]


def _load(plant: int = 0) -> ctypes.CDLL:
    with _lock:
        if plant in _libs:
            return _libs[plant]
        lib = ctypes.CDLL(build(plant))
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.wmo_verify.argtypes = [ctypes.POINTER(_KV), I32, I32, P, P, D, P, I64, P, P]
        lib.wmo_draft.argtypes = [ctypes.POINTER(_KV), I32, P, P, I64, I64, D, P, I64, P, P]
        lib.wmo_draft_mem.argtypes = [ctypes.POINTER(_KV), ctypes.POINTER(_KV), P, I32, P, P, I64, I64, D, P,
                                      I64, P, P]
        lib.wmo_attend_subset.argtypes = [P, P, P, P, I64, I32, D, P, P]
        lib.wmo_lse_merge.argtypes = [P, P, I32, I64, I32, P, P]
        for f in (lib.wmo_verify, lib.wmo_draft, lib.wmo_draft_mem, lib.wmo_attend_subset, lib.wmo_lse_merge):
            f.restype = ctypes.c_int
        lib.wmo_num_threads.restype = ctypes.c_int
        lib.wmo_set_num_threads.argtypes = [ctypes.c_int]
        lib.wmo_set_num_threads.restype = None
        _libs[plant] = lib
        return lib


def _bits(x) -> np.ndarray:
    """bf16 data as a C-contiguous uint16 array of bit patterns."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch  # local: only for tensor inputs

    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bf16 tensor, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i64(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
    return np.ascontiguousarray(x, dtype=np.int64)


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy() if hasattr(x, "detach") else np.asarray(x)
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


class KV:
    """A K/V store seen by logical (sequence, kv head, position).

    contiguous: ``k``/``v`` shaped [batch, n_kv_heads, n_cap, head_dim];
    paged: ``k``/``v`` shaped [n_pages, n_kv_heads, page_size, head_dim] plus a
    ``block_table`` [batch, max_pages] (position j of sequence b lives in page
    block_table[b, j // page_size], row j % page_size).
    """

    def __init__(self, k, v, block_table=None, batch: int | None = None):
        self.k = _bits(k)
        self.v = _bits(v)
        if self.k.shape != self.v.shape or self.k.ndim != 4:
            raise ValueError("k and v must share a 4-d shape")
        self.block_table = None if block_table is None else _i32(block_table)
        s = _KV()
        s.k, s.v = _ptr(self.k), _ptr(self.v)
        s.n_kv_heads, s.head_dim = self.k.shape[1], self.k.shape[3]
        if self.block_table is None:
            s.block_table = None
            s.batch, s.n_cap = self.k.shape[0], self.k.shape[2]
            s.n_pages, s.page_size, s.max_pages = 0, 0, 0
        else:
            s.block_table = _ptr(self.block_table)
            s.batch = self.block_table.shape[0] if batch is None else batch
            s.max_pages = self.block_table.shape[1]
            s.n_pages, s.page_size, s.n_cap = self.k.shape[0], self.k.shape[2], 0
        self.c = s

    @property
    def head_dim(self) -> int:
        return self.c.head_dim


def _rows(rows, total: int):
    if rows is None:
        return None, total
    r = _i64(rows).reshape(-1)
    return r, r.size


def _check_batch(kv: KV, batch: int, n_pos: int, head_dim: int) -> None:
    # The C routines index queries and positions by the store's batch: a query
    # batch or position list of another size would be read or written out of
    # bounds.
    if batch != kv.c.batch or n_pos != batch or head_dim != kv.c.head_dim:
        raise ValueError(f"query batch {batch} / positions {n_pos} / head_dim {head_dim} do not match "
                         f"the store (batch {kv.c.batch}, head_dim {kv.c.head_dim})")


def verify(kv: KV, q, seq_lens, scale: float, rows=None, plant: int = 0):
    """Full-context causal attention of the T proposed positions.

    q: bf16 [batch, T, Hq, D].  Query (b, i) sits at position seq_lens[b]-T+i.
    Returns (out [n, D], lse [n]) float64 for the selected flattened rows
    (all rows of [batch, T, Hq] when ``rows`` is None).
    """
    qb = _bits(q)
    B, T, Hq, D = qb.shape
    sl = _i64(seq_lens)
    _check_batch(kv, B, sl.size, D)
    r, n = _rows(rows, B * T * Hq)
    out = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load(plant).wmo_verify(ctypes.byref(kv.c), T, Hq, _ptr(qb), _ptr(sl), float(scale),
                                 _ptr(r), n, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle verify failed ({rc})")
    return out, lse


def draft(hist: KV, q, pos, sink: int, window: int, scale: float, rows=None, plant: int = 0):
    """Sink + sliding-window attention of one query per head.

    hist: the draft KV history by absolute position; q: bf16 [batch, Hq, D];
    pos: [batch] query positions.  Returns (out [n, D], lse [n]) float64.
    """
    qb = _bits(q)
    B, Hq, D = qb.shape
    p = _i64(pos)
    _check_batch(hist, B, p.size, D)
    r, n = _rows(rows, B * Hq)
    out = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load(plant).wmo_draft(ctypes.byref(hist.c), Hq, _ptr(qb), _ptr(p), int(sink), int(window),
                                float(scale), _ptr(r), n, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle draft failed ({rc})")
    return out, lse


def draft_mem(hist: KV, mem: KV, mem_count, q, pos, sink: int, window: int, scale: float, rows=None,
              plant: int = 0):
    """Sink + window attention plus every materialized memory slot
    (memory-augmented sliding-window drafting).

    mem: contiguous store [batch, Hkv, capacity, D] of memory-slot K/V;
    mem_count: [batch] slots materialized so far.  Otherwise as draft().
    """
    qb = _bits(q)
    B, Hq, D = qb.shape
    p = _i64(pos)
    mc = _i64(mem_count)
    _check_batch(hist, B, p.size, D)
    _check_batch(mem, B, mc.size, D)
    r, n = _rows(rows, B * Hq)
    out = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load(plant).wmo_draft_mem(ctypes.byref(hist.c), ctypes.byref(mem.c), _ptr(mc), Hq, _ptr(qb), _ptr(p),
                                    int(sink), int(window), float(scale), _ptr(r), n, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle draft_mem failed ({rc})")
    return out, lse


def attend_subset(q, k, v, member, scale: float, plant: int = 0):
    """Attention of one bf16 query [D] over the keys k, v [n, D] where member[j]."""
    qb, kb, vb = _bits(q).reshape(-1), _bits(k), _bits(v)
    m = np.ascontiguousarray(np.asarray(member, dtype=bool).astype(np.uint8))
    n, D = kb.shape
    out = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    rc = _load(plant).wmo_attend_subset(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(m), n, D, float(scale),
                                        _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle attend_subset failed ({rc})")
    return out, float(lse[0])


def lse_merge(o_parts, lse_parts):
    """Merge partials o_parts [rows, n_parts, D], lse_parts [rows, n_parts] (natural log)."""
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    ls = np.ascontiguousarray(lse_parts, dtype=np.float64)
    rows, n_parts, D = o.shape
    out = np.zeros((rows, D), np.float64)
    lse = np.zeros((rows,), np.float64)
    rc = _load().wmo_lse_merge(_ptr(o), _ptr(ls), n_parts, rows, D, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"oracle lse_merge failed ({rc})")
    return out, lse


def num_threads() -> int:
    """Host threads the oracle's OpenMP loops use."""
    return int(_load().wmo_num_threads())


def set_num_threads(n: int) -> None:
    """Host threads for the oracle's OpenMP loops from now on."""
    _load().wmo_set_num_threads(int(n))
