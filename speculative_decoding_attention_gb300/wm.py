"""ctypes binding of ``libwm.so`` (declared in ``include/wm_api.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  If the library has not been built, ``load()`` raises -- there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import build as _build

WM_OK, WM_ERR_INVALID_ARG, WM_ERR_UNSUPPORTED, WM_ERR_WORKSPACE, WM_ERR_CUDA, WM_ERR_DEVICE_DATA = range(6)
WM_OP_DRAFT, WM_OP_VERIFY, WM_OP_DRAFT_STEP, WM_OP_DRAFT_MEM = 0, 1, 2, 3
WM_DRAFT_MATH_MMA, WM_DRAFT_MATH_FMA = 0, 1
DEVERR_NAMES = {0: "none", 1: "bad length", 2: "bad page", 3: "pipeline wait timeout", 4: "internal check"}

EXPORTED = ("wm_ring_append", "wm_ring_fill", "wm_ring_rollback", "wm_draft_attn", "wm_verify_attn",
            "wm_lse_merge", "wm_plan_splits", "wm_verify_persistent", "wm_workspace_size", "wm_get_device_error",
            "wm_status_string", "wm_version", "wm_draft_attn_static", "wm_draft_step", "wm_draft_attn_mem",
            "wm_mem_append", "wm_mem_rollback", "wm_set_test_stall", "wm_set_draft_math")
STATIC_SCRATCH_BYTES = 8 << 20  # WM_STATIC_SCRATCH_BYTES

_lib = None
_lock = threading.Lock()


class WmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class _Ring(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos_tag", ctypes.c_void_p),
                ("n_seen", ctypes.c_void_p), ("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("sink", ctypes.c_int32), ("window", ctypes.c_int32)]


class _Mem(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("count", ctypes.c_void_p),
                ("capacity", ctypes.c_int64), ("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


class _KV(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("n_cap", ctypes.c_int64), ("n_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libwm.so; raises if it was not built (``__graft_entry__.build()``)."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded already: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libwm.so not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.wm_ring_append.argtypes = [P, P, P, P]
        lib.wm_ring_fill.argtypes = [P, P, P]
        lib.wm_ring_rollback.argtypes = [P, P, P]
        lib.wm_draft_attn.argtypes = [P, P, I32, F, I32, P, P, P, ctypes.c_size_t, P]
        lib.wm_verify_attn.argtypes = [P, P, I32, I32, F, I32, P, P, P, ctypes.c_size_t, P]
        lib.wm_draft_attn_static.argtypes = [P, P, I32, F, I32, P, P, P]
        lib.wm_draft_step.argtypes = [P, P, P, P, P, I32, F, I32, P, P, P, ctypes.c_size_t, P]
        lib.wm_draft_attn_mem.argtypes = [P, P, P, I32, F, I32, P, P, P, ctypes.c_size_t, P]
        lib.wm_mem_append.argtypes = [P, P, P, P]
        lib.wm_mem_rollback.argtypes = [P, P, P]
        lib.wm_lse_merge.argtypes = [P, P, I32, I64, I32, P, P, P]
        lib.wm_plan_splits.argtypes = [I32, I32, I32, I32, I32, I32, I64, I32]
        lib.wm_plan_splits.restype = I32
        lib.wm_verify_persistent.argtypes = [I32, I32, I32, I32, I32, I64, I32]
        lib.wm_verify_persistent.restype = I32
        lib.wm_workspace_size.argtypes = [I32, I32, I32, I32, I32, I32, I64, I32]
        lib.wm_workspace_size.restype = ctypes.c_size_t
        lib.wm_get_device_error.argtypes = [ctypes.POINTER(I32), P]
        lib.wm_status_string.argtypes = [I32]
        lib.wm_status_string.restype = ctypes.c_char_p
        lib.wm_version.restype = I32
        lib.wm_set_test_stall.argtypes = [I32, ctypes.c_uint32]
        lib.wm_set_test_stall.restype = I32
        lib.wm_set_draft_math.argtypes = [I32]
        lib.wm_set_draft_math.restype = I32
        for name in ("wm_ring_append", "wm_ring_fill", "wm_ring_rollback", "wm_draft_attn", "wm_draft_attn_static",
                     "wm_verify_attn", "wm_lse_merge", "wm_get_device_error"):
            getattr(lib, name).restype = I32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().wm_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != WM_OK:
        raise WmError(status, what)


# The current stream's handle without building a Stream object (a third of a
# short call's host time otherwise); the public query where it is missing.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int | None:
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, what: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{what} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


@dataclass
class Ring:
    """A draft ring buffer (``wm_ring``): sink + window slots per sequence."""
    k: torch.Tensor          # [B, Hkv, S+W, D] bf16
    v: torch.Tensor
    pos_tag: torch.Tensor    # [B, S+W] int32, -1 = empty
    n_seen: torch.Tensor     # [B] int64
    sink: int
    window: int

    @classmethod
    def create(cls, batch: int, n_kv_heads: int, head_dim: int, sink: int, window: int,
               device="cuda") -> "Ring":
        slots = sink + window
        k = torch.zeros((batch, n_kv_heads, slots, head_dim), dtype=torch.bfloat16, device=device)
        v = torch.zeros_like(k)
        tag = torch.full((batch, slots), -1, dtype=torch.int32, device=device)
        seen = torch.zeros((batch,), dtype=torch.int64, device=device)
        return cls(k, v, tag, seen, sink, window)

    @property
    def batch(self) -> int:
        return self.k.shape[0]

    @property
    def n_kv_heads(self) -> int:
        return self.k.shape[1]

    @property
    def head_dim(self) -> int:
        return self.k.shape[3]

    def c(self) -> _Ring:
        r = _Ring()
        r.k = _dev(self.k, torch.bfloat16, "ring.k")
        r.v = _dev(self.v, torch.bfloat16, "ring.v")
        r.pos_tag = _dev(self.pos_tag, torch.int32, "ring.pos_tag")
        r.n_seen = _dev(self.n_seen, torch.int64, "ring.n_seen")
        r.batch, r.n_kv_heads, r.head_dim = self.batch, self.n_kv_heads, self.head_dim
        r.sink, r.window = self.sink, self.window
        return r


@dataclass
class Mem:
    """Memory slots of a memory-augmented draft (``wm_mem``): K/V
    [B, Hkv, capacity, D] bf16 and the per-sequence count of materialized slots."""
    k: torch.Tensor
    v: torch.Tensor
    count: torch.Tensor      # [B] int64

    @classmethod
    def create(cls, batch: int, n_kv_heads: int, head_dim: int, capacity: int, device="cuda") -> "Mem":
        k = torch.zeros((batch, n_kv_heads, capacity, head_dim), dtype=torch.bfloat16, device=device)
        return cls(k, torch.zeros_like(k), torch.zeros((batch,), dtype=torch.int64, device=device))

    @property
    def capacity(self) -> int:
        return self.k.shape[2]

    def c(self) -> _Mem:
        m = _Mem()
        m.k = _dev(self.k, torch.bfloat16, "mem.k")
        m.v = _dev(self.v, torch.bfloat16, "mem.v")
        m.count = _dev(self.count, torch.int64, "mem.count")
        m.capacity = self.capacity
        m.batch, m.n_kv_heads, m.head_dim = self.k.shape[0], self.k.shape[1], self.k.shape[3]
        return m


def mem_keys(ring: "Ring", mem: Mem) -> int:
    """max_keys of WM_OP_DRAFT_MEM: the ring's slots in whole 64-key tiles plus the memory capacity."""
    return -(-(ring.sink + ring.window) // 64) * 64 + mem.capacity


@dataclass
class KVCache:
    """A full-context cache (``wm_kv``): contiguous [B, Hkv, n_cap, D] or paged
    [n_pages, Hkv, page_size, D] with a block table [B, max_pages]."""
    k: torch.Tensor
    v: torch.Tensor
    seq_lens: torch.Tensor               # [B] int64
    block_table: torch.Tensor | None = None

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def batch(self) -> int:
        return self.seq_lens.shape[0]

    @property
    def n_kv_heads(self) -> int:
        return self.k.shape[1]

    @property
    def head_dim(self) -> int:
        return self.k.shape[3]

    @property
    def capacity(self) -> int:
        if self.paged:
            return self.block_table.shape[1] * self.k.shape[2]
        return self.k.shape[2]

    def c(self) -> _KV:
        s = _KV()
        s.k = _dev(self.k, torch.bfloat16, "kv.k")
        s.v = _dev(self.v, torch.bfloat16, "kv.v")
        s.seq_lens = _dev(self.seq_lens, torch.int64, "kv.seq_lens")
        s.n_kv_heads, s.head_dim, s.batch = self.n_kv_heads, self.head_dim, self.batch
        if self.paged:
            s.block_table = _dev(self.block_table, torch.int32, "kv.block_table")
            s.n_pages, s.page_size = self.k.shape[0], self.k.shape[2]
            s.max_pages = self.block_table.shape[1]
            s.n_cap = 0
        else:
            s.block_table = None
            s.n_cap = self.k.shape[2]
            s.n_pages = s.page_size = s.max_pages = 0
        return s


def ring_append(ring: Ring, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Append one entry per sequence (k_new, v_new: [B, Hkv, D] bf16)."""
    r = ring.c()
    _check(load().wm_ring_append(ctypes.byref(r), _dev(k_new, torch.bfloat16, "k_new"),
                                 _dev(v_new, torch.bfloat16, "v_new"), _stream(stream)), "wm_ring_append")


def ring_fill(ring: Ring, hist: KVCache, stream=None) -> None:
    """Bulk-fill the ring with positions 0..hist.seq_lens[b]-1 of ``hist``."""
    r, h = ring.c(), hist.c()
    _check(load().wm_ring_fill(ctypes.byref(r), ctypes.byref(h), _stream(stream)), "wm_ring_fill")


def ring_rollback(ring: Ring, new_len: torch.Tensor, stream=None) -> None:
    """Forget draft entries at positions >= new_len[b] (int64 [B] device tensor)."""
    r = ring.c()
    _check(load().wm_ring_rollback(ctypes.byref(r), _dev(new_len, torch.int64, "new_len"),
                                   _stream(stream)), "wm_ring_rollback")


def plan_splits(op: int, batch: int, n_kv_heads: int, n_q_heads: int, n_q: int, head_dim: int,
                max_keys: int, n_split: int = 0) -> int:
    return int(load().wm_plan_splits(op, batch, n_kv_heads, n_q_heads, n_q, head_dim, max_keys, n_split))


def verify_persistent(batch: int, n_kv_heads: int, n_q_heads: int, n_q: int, head_dim: int, max_keys: int,
                      n_split: int = 0) -> int:
    """CTA count of the persistent verify for these arguments, 0 when the call
    runs the split plan (see wm_verify_persistent in include/wm_api.h)."""
    return int(load().wm_verify_persistent(batch, n_kv_heads, n_q_heads, n_q, head_dim, max_keys, n_split))


def workspace_size(op: int, batch: int, n_kv_heads: int, n_q_heads: int, n_q: int, head_dim: int,
                   max_keys: int, n_split: int = 0) -> int:
    n = load().wm_workspace_size(op, batch, n_kv_heads, n_q_heads, n_q, head_dim, max_keys, n_split)
    if n == ctypes.c_size_t(-1).value:
        raise WmError(WM_ERR_INVALID_ARG, "wm_workspace_size")
    return int(n)


def _workspace(nbytes: int, device, workspace: torch.Tensor | None) -> tuple[int, int]:
    if nbytes == 0:
        return (workspace.data_ptr() if workspace is not None else 0), \
            (workspace.numel() if workspace is not None else 0)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _keepalive.append(workspace)
        if len(_keepalive) > 8:
            del _keepalive[0]
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


_keepalive: list[torch.Tensor] = []


def _new_out(shape, dtype, device) -> torch.Tensor:
    """Output buffer of a call that was given none.  Uninitialised: every
    element is written by the call."""
    return torch.empty(tuple(shape), dtype=dtype, device=device)


def draft_attn(ring: Ring, q: torch.Tensor, scale: float, n_split: int = 0, out=None, lse=None,
               workspace=None, stream=None):
    """Sink + window draft attention of q [B, Hq, D]; returns (out bf16, lse fp32)."""
    B, Hq, D = q.shape
    if out is None:
        out = _new_out(q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = _new_out((B, Hq), torch.float32, q.device)
    need = workspace_size(WM_OP_DRAFT, B, ring.n_kv_heads, Hq, 1, D, ring.sink + ring.window, n_split)
    ws, ws_bytes = _workspace(need, q.device, workspace)
    r = ring.c()
    _check(load().wm_draft_attn(ctypes.byref(r), _dev(q, torch.bfloat16, "q"), Hq, float(scale), n_split,
                                _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"), ws,
                                ws_bytes, _stream(stream)), "wm_draft_attn")
    return out, lse


def step_workspace(ring: Ring, n_q_heads: int, n_split: int = 0, device=None, mem: Mem | None = None
                   ) -> torch.Tensor:
    """A workspace for draft_step (or draft_attn_mem) on this ring (split
    partials; never empty)."""
    if mem is None:
        need = workspace_size(WM_OP_DRAFT_STEP, ring.batch, ring.n_kv_heads, n_q_heads, 1, ring.head_dim,
                              ring.sink + ring.window, n_split)
    else:
        need = workspace_size(WM_OP_DRAFT_MEM, ring.batch, ring.n_kv_heads, n_q_heads, 1, ring.head_dim,
                              mem_keys(ring, mem), n_split)
    return torch.empty(need, dtype=torch.uint8, device=device if device is not None else ring.k.device)


def draft_step(ring: Ring, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, scale: float,
               workspace: torch.Tensor, n_split: int = 0, out=None, lse=None, stream=None, mem: Mem | None = None):
    """Fused ring append + draft attention: append (k_new, v_new) [B, Hkv, D]
    at p = n_seen[b] and attend q [B, Hq, D] from position p over the sinks and
    the window, in one attention launch (plus the split merge, which commits
    n_seen).  ``workspace`` comes from step_workspace().  Returns (out bf16,
    lse fp32), bit-identical to ring_append followed by draft_attn (draft_attn_mem
    when ``mem`` is given: the query then also attends to the memory slots)."""
    B, Hq, D = q.shape
    if out is None:
        out = _new_out(q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = _new_out((B, Hq), torch.float32, q.device)
    r = ring.c()
    m = mem.c() if mem is not None else None
    _check(load().wm_draft_step(ctypes.byref(r), ctypes.byref(m) if m is not None else None,
                                _dev(k_new, torch.bfloat16, "k_new"),
                                _dev(v_new, torch.bfloat16, "v_new"), _dev(q, torch.bfloat16, "q"), Hq,
                                float(scale), n_split, _dev(out, torch.bfloat16, "out"),
                                _dev(lse, torch.float32, "lse"), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "wm_draft_step")
    return out, lse


def draft_attn_mem(ring: Ring, mem: Mem, q: torch.Tensor, scale: float, n_split: int = 0, out=None, lse=None,
                   workspace=None, stream=None):
    """Draft attention over the sinks, the window and the memory slots
    0..mem.count[b]-1 (memory-augmented draft); returns (out bf16, lse fp32)."""
    B, Hq, D = q.shape
    if out is None:
        out = _new_out(q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = _new_out((B, Hq), torch.float32, q.device)
    need = workspace_size(WM_OP_DRAFT_MEM, B, ring.n_kv_heads, Hq, 1, D, mem_keys(ring, mem), n_split)
    ws, ws_bytes = _workspace(need, q.device, workspace)
    r, m = ring.c(), mem.c()
    _check(load().wm_draft_attn_mem(ctypes.byref(r), ctypes.byref(m), _dev(q, torch.bfloat16, "q"), Hq,
                                    float(scale), n_split, _dev(out, torch.bfloat16, "out"),
                                    _dev(lse, torch.float32, "lse"), ws, ws_bytes, _stream(stream)),
           "wm_draft_attn_mem")
    return out, lse


def mem_append(mem: Mem, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Materialize one memory slot per sequence (k_new, v_new: [B, Hkv, D] bf16)."""
    m = mem.c()
    _check(load().wm_mem_append(ctypes.byref(m), _dev(k_new, torch.bfloat16, "k_new"),
                                _dev(v_new, torch.bfloat16, "v_new"), _stream(stream)), "wm_mem_append")


def mem_rollback(mem: Mem, new_count: torch.Tensor, stream=None) -> None:
    """Discard memory slots beyond new_count[b] (int64 [B] device tensor)."""
    m = mem.c()
    _check(load().wm_mem_rollback(ctypes.byref(m), _dev(new_count, torch.int64, "new_count"), _stream(stream)),
           "wm_mem_rollback")


def draft_attn_static(ring: Ring, q: torch.Tensor, scale: float, n_split: int = 0, out=None, lse=None,
                      stream=None):
    """Draft attention for callers that cannot allocate device memory: the
    split partials live in a fixed scratch array inside the library
    (STATIC_SCRATCH_BYTES per device) instead of a workspace, so this call
    allocates nothing beyond the outputs it is not given.  Calls that can
    overlap on the GPU share that array and race; keep them on one stream."""
    B, Hq, D = q.shape
    if out is None:
        out = _new_out(q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = _new_out((B, Hq), torch.float32, q.device)
    r = ring.c()
    _check(load().wm_draft_attn_static(ctypes.byref(r), _dev(q, torch.bfloat16, "q"), Hq, float(scale),
                                       n_split, _dev(out, torch.bfloat16, "out"),
                                       _dev(lse, torch.float32, "lse"), _stream(stream)),
           "wm_draft_attn_static")
    return out, lse


def verify_attn(kv: KVCache, q: torch.Tensor, scale: float, n_split: int = 0, out=None, lse=None,
                workspace=None, stream=None):
    """Full-context causal attention of q [B, T, Hq, D]; returns (out bf16, lse fp32)."""
    B, T, Hq, D = q.shape
    if out is None:
        out = _new_out(q.shape, torch.bfloat16, q.device)
    if lse is None:
        lse = _new_out((B, T, Hq), torch.float32, q.device)
    need = workspace_size(WM_OP_VERIFY, B, kv.n_kv_heads, Hq, T, D, kv.capacity, n_split)
    ws, ws_bytes = _workspace(need, q.device, workspace)
    s = kv.c()
    _check(load().wm_verify_attn(ctypes.byref(s), _dev(q, torch.bfloat16, "q"), T, Hq, float(scale),
                                 n_split, _dev(out, torch.bfloat16, "out"), _dev(lse, torch.float32, "lse"),
                                 ws, ws_bytes, _stream(stream)), "wm_verify_attn")
    return out, lse


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out=None, lse=None, stream=None):
    """Merge partials o_parts [rows, n_parts, D] fp32 with lse_parts [rows, n_parts]."""
    rows, n_parts, D = o_parts.shape
    if out is None:
        out = _new_out((rows, D), torch.bfloat16, o_parts.device)
    if lse is None:
        lse = _new_out((rows,), torch.float32, o_parts.device)
    _check(load().wm_lse_merge(_dev(o_parts, torch.float32, "o_parts"), _dev(lse_parts, torch.float32,
                                                                             "lse_parts"),
                               n_parts, rows, D, _dev(out, torch.bfloat16, "out"),
                               _dev(lse, torch.float32, "lse"), _stream(stream)), "wm_lse_merge")
    return out, lse


def set_draft_math(math: int) -> None:
    """The draft kernel's arithmetic for this thread's draft calls:
    WM_DRAFT_MATH_MMA (tensor cores, the default) or WM_DRAFT_MATH_FMA (CUDA
    cores; kept to measure the choice).  See wm_set_draft_math in include/wm_api.h."""
    _check(load().wm_set_draft_math(int(math)), "wm_set_draft_math")


def set_test_stall(stall_tile: int, wait_polls: int = 0) -> None:
    """Tests of the timeout path only: make this thread's attention launches
    stop issuing copies at copy unit ``stall_tile`` of each split and give up a
    wait after ``wait_polls`` polls (``stall_tile=-1`` restores the defaults).
    See wm_set_test_stall in include/wm_api.h."""
    _check(load().wm_set_test_stall(int(stall_tile), int(wait_polls)), "wm_set_test_stall")


def get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error code (0 = none)."""
    code = ctypes.c_int32(0)
    st = load().wm_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (WM_OK, WM_ERR_DEVICE_DATA):
        raise WmError(st, "wm_get_device_error")
    return int(code.value)
