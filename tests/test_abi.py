"""The C ABI library (no GPU needed): it loads, exports every declared symbol,
and rejects invalid arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest
import torch

from speculative_decoding_attention_gb300 import build as wm_build
from speculative_decoding_attention_gb300 import wm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wm_api.h")


@pytest.fixture(scope="module")
def lib():
    wm_build.build()
    return wm.load()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wm_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert set(declared_functions()) == set(wm.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert wm.status_string(wm.WM_OK) == "ok"
    assert "workspace" in wm.status_string(wm.WM_ERR_WORKSPACE)
    assert lib.wm_version() >= 100


def test_invalid_arguments_are_rejected_on_the_host(lib):
    P = ctypes.c_void_p
    assert lib.wm_ring_append(None, P(16), P(16), None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_ring_fill(None, None, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_ring_rollback(None, None, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_draft_attn(None, P(16), 8, 1.0, 0, P(16), None, None, 0, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_verify_attn(None, P(16), 2, 8, 1.0, 0, P(16), None, None, 0, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_lse_merge(None, None, 4, 10, 128, None, None, None) == wm.WM_ERR_INVALID_ARG


def _ring(**over):
    r = wm._Ring()
    r.k, r.v, r.pos_tag, r.n_seen = 1 << 20, 2 << 20, 3 << 20, 4 << 20
    r.batch, r.n_kv_heads, r.head_dim, r.sink, r.window = 1, 2, 128, 4, 256
    for k, v in over.items():
        setattr(r, k, v)
    return r


def _kv(**over):
    s = wm._KV()
    s.k, s.v, s.seq_lens, s.block_table = 1 << 20, 2 << 20, 3 << 20, None
    s.n_cap, s.n_pages, s.page_size, s.max_pages = 4096, 0, 0, 0
    s.batch, s.n_kv_heads, s.head_dim = 1, 2, 128
    for k, v in over.items():
        setattr(s, k, v)
    return s


@pytest.mark.parametrize("over,status", [
    (dict(head_dim=96), wm.WM_ERR_INVALID_ARG),
    (dict(window=0), wm.WM_ERR_INVALID_ARG),
    (dict(sink=-1), wm.WM_ERR_INVALID_ARG),
    (dict(k=(1 << 20) + 2), wm.WM_ERR_INVALID_ARG),
    (dict(batch=0), wm.WM_ERR_INVALID_ARG),
])
def test_bad_ring_shapes(lib, over, status):
    r = _ring(**over)
    P = ctypes.c_void_p
    assert lib.wm_draft_attn(ctypes.byref(r), P(1 << 24), 8, 1.0, 0, P(1 << 25), None, None, 0,
                             None) == status


def test_bad_draft_heads(lib):
    r = _ring()
    P = ctypes.c_void_p
    # 7 query heads do not divide over 2 KV heads
    assert lib.wm_draft_attn(ctypes.byref(r), P(1 << 24), 7, 1.0, 0, P(1 << 25), None, None, 0,
                             None) == wm.WM_ERR_INVALID_ARG
    # non-finite scale
    assert lib.wm_draft_attn(ctypes.byref(r), P(1 << 24), 8, float("nan"), 0, P(1 << 25), None, None,
                             0, None) == wm.WM_ERR_INVALID_ARG


@pytest.mark.parametrize("over,n_q,hq,status", [
    (dict(head_dim=80), 2, 8, wm.WM_ERR_UNSUPPORTED),
    (dict(), 9, 64, wm.WM_ERR_UNSUPPORTED),              # 9 positions x 32 grouped heads > 64 rows
    (dict(), 2, 9, wm.WM_ERR_INVALID_ARG),               # 9 query heads over 2 KV heads
    (dict(n_cap=0), 2, 8, wm.WM_ERR_INVALID_ARG),
    (dict(block_table=5 << 20, page_size=16, max_pages=4, n_pages=8), 2, 8, wm.WM_ERR_UNSUPPORTED),
    (dict(block_table=5 << 20, page_size=64, max_pages=0, n_pages=8), 2, 8, wm.WM_ERR_INVALID_ARG),
    (dict(block_table=5 << 20, page_size=1 << 16, max_pages=1 << 15, n_pages=8), 2, 8,
     wm.WM_ERR_UNSUPPORTED),                                                  # 2^31 positions per sequence
    (dict(n_cap=1 << 31), 2, 8, wm.WM_ERR_UNSUPPORTED),
])
def test_bad_verify_shapes(lib, over, n_q, hq, status):
    s = _kv(**over)
    P = ctypes.c_void_p
    assert lib.wm_verify_attn(ctypes.byref(s), P(1 << 24), n_q, hq, 1.0, 0, P(1 << 25), None, None, 0,
                              None) == status


def test_draft_step_rejects_bad_arguments(lib):
    r = _ring()
    P = ctypes.c_void_p
    q, out, ws = P(1 << 24), P(1 << 25), P(1 << 26)

    def call(k_new=P(1 << 23), v_new=P(3 << 22), hq=8, scale=1.0, ws_ptr=ws, ws_bytes=1 << 20, ring=r):
        # an explicit split count: the plan needs no device query
        return lib.wm_draft_step(ctypes.byref(ring), None, k_new, v_new, q, hq, scale, 4, out, None, ws_ptr,
                                 ws_bytes, None)

    assert lib.wm_draft_step(None, None, P(16), P(16), q, 8, 1.0, 0, out, None, ws, 1 << 20, None) == \
        wm.WM_ERR_INVALID_ARG
    assert call(k_new=None) == wm.WM_ERR_INVALID_ARG
    assert call(v_new=P((1 << 23) + 8)) == wm.WM_ERR_INVALID_ARG      # misaligned
    assert call(hq=7) == wm.WM_ERR_INVALID_ARG                         # 7 heads over 2 KV heads
    assert call(scale=float("inf")) == wm.WM_ERR_INVALID_ARG
    assert call(ring=_ring(head_dim=96)) == wm.WM_ERR_INVALID_ARG
    assert call(ws_ptr=None) == wm.WM_ERR_WORKSPACE
    assert call(ws_ptr=P((1 << 26) + 16)) == wm.WM_ERR_WORKSPACE      # not 256-byte aligned
    assert call(ws_bytes=8) == wm.WM_ERR_WORKSPACE


def _mem(**over):
    m = wm._Mem()
    m.k, m.v, m.count = 5 << 20, 6 << 20, 7 << 20
    m.capacity, m.batch, m.n_kv_heads, m.head_dim = 64, 1, 2, 128
    for k, v in over.items():
        setattr(m, k, v)
    return m


@pytest.mark.parametrize("over", [dict(capacity=0), dict(count=None), dict(head_dim=64), dict(n_kv_heads=4),
                                  dict(batch=2), dict(k=(5 << 20) + 8)])
def test_draft_with_memory_rejects_bad_stores(lib, over):
    r, m = _ring(), _mem(**over)
    P = ctypes.c_void_p
    assert lib.wm_draft_attn_mem(ctypes.byref(r), ctypes.byref(m), P(1 << 24), 8, 1.0, 2, P(1 << 25), None,
                                 P(1 << 26), 1 << 20, None) == wm.WM_ERR_INVALID_ARG


def test_memory_store_calls_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    r = _ring()
    assert lib.wm_draft_attn_mem(ctypes.byref(r), None, P(1 << 24), 8, 1.0, 2, P(1 << 25), None, P(1 << 26),
                                 1 << 20, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_mem_append(None, P(16), P(16), None) == wm.WM_ERR_INVALID_ARG
    m = _mem()
    assert lib.wm_mem_append(ctypes.byref(m), None, P(16), None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_mem_append(ctypes.byref(m), P(16), P(24), None) == wm.WM_ERR_INVALID_ARG  # misaligned
    assert lib.wm_mem_rollback(ctypes.byref(m), None, None) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_mem_rollback(ctypes.byref(_mem(capacity=-1)), P(16), None) == wm.WM_ERR_INVALID_ARG


def test_memory_draft_plans_over_ring_tiles_plus_capacity(lib):
    # the memory region starts at the ring's slots rounded up to whole 64-key tiles
    ring = wm.Ring(None, None, None, None, 4, 4096)
    mem = wm.Mem(torch.empty((1, 2, 300, 8)), None, None)
    assert wm.mem_keys(ring, mem) == 4160 + 300
    assert wm.plan_splits(wm.WM_OP_DRAFT_MEM, 1, 2, 16, 1, 256, 4460, 1000) == 70  # 65 + 5 tiles


def test_too_many_sequence_head_pairs_are_unsupported(lib):
    # 65536 (sequence, KV head) pairs exceed the launch grid: refused on the host
    P = ctypes.c_void_p
    r = _ring(batch=32768, n_kv_heads=2)
    assert lib.wm_draft_attn(ctypes.byref(r), P(1 << 24), 8, 1.0, 4, P(1 << 25), None, P(1 << 26), 1 << 40,
                             None) == wm.WM_ERR_UNSUPPORTED
    s = _kv(batch=65536, n_kv_heads=1)
    assert lib.wm_verify_attn(ctypes.byref(s), P(1 << 24), 2, 8, 1.0, 4, P(1 << 25), None, P(1 << 26), 1 << 40,
                              None) == wm.WM_ERR_UNSUPPORTED


def test_draft_step_workspace(lib):
    # split partials (o then lse) even when unsplit: the merge commits n_seen
    for ns in (1, 4, 5):  # split counts the 65 tiles of 4100 slots divide into exactly
        rows, D = 16, 128
        o = rows * ns * D * 4
        assert wm.workspace_size(wm.WM_OP_DRAFT_STEP, 1, 2, 16, 1, D, 4100, ns) == \
            ((o + 255) // 256) * 256 + rows * ns * 4
    assert wm.plan_splits(wm.WM_OP_DRAFT_STEP, 1, 2, 16, 1, 256, 4100, 1000) == 65  # one tile per split at most
    # up to 8 query heads per KV head the draft splits are balanced (any count up
    # to the tile count); more rows keep uniform splits of whole tiles
    assert wm.plan_splits(wm.WM_OP_DRAFT_STEP, 1, 2, 16, 1, 128, 4100, 30) == 30
    assert wm.plan_splits(wm.WM_OP_DRAFT_STEP, 1, 2, 32, 1, 128, 4100, 30) == 22  # 3 tiles per split
    assert wm.plan_splits(wm.WM_OP_DRAFT_STEP, 1, 2, 16, 2, 256, 4100, 4) == 0      # one query position only


def test_workspace_size_with_explicit_splits(lib):
    # Explicit split counts need no device query.
    assert wm.workspace_size(wm.WM_OP_VERIFY, 1, 2, 16, 4, 256, 1 << 20, 1) == 0
    rows, ns, D = 1 * 4 * 16, 8, 256
    o = rows * ns * D * 4
    assert wm.workspace_size(wm.WM_OP_VERIFY, 1, 2, 16, 4, 256, 1 << 20, ns) == \
        ((o + 255) // 256) * 256 + rows * ns * 4
    # capped at one key tile per split: the draft kernel's 64-key tiles, the
    # verify kernel's 128-key tiles (tensor-core kernel) at head_dim 128/256
    assert wm.plan_splits(wm.WM_OP_DRAFT, 1, 2, 16, 1, 256, 4100, 1000) == 65
    assert wm.plan_splits(wm.WM_OP_VERIFY, 1, 2, 16, 1, 256, 4100, 1000) == 33
    assert wm.plan_splits(wm.WM_OP_VERIFY, 1, 2, 16, 1, 64, 4100, 1000) == 65
    with pytest.raises(wm.WmError):
        wm.workspace_size(wm.WM_OP_VERIFY, 1, 2, 16, 4, 96, 1 << 20, 0)


def _needed_libraries(path: str) -> list[str]:
    """DT_NEEDED entries of a 64-bit little-endian ELF shared object (the
    dynamic section's library names; nothing else of the file is read)."""
    import struct

    with open(path, "rb") as f:
        ident = f.read(64)
        assert ident[:4] == b"\x7fELF" and ident[4] == 2 and ident[5] == 1
        shoff, = struct.unpack_from("<Q", ident, 0x28)
        shentsize, shnum = struct.unpack_from("<HH", ident, 0x3A)
        f.seek(shoff)
        sections = [struct.unpack("<IIQQQQIIQQ", f.read(shentsize)) for _ in range(shnum)]
        dyn = next(sec for sec in sections if sec[1] == 6)  # SHT_DYNAMIC
        strtab = sections[dyn[6]]                             # its sh_link: the string table
        f.seek(strtab[4])
        strings = f.read(strtab[5])
        f.seek(dyn[4])
        entries = [struct.unpack("<qQ", f.read(16)) for _ in range(dyn[5] // 16)]
    names = []
    for tag, val in entries:
        if tag == 1:  # DT_NEEDED
            names.append(strings[val:strings.index(b"\0", val)].decode())
    return names


def test_library_has_no_torch_dependency(lib):
    # The C ABI is plain pointers and sizes: the shared object links no torch.
    needed = _needed_libraries(wm.library_path())
    assert needed and not any("torch" in n or "c10" in n for n in needed), needed


def test_split_calls_without_enough_workspace(lib):
    """Split draft and verify calls check their workspace on the host: missing,
    misaligned or short -> WM_ERR_WORKSPACE, nothing launched (no device here)."""
    P = ctypes.c_void_p
    q, out = P(1 << 24), P(1 << 25)
    need_v = wm.workspace_size(wm.WM_OP_VERIFY, 1, 2, 8, 2, 128, 4096, 4)
    need_d = wm.workspace_size(wm.WM_OP_DRAFT, 1, 2, 8, 1, 128, 260, 4)
    assert need_v > 0 and need_d > 0
    s, r = _kv(), _ring()
    for ws, nbytes in [(None, need_v), (P((1 << 26) + 16), need_v), (P(1 << 26), need_v - 1)]:
        assert lib.wm_verify_attn(ctypes.byref(s), q, 2, 8, 1.0, 4, out, None, ws, nbytes, None) == \
            wm.WM_ERR_WORKSPACE
    for ws, nbytes in [(None, need_d), (P((1 << 26) + 16), need_d), (P(1 << 26), need_d - 1)]:
        assert lib.wm_draft_attn(ctypes.byref(r), q, 8, 1.0, 4, out, None, ws, nbytes, None) == \
            wm.WM_ERR_WORKSPACE


def test_static_scratch_draft_reports_bad_arguments_first(lib):
    """wm_draft_attn_static runs wm_draft_attn's host checks before it looks
    at its scratch size: a bad argument is WM_ERR_INVALID_ARG from both, even
    when the plan would also not fit the scratch array."""
    P = ctypes.c_void_p
    big = _ring(batch=64, n_kv_heads=8, window=8192, sink=16)  # a plan far beyond the scratch array
    cases = [
        (big, 8 * 8 + 3, 1.0, P(16), P(16)),          # query heads not a multiple of the KV heads
        (big, 64, float("nan"), P(16), P(16)),         # non-finite scale
        (big, 64, 1.0, P(17), P(16)),                  # misaligned q
        (big, 64, 1.0, P(16), P(18)),                  # misaligned out
        (_ring(batch=64, n_kv_heads=8, window=0), 64, 1.0, P(16), P(16)),  # empty window
        (_ring(batch=64, n_kv_heads=8, head_dim=96), 64, 1.0, P(16), P(16)),
    ]
    for r, hq, scale, q, out in cases:
        a = lib.wm_draft_attn(ctypes.byref(r), q, hq, scale, 0, out, None, None, 0, None)
        s = lib.wm_draft_attn_static(ctypes.byref(r), q, hq, scale, 0, out, None, None)
        assert a == wm.WM_ERR_INVALID_ARG and s == wm.WM_ERR_INVALID_ARG, (hq, scale, a, s)


def test_test_stall_hook_rejects_bad_settings(lib):
    assert lib.wm_set_test_stall(-2, 100) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_set_test_stall(0, 0) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_set_test_stall(3, 100) == wm.WM_OK
    assert lib.wm_set_test_stall(-1, 0) == wm.WM_OK


def test_draft_math_setting(lib):
    assert lib.wm_set_draft_math(2) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_set_draft_math(-1) == wm.WM_ERR_INVALID_ARG
    assert lib.wm_set_draft_math(wm.WM_DRAFT_MATH_FMA) == wm.WM_OK
    assert lib.wm_set_draft_math(wm.WM_DRAFT_MATH_MMA) == wm.WM_OK


def test_verify_persistent_selection(lib):
    """The persistent verify serves batches of several sequences left to the
    library at head_dim 128 (<= 64 rows) and 256 (<= 32 rows), up to 2^30 key
    tiles per call; everything else runs the split plan.  Without a device the
    CTA count is one per SM of an unknown device: 1."""
    vp = wm.verify_persistent
    assert vp(2, 2, 8, 3, 128, 4096) > 0
    assert vp(2, 8, 64, 8, 128, 4096) > 0      # 64 rows
    assert vp(2, 2, 16, 4, 256, 4096) > 0      # 32 rows at head_dim 256
    assert vp(2, 2, 16, 5, 256, 4096) == 0     # 40 rows at head_dim 256: V in half tiles
    assert vp(1, 2, 8, 3, 128, 4096) == 0      # one sequence: the split plan is balanced already
    assert vp(2, 2, 8, 3, 128, 4096, 4) == 0   # explicit split count
    assert vp(2, 2, 8, 3, 64, 4096) == 0       # head_dim 64: mma.sync kernel
    assert vp(4, 8, 32, 3, 128, 1 << 25) > 0   # 4 x 8 x 2^18 = 2^23 key tiles
    assert vp(4096, 16, 64, 3, 128, 1 << 31) == 0  # 2^12 x 2^4 x 2^24 tiles > 2^30
    assert vp(2, 3, 8, 3, 128, 4096) == 0      # n_q_heads not a multiple of n_kv_heads
    assert vp(0, 2, 8, 3, 128, 4096) == 0


def test_verify_persistent_workspace_layout(lib):
    """Workspace of the persistent verify: partials of n_cta + units - 1
    segments (rows x head_dim fp32, then rows fp32), the schedule (batch + 3
    int64) and the CTAs' first tiles (16 bytes each), each part 256-byte
    aligned, and WM_ERR_WORKSPACE one byte short."""
    up = lambda x: (x + 255) // 256 * 256
    B, Hkv, G, T, D = 5, 2, 4, 3, 128
    n_cta = wm.verify_persistent(B, Hkv, Hkv * G, T, D, 4096)
    assert n_cta >= 1
    assert wm.plan_splits(wm.WM_OP_VERIFY, B, Hkv, Hkv * G, T, D, 4096, 0) == n_cta
    rows, seg = T * G, n_cta + B * Hkv - 1
    want = up(seg * rows * D * 4) + up(seg * rows * 4) + up((B + 3) * 8) + n_cta * 16
    need = wm.workspace_size(wm.WM_OP_VERIFY, B, Hkv, Hkv * G, T, D, 4096, 0)
    assert need == want
    P = ctypes.c_void_p
    s = _kv(batch=B, n_kv_heads=Hkv)
    assert lib.wm_verify_attn(ctypes.byref(s), P(1 << 24), T, Hkv * G, 1.0, 0, P(1 << 25), None, P(1 << 26),
                              need - 1, None) == wm.WM_ERR_WORKSPACE
