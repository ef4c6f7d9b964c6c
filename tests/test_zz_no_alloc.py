"""wm_draft_attn_static: draft attention for callers that cannot allocate.

Some callers of the draft step have no way to hand the library a workspace:
runtimes that reserve all device memory at start-up and refuse later
allocations, or plugins whose host framework owns the allocator.  For them the
library keeps the split partials in a scratch array of its own.  This test
calls that entry point through the C ABI twice in a row and checks each result
against the workspace-taking wm_draft_attn, within the parity tolerance of the
other GPU tests; it also checks that an oversized request is refused.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test already.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from speculative_decoding_attention_gb300 import wm

from parity import ATOL, LSE_TOL, RTOL, gpu

pytestmark = pytest.mark.gpu


def _close(a_out, a_lse, b_out, b_lse):
    a, b = a_out.float().cpu().numpy(), b_out.float().cpu().numpy()
    assert np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b))
    la, lb = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    assert np.array_equal(np.isfinite(la), np.isfinite(lb))
    fin = np.isfinite(lb)
    assert np.all(np.abs(la[fin] - lb[fin]) <= LSE_TOL)


def test_static_scratch_draft_matches_workspace_draft_twice():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(77)
    B, Hkv, G, D, S, W = 2, 2, 8, 256, 4, 4096
    n = 6000
    hk = torch.randn((B, Hkv, n, D), generator=gen, device=dev).to(torch.bfloat16)
    hv = torch.randn((B, Hkv, n, D), generator=gen, device=dev).to(torch.bfloat16)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.full((B,), n, dtype=torch.int64, device=dev)))
    splits = wm.plan_splits(wm.WM_OP_DRAFT, B, Hkv, Hkv * G, 1, D, S + W)
    assert splits > 1  # the scratch array is really used
    assert wm.workspace_size(wm.WM_OP_DRAFT, B, Hkv, Hkv * G, 1, D, S + W) <= wm.STATIC_SCRATCH_BYTES
    for call in range(2):
        q = (torch.randn((B, Hkv * G, D), generator=gen, device=dev) / math.sqrt(D)).to(torch.bfloat16)
        ref_out, ref_lse = wm.draft_attn(ring, q, 1.0)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hkv * G), float("nan"), dtype=torch.float32, device=dev)
        r = ring.c()
        st = wm.load().wm_draft_attn_static(ctypes.byref(r), ctypes.c_void_p(q.data_ptr()), Hkv * G, 1.0, 0,
                                            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == wm.WM_OK, wm.status_string(st)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
    assert wm.get_device_error() == 0


def test_static_scratch_refuses_requests_beyond_its_size():
    dev = gpu()
    B, Hkv, G, D, S, W = 64, 8, 8, 256, 4, 60000
    n_split = 64
    need = wm.workspace_size(wm.WM_OP_DRAFT, B, Hkv, Hkv * G, 1, D, S + W, n_split)
    assert need > wm.STATIC_SCRATCH_BYTES
    r = wm._Ring()
    r.k, r.v, r.pos_tag, r.n_seen = 1 << 20, 2 << 20, 3 << 20, 4 << 20  # never dereferenced
    r.batch, r.n_kv_heads, r.head_dim, r.sink, r.window = B, Hkv, D, S, W
    st = wm.load().wm_draft_attn_static(ctypes.byref(r), ctypes.c_void_p(1 << 24), Hkv * G, 1.0, n_split,
                                        ctypes.c_void_p(1 << 25), None, None)
    assert st == wm.WM_ERR_WORKSPACE
    del dev
