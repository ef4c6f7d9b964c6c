"""The bounded-wait timeout path of the attention kernels, made reachable on
purpose: a test hook (wm_set_test_stall) makes the producer warp stop issuing
copies at a given copy unit and shortens every wait to a few thousand polls.
The consumer's wait for the tile that never comes must give up, record
WM_DEVERR_TIMEOUT, and let the kernel return; the next normal call must match
the oracle.  Nothing faults or hangs: the copies that were issued are waited
for (bounded) before the CTA exits."""
import math

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu

WM_DEVERR_TIMEOUT = 3
POLLS = 4000


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


def _stalled(call, stall_tile):
    wm.set_test_stall(stall_tile, POLLS)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        wm.set_test_stall(-1)


@pytest.mark.parametrize("G", [8, 16])  # 8 rows: keys-as-M draft kernel; 16: row-major mma.sync kernel
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("stall_tile", [0, 1, 3])
def test_draft_wait_times_out_then_next_call_is_clean(G, D, stall_tile):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(900 + G + D + stall_tile)
    B, Hkv, S, W, n = 1, 2, 4, 600, 900
    k, v = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(k, v, torch.tensor([n], device=dev)))
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    torch.cuda.synchronize()
    assert wm.get_device_error() == 0
    # one split: the CTA streams all 10 tiles of the ring, so tile 1 and 3 exist
    _stalled(lambda: wm.draft_attn(ring, q, 1.0, n_split=1), stall_tile)
    assert wm.get_device_error() == WM_DEVERR_TIMEOUT
    out, lse = wm.draft_attn(ring, q, 1.0)
    ref, ref_lse = oracle.draft(oracle_kv(k, v), q.cpu(), [n - 1], S, W, 1.0)
    assert_close(f"after the timeout G={G} D={D}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_fused_step_wait_times_out_then_next_step_is_clean():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(950)
    B, Hkv, G, D, S, W, n = 2, 2, 8, 128, 4, 500, 800
    k, v = rand_bf16((B, Hkv, n + 1, D), gen, dev), rand_bf16((B, Hkv, n + 1, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(k, v, torch.tensor([n, n], device=dev)))
    saved = [t.clone() for t in (ring.k, ring.v, ring.pos_tag, ring.n_seen)]
    ws = wm.step_workspace(ring, Hkv * G, n_split=2)
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    kn, vn = k[:, :, n].contiguous(), v[:, :, n].contiguous()
    _stalled(lambda: wm.draft_step(ring, kn, vn, q, 1.0, ws, n_split=2), 2)
    assert wm.get_device_error() == WM_DEVERR_TIMEOUT
    for t, c in zip((ring.k, ring.v, ring.pos_tag, ring.n_seen), saved):
        t.copy_(c)
    out, lse = wm.draft_step(ring, kn, vn, q, 1.0, ws, n_split=2)
    ref, ref_lse = oracle.draft(oracle_kv(k, v), q.cpu(), [n, n], S, W, 1.0)
    assert_close("fused step after the timeout", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("stall_tile", [0, 2])
def test_verify_head_dim_64_wait_times_out_then_next_call_is_clean(stall_tile):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(970 + stall_tile)
    B, Hkv, G, T, D, n = 1, 2, 4, 3, 64, 700
    k, v = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor([n], device=dev))
    q = rand_bf16((B, T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    _stalled(lambda: wm.verify_attn(kv, q, 1.0, n_split=1), stall_tile)
    assert wm.get_device_error() == WM_DEVERR_TIMEOUT
    out, lse = wm.verify_attn(kv, q, 1.0)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), [n], 1.0)
    assert_close("verify after the timeout", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D,G,T", [(128, 4, 4), (128, 8, 4), (128, 8, 5), (256, 8, 4), (256, 8, 6)])
@pytest.mark.parametrize("stall_unit", [0, 1, 3, 6])
def test_tcgen05_verify_wait_times_out_then_next_call_is_clean(D, G, T, stall_unit):
    """The tcgen05 verify kernel (16-64 rows; at head_dim 256 with more than 32
    rows V is staged in 64-key halves by a second producer warp): the MMA
    issuer's and the softmax warps' bounded waits give up, the kernel drains
    its copies, frees its tensor memory and returns."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(990 + D + G + T + stall_unit)
    B, Hkv, n = 1, 2, 1000  # 8 key tiles of 128 in one split
    k, v = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor([n], device=dev))
    q = rand_bf16((B, T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    _stalled(lambda: wm.verify_attn(kv, q, 1.0, n_split=1), stall_unit)
    assert wm.get_device_error() == WM_DEVERR_TIMEOUT
    out, lse = wm.verify_attn(kv, q, 1.0)
    ref, ref_lse = oracle.verify(oracle_kv(k, v), q.cpu(), [n], 1.0)
    assert_close(f"tcgen05 verify after the timeout D={D} G={G} T={T}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
