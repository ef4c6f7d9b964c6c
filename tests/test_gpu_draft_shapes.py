"""Shapes of the keys-as-M draft kernel that the workloads do not reach:
every group size from 1 to 8 query heads per KV head (the MMA's N = 8 holds
the real rows, the rest padding), rings whose slot count is not a multiple
of the 64-key tile, split counts beyond the tile count, the appended slot on
the first and last key of a tile, and splits made only of memory slots."""
import math

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7, 8])
def test_every_group_size(D, G):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(1100 + 10 * G + D)
    B, Hkv, S, W = 2, 3, 3, 130  # 133 slots: three tiles, the last one 5 keys
    n = [400, 177]
    hk, hv = rand_bf16((B, Hkv, 402, D), gen, dev), rand_bf16((B, Hkv, 402, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor(n, device=dev)))
    hist = oracle_kv(hk, hv)
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    for ns in (0, 2, 100):  # 100: more splits than tiles, clamped to one tile each
        out, lse = wm.draft_attn(ring, q, 1.0, n_split=ns)
        ref, ref_lse = oracle.draft(hist, q.cpu(), [x - 1 for x in n], S, W, 1.0)
        assert_close(f"draft D={D} G={G} ns={ns}", out, lse, ref, ref_lse)
    ws = wm.step_workspace(ring, Hkv * G, 2)
    for j in range(2):
        kn = torch.stack([hk[b, :, n[b] + j] for b in range(B)]).contiguous()
        vn = torch.stack([hv[b, :, n[b] + j] for b in range(B)]).contiguous()
        q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
        out, lse = wm.draft_step(ring, kn, vn, q, 1.0, ws, n_split=2)
        ref, ref_lse = oracle.draft(hist, q.cpu(), [x + j for x in n], S, W, 1.0)
        assert_close(f"fused step {j} D={D} G={G}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("target_slot", [0, 63, 64, 127])
def test_appended_slot_on_tile_edges(target_slot):
    """With S = 0 and W = 128 the slot of position p is p mod 128: fill to
    the position whose slot is a tile's first or last key, then append it in
    the fused step, one split per tile and a single split."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(1200 + target_slot)
    B, Hkv, G, D, S, W = 1, 2, 8, 128, 0, 128
    p = 3 * W + target_slot
    hk, hv = rand_bf16((B, Hkv, p + 1, D), gen, dev), rand_bf16((B, Hkv, p + 1, D), gen, dev)
    hist = oracle_kv(hk, hv)
    for ns in (1, 2):
        ring = wm.Ring.create(B, Hkv, D, S, W, dev)
        wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor([p], device=dev)))
        ws = wm.step_workspace(ring, Hkv * G, ns)
        q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
        out, lse = wm.draft_step(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous(), q, 1.0, ws, n_split=ns)
        ref, ref_lse = oracle.draft(hist, q.cpu(), [p], S, W, 1.0)
        assert_close(f"slot {target_slot} ns={ns}", out, lse, ref, ref_lse)
        torch.cuda.synchronize()
        assert int(ring.pos_tag[0, target_slot]) == p and int(ring.n_seen[0]) == p + 1
        assert torch.equal(ring.k[0, :, target_slot], hk[0, :, p]) and torch.equal(ring.v[0, :, target_slot], hv[0, :, p])
    assert wm.get_device_error() == 0


def test_split_of_memory_slots_only():
    """Enough splits that the last ones cover only memory slots (past the
    ring's tile-rounded slots), with a partly filled memory store."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(1300)
    B, Hkv, G, D, S, W, cap = 2, 2, 8, 128, 4, 60, 300  # ring: one tile; memory: 5 tiles
    n = [500, 90]
    hk, hv = rand_bf16((B, Hkv, 500, D), gen, dev), rand_bf16((B, Hkv, 500, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor(n, device=dev)))
    mem = wm.Mem.create(B, Hkv, D, cap, dev)
    mem.k.copy_(rand_bf16(mem.k.shape, gen, dev))
    mem.v.copy_(rand_bf16(mem.v.shape, gen, dev))
    counts = [300, 130]
    mem.count.copy_(torch.tensor(counts, dtype=torch.int64, device=dev))
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    for ns in (0, 3, 6):
        out, lse = wm.draft_attn_mem(ring, mem, q, 1.0, n_split=ns)
        ref, ref_lse = oracle.draft_mem(oracle_kv(hk, hv), oracle_kv(mem.k, mem.v), counts, q.cpu(),
                                        [x - 1 for x in n], S, W, 1.0)
        assert_close(f"memory-only splits ns={ns}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
