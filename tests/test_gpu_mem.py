"""Memory-augmented draft on the GPU: memory slots (materialized K/V that the
draft query attends to together with the sinks and the window) against the
oracle, the slot store bit-exact, and the fused step with memory bit-identical
to ring append + memory draft attention.
"""
import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def rand_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device).to(torch.bfloat16)


def build(B, Hkv, D, S, W, lens, cap, counts, seed, extra=0):
    """History of max(lens) + extra positions filled into a ring; a memory store
    with counts[b] slots materialized through wm_mem_append."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(seed)
    n = max(lens) + extra
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    mk, mv = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    mem = wm.Mem.create(B, Hkv, D, cap, dev)
    for i in range(max(counts)):
        wm.mem_append(mem, mk[:, :, i].contiguous(), mv[:, :, i].contiguous())
    mem.count.copy_(torch.tensor(counts, device=dev))  # per-sequence counts (rows beyond stay written)
    return dev, gen, hk, hv, ring, mk, mv, mem


CASES = [
    # B, Hkv, G, D, S, W, lens, cap, counts, n_split
    (2, 2, 8, 128, 4, 256, [1000, 300], 40, [40, 7], 0),
    (1, 2, 8, 256, 4, 4096, [20000], 300, [257], 0),      # the 1M hybrid ring with 257 slots
    (1, 1, 64, 64, 0, 100, [37], 70, [65], 0),            # 64 rows; ring not full; slots span 2 tiles
    (2, 2, 4, 128, 16, 500, [900, 2], 64, [0, 64], 3),    # no slot for b=0, a full store for b=1
    (3, 2, 4, 64, 4, 60, [63, 200, 5], 10, [1, 10, 3], 1),
]


@pytest.mark.parametrize("B,Hkv,G,D,S,W,lens,cap,counts,n_split", CASES)
def test_memory_draft_matches_oracle(B, Hkv, G, D, S, W, lens, cap, counts, n_split):
    dev, gen, hk, hv, ring, mk, mv, mem = build(B, Hkv, D, S, W, lens, cap, counts, seed=40 + D + cap)
    q = rand_bf16((B, Hkv * G, D), gen, dev)
    scale = D ** -0.5
    out, lse = wm.draft_attn_mem(ring, mem, q, scale, n_split=n_split)
    torch.cuda.synchronize()
    assert wm.get_device_error() == 0
    ref, ref_lse = oracle.draft_mem(oracle_kv(hk, hv), oracle_kv(mk, mv), counts, q.cpu(), [n - 1 for n in lens],
                                    S, W, scale)
    assert_close("memory draft", out, lse, ref, ref_lse)


def test_memory_slot_store_appends_and_rolls_back_bit_exact():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(41)
    B, Hkv, D, cap = 3, 2, 128, 5
    mem = wm.Mem.create(B, Hkv, D, cap, dev)
    rows = [(rand_bf16((B, Hkv, D), gen, dev), rand_bf16((B, Hkv, D), gen, dev)) for _ in range(cap + 1)]
    for i in range(cap):
        wm.mem_append(mem, *rows[i])
    assert mem.count.tolist() == [cap] * B
    for i in range(cap):
        assert torch.equal(mem.k[:, :, i].view(torch.int16), rows[i][0].view(torch.int16))
        assert torch.equal(mem.v[:, :, i].view(torch.int16), rows[i][1].view(torch.int16))
    assert wm.get_device_error() == 0
    before = mem.k.clone()
    wm.mem_append(mem, *rows[cap])  # full store: recorded, nothing written
    torch.cuda.synchronize()
    assert wm.get_device_error() == 1 and mem.count.tolist() == [cap] * B
    assert torch.equal(mem.k.view(torch.int16), before.view(torch.int16))
    wm.mem_rollback(mem, torch.tensor([2, 7, 0], device=dev))
    assert mem.count.tolist() == [2, cap, 0]
    wm.mem_append(mem, *rows[0])
    assert mem.count.tolist() == [3, cap, 1]
    assert torch.equal(mem.k[0, :, 2].view(torch.int16), rows[0][0][0].view(torch.int16))
    assert wm.get_device_error() == 1  # the one full sequence (b=1)


@pytest.mark.parametrize("D,S,W,cap,counts,n_split", [(128, 4, 256, 40, [40, 3], 0), (256, 4, 4096, 300, [257, 0], 0),
                                                      (64, 0, 60, 9, [2, 9], 2)])
def test_fused_step_with_memory(D, S, W, cap, counts, n_split):
    """Fused step with memory: matches the oracle, and is bit-identical to
    ring append followed by the memory draft attention."""
    B, Hkv, G, lens, steps = 2, 2, 8, [3 * (S + W) + 5, S + W // 2], 3
    dev, gen, hk, hv, ring, mk, mv, mem = build(B, Hkv, D, S, W, lens, cap, counts, seed=50 + D, extra=steps)
    two = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(two, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    ws = wm.step_workspace(ring, Hkv * G, n_split, mem=mem)
    scale = D ** -0.5
    hist, mhist = oracle_kv(hk, hv), oracle_kv(mk, mv)
    for j in range(steps):
        q = rand_bf16((B, Hkv * G, D), gen, dev)
        kn = torch.stack([hk[b, :, n + j] for b, n in enumerate(lens)]).contiguous()
        vn = torch.stack([hv[b, :, n + j] for b, n in enumerate(lens)]).contiguous()
        out, lse = wm.draft_step(ring, kn, vn, q, scale, ws, n_split=n_split, mem=mem)
        wm.ring_append(two, kn, vn)
        out2, lse2 = wm.draft_attn_mem(two, mem, q, scale, n_split=n_split)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
        ref, ref_lse = oracle.draft_mem(hist, mhist, counts, q.cpu(), [n + j for n in lens], S, W, scale)
        assert_close(f"fused step {j} with memory", out, lse, ref, ref_lse)
    assert torch.equal(ring.pos_tag, two.pos_tag) and torch.equal(ring.n_seen, two.n_seen)
    assert wm.get_device_error() == 0


def test_memory_count_beyond_capacity_is_clamped_and_reported():
    B, Hkv, G, D, S, W, lens, cap = 1, 2, 4, 128, 4, 128, [500], 8
    dev, gen, hk, hv, ring, mk, mv, mem = build(B, Hkv, D, S, W, lens, cap, [cap], seed=60)
    q = rand_bf16((B, Hkv * G, D), gen, dev)
    ref_out, ref_lse = wm.draft_attn_mem(ring, mem, q, 0.1)
    ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
    mem.count.fill_(cap + 5)
    out, lse = wm.draft_attn_mem(ring, mem, q, 0.1)
    torch.cuda.synchronize()
    assert wm.get_device_error() == 1
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)) and torch.equal(lse, ref_lse)


def test_memory_rollback_then_draft_sees_the_kept_slots():
    """After a rejection the slots materialized past the accepted prefix are
    discarded: the draft attends to slots 0..new_count-1 only."""
    B, Hkv, G, D, S, W, lens, cap = 2, 2, 4, 128, 4, 128, [700, 300], 12
    dev, gen, hk, hv, ring, mk, mv, mem = build(B, Hkv, D, S, W, lens, cap, [12, 9], seed=61)
    wm.mem_rollback(mem, torch.tensor([5, 9], device=dev))
    assert mem.count.tolist() == [5, 9]
    q = rand_bf16((B, Hkv * G, D), gen, dev)
    out, lse = wm.draft_attn_mem(ring, mem, q, D ** -0.5)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.draft_mem(oracle_kv(hk, hv), oracle_kv(mk, mv), [5, 9], q.cpu(), [n - 1 for n in lens],
                                    S, W, D ** -0.5)
    assert_close("after memory rollback", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


def test_fused_step_with_memory_in_a_graph():
    """A captured fused step with memory, replayed: each replay appends the next
    position to the ring, a slot is materialized between replays."""
    B, Hkv, G, D, S, W, lens, cap, steps = 1, 2, 8, 128, 4, 256, [1500], 8, 4
    dev, gen, hk, hv, ring, mk, mv, mem = build(B, Hkv, D, S, W, lens, cap, [2], seed=62, extra=steps)
    ws = wm.step_workspace(ring, Hkv * G, mem=mem)
    kn = torch.stack([hk[b, :, n] for b, n in enumerate(lens)]).contiguous()
    vn = torch.stack([hv[b, :, n] for b, n in enumerate(lens)]).contiguous()
    q = rand_bf16((B, Hkv * G, D), gen, dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hkv * G), float("nan"), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        wm.draft_step(ring, kn, vn, q, D ** -0.5, ws, out=out, lse=lse, stream=side, mem=mem)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    hist, mhist = oracle_kv(hk, hv), oracle_kv(mk, mv)
    ref, ref_lse = oracle.draft_mem(hist, mhist, [2], q.cpu(), [lens[0]], S, W, D ** -0.5)
    assert_close("eager", out, lse, ref, ref_lse)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wm.draft_step(ring, kn, vn, q, D ** -0.5, ws, out=out, lse=lse, stream=torch.cuda.current_stream(), mem=mem)
    for j in range(1, steps):
        wm.mem_append(mem, mk[:, :, 1 + j].contiguous(), mv[:, :, 1 + j].contiguous())
        kn.copy_(torch.stack([hk[b, :, n + j] for b, n in enumerate(lens)]))
        vn.copy_(torch.stack([hv[b, :, n + j] for b, n in enumerate(lens)]))
        q.copy_(rand_bf16((B, Hkv * G, D), gen, dev))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle.draft_mem(hist, mhist, [2 + j], q.cpu(), [lens[0] + j], S, W, D ** -0.5)
        assert_close(f"replay {j}", out, lse, ref, ref_lse)
    assert ring.n_seen.tolist() == [lens[0] + steps] and mem.count.tolist() == [2 + steps - 1]
    assert wm.get_device_error() == 0
