"""The fused draft step (ring append folded into the draft attention launch)
against the oracle, and its ring state against the slot rule.

For every step j the query sits at p = n_seen[b] (the position being
appended); the oracle evaluates sink + window attention from the draft KV
history by absolute position, which already holds the appended entry at p.
The ring after the steps must hold exactly the sinks and the last W positions
with their K/V bytes (bit-exact) and n_seen must have advanced by the step
count.  Against the unfused calls (ring append, then draft attention with the
same split plan) everything is bit-identical.
"""
import pytest
import torch

import oracle
from oracle.ring_model import held_after
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def slot_rule(p, S, W):
    return p if p < S else S + (p - S) % W


def rand_bf16(shape, gen, device, scale=1.0):
    return (torch.randn(shape, generator=gen, device=device) * scale).to(torch.bfloat16)


def gather_pos(h, lens, j):
    """[B, Hkv, D] rows of the history at position lens[b] + j of each sequence."""
    return torch.stack([h[b, :, n + j] for b, n in enumerate(lens)]).contiguous()


def check_ring(ring, hk, hv, lens_now):
    tags = ring.pos_tag.cpu()
    for b, n in enumerate(lens_now):
        t = tags[b]
        assert sorted(int(x) for x in t[t >= 0]) == held_after(ring.sink, ring.window, n)
        for s in torch.nonzero(t >= 0).flatten().tolist():
            p = int(t[s])
            assert s == slot_rule(p, ring.sink, ring.window)
            assert torch.equal(ring.k[b, :, s].view(torch.int16), hk[b, :, p].view(torch.int16))
            assert torch.equal(ring.v[b, :, s].view(torch.int16), hv[b, :, p].view(torch.int16))
    assert ring.n_seen.tolist() == list(lens_now)


def setup(B, Hkv, G, D, S, W, lens, steps, seed):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(seed)
    cap = max(lens) + steps
    hk, hv = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    qs = [rand_bf16((B, Hkv * G, D), gen, dev) for _ in range(steps)]
    return dev, hk, hv, ring, qs


CASES = [
    # B, Hkv, G, D, S, W, lens, steps, n_split
    (1, 2, 4, 128, 4, 256, [4096], 3, 0),                # the tiny workload's shape
    (1, 2, 8, 256, 4, 4096, [5000], 3, 0),               # the 1M hybrid ring
    (2, 8, 8, 128, 16, 8192, [9000, 20000], 2, 0),       # the NoPE ring
    (3, 2, 32, 128, 16, 512, [0, 300, 2000], 4, 0),      # ragged, 32 rows, one empty history
    (1, 1, 64, 64, 0, 100, [37], 5, 0),                  # 64 rows, no sink, ring not yet full
    (2, 2, 4, 64, 4, 60, [63, 10], 3, 1),                # unsplit; b=0 wraps at the first step
    (2, 2, 4, 64, 4, 200, [203, 10], 3, 3),              # 3 splits; b=0 wraps
    (2, 2, 4, 256, 4, 400, [700, 10], 3, 6),             # ragged last split
    (2, 2, 4, 128, 4, 1020, [3000, 1500], 3, 16),
    (1, 2, 8, 128, 4, 200, [500], 2, 100),               # more splits requested than tiles
    (1, 2, 8, 128, 4, 2000, [5000], 2, 1),               # a split longer than the staged tags
    (2, 2, 4, 256, 4, 3000, [3500, 900], 2, 2),          # the same at head_dim 256, two splits
]


@pytest.mark.parametrize("B,Hkv,G,D,S,W,lens,steps,n_split", CASES)
def test_step_matches_oracle_and_ring(B, Hkv, G, D, S, W, lens, steps, n_split):
    dev, hk, hv, ring, qs = setup(B, Hkv, G, D, S, W, lens, steps, seed=100 + D + S + W + n_split)
    scale = D ** -0.5
    ws = wm.step_workspace(ring, Hkv * G, n_split)
    hist = oracle_kv(hk, hv)
    for j in range(steps):
        out, lse = wm.draft_step(ring, gather_pos(hk, lens, j), gather_pos(hv, lens, j), qs[j], scale, ws,
                                 n_split=n_split)
        torch.cuda.synchronize()
        ref, ref_lse = oracle.draft(hist, qs[j].cpu(), [n + j for n in lens], S, W, scale)
        assert_close(f"step {j}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
    check_ring(ring, hk, hv, [n + steps for n in lens])


@pytest.mark.parametrize("D,S,W,n_split", [(128, 4, 256, 0), (256, 4, 4096, 0), (64, 4, 60, 6), (128, 16, 500, 1),
                                           (256, 0, 300, 2)])
def test_step_equals_append_then_draft(D, S, W, n_split):
    """Bit-identical to wm_ring_append followed by wm_draft_attn with the same
    split count: ring bytes, tags, n_seen, out and lse."""
    B, Hkv, G, lens, steps = 2, 2, 8, [3 * (S + W) + 5, S + W // 2], 3
    dev, hk, hv, ring, qs = setup(B, Hkv, G, D, S, W, lens, steps, seed=7 + D)
    two = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(two, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    ws = wm.step_workspace(ring, Hkv * G, n_split)
    scale = D ** -0.5
    for j in range(steps):
        kn, vn = gather_pos(hk, lens, j), gather_pos(hv, lens, j)
        out, lse = wm.draft_step(ring, kn, vn, qs[j], scale, ws, n_split=n_split)
        wm.ring_append(two, kn, vn)
        out2, lse2 = wm.draft_attn(two, qs[j], scale, n_split=n_split)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), f"step {j}: out differs"
        assert torch.equal(lse, lse2), f"step {j}: lse differs"
    for name in ("k", "v"):
        assert torch.equal(getattr(ring, name).view(torch.int16), getattr(two, name).view(torch.int16))
    assert torch.equal(ring.pos_tag, two.pos_tag) and torch.equal(ring.n_seen, two.n_seen)
    assert wm.get_device_error() == 0


def test_step_graph_replays_advance_the_ring():
    """One captured step replayed: each replay appends the next position (the
    inputs are refreshed in place)."""
    B, Hkv, G, D, S, W, lens, steps = 1, 2, 8, 256, 4, 4096, [6000], 5
    dev, hk, hv, ring, qs = setup(B, Hkv, G, D, S, W, lens, steps, seed=55)
    scale = D ** -0.5
    ws = wm.step_workspace(ring, Hkv * G)
    kn, vn, q = gather_pos(hk, lens, 0), gather_pos(hv, lens, 0), qs[0].clone()
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hkv * G), float("nan"), dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the graph: plans and attributes are cached
        wm.draft_step(ring, kn, vn, q, scale, ws, out=out, lse=lse, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    hist = oracle_kv(hk, hv)
    ref, ref_lse = oracle.draft(hist, q.cpu(), [lens[0]], S, W, scale)
    assert_close("eager step 0", out, lse, ref, ref_lse)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wm.draft_step(ring, kn, vn, q, scale, ws, out=out, lse=lse, stream=torch.cuda.current_stream())
    for j in range(1, steps):
        kn.copy_(gather_pos(hk, lens, j))
        vn.copy_(gather_pos(hv, lens, j))
        q.copy_(qs[j])
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle.draft(hist, q.cpu(), [lens[0] + j], S, W, scale)
        assert_close(f"replay {j}", out, lse, ref, ref_lse)
    check_ring(ring, hk, hv, [lens[0] + steps])
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("bad", [-5, 2 ** 31 - 1, 2 ** 40])
def test_step_bad_n_seen_is_reported_and_skipped(bad):
    """An n_seen that is negative or does not fit an int32 tag is bad device
    data: recorded, nothing appended for that sequence, its rows 0 / -inf; the
    other sequence steps normally."""
    B, Hkv, G, D, S, W, lens = 2, 2, 4, 128, 4, 256, [1000, 1000]
    dev, hk, hv, ring, qs = setup(B, Hkv, G, D, S, W, lens, 1, seed=9)
    ring.n_seen[1] = bad
    tags_before = ring.pos_tag.clone()
    ws = wm.step_workspace(ring, Hkv * G)
    out, lse = wm.draft_step(ring, gather_pos(hk, lens, 0), gather_pos(hv, lens, 0), qs[0], 1.0 / D ** 0.5, ws)
    torch.cuda.synchronize()
    assert wm.get_device_error() == 1  # WM_DEVERR_BAD_LENGTH
    assert ring.n_seen.tolist() == [1001, bad]
    assert torch.equal(ring.pos_tag[1], tags_before[1])
    assert bool((out[1] == 0).all()) and bool(torch.isneginf(lse[1]).all())
    ref, ref_lse = oracle.draft(oracle_kv(hk, hv), qs[0].cpu(), [1000, 1000], S, W, 1.0 / D ** 0.5)
    Hq = Hkv * G
    assert_close("sequence 0", out[:1], lse[:1], ref[:Hq], ref_lse[:Hq])


def test_step_plan_and_workspace():
    gpu()
    # the fused step splits exactly as the draft attention, and always needs partials
    for args in [(1, 2, 16, 1, 256, 4100), (2, 8, 64, 1, 128, 8208), (8, 8, 32, 1, 128, 1028)]:
        for ns in (0, 1, 7):
            assert wm.plan_splits(wm.WM_OP_DRAFT_STEP, *args, ns) == wm.plan_splits(wm.WM_OP_DRAFT, *args, ns)
    assert wm.workspace_size(wm.WM_OP_DRAFT, 1, 2, 16, 1, 256, 4100, 1) == 0
    assert wm.workspace_size(wm.WM_OP_DRAFT_STEP, 1, 2, 16, 1, 256, 4100, 1) > 0
