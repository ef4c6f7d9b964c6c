"""The draft kernel's CUDA-core variant (fp32 FMA products, warp-shuffle
softmax; wm_set_draft_math) against the oracle, on the same cases as the
tensor-core kernel: ring wraps, head dims, group sizes, the fused step, memory
slots and NaN patterns in never-written ring slots.  Kept to measure the
choice between the two; it must be just as correct."""
import math

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


@pytest.fixture
def fma_math():
    gpu()
    wm.set_draft_math(wm.WM_DRAFT_MATH_FMA)
    yield
    wm.set_draft_math(wm.WM_DRAFT_MATH_MMA)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("S,W", [(0, 1), (4, 60), (16, 200)])
def test_fma_draft_ring_wraps(fma_math, D, G, S, W):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(500 + D + G + S + W)
    B, Hkv = 2, 2
    n_pos = 3 * (S + W) + 7
    hk, hv = rand_bf16((B, Hkv, n_pos, D), gen, dev), rand_bf16((B, Hkv, n_pos, D), gen, dev)
    hist = oracle_kv(hk, hv)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    q = rand_bf16((n_pos, B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    check_at = sorted({0, S + W - 1, S + W, n_pos // 2, n_pos - 1})
    for p in range(n_pos):
        wm.ring_append(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous())
        if p in check_at:
            for ns in (0, 1, 3):
                out, lse = wm.draft_attn(ring, q[p], 1.0, n_split=ns)
                ref, ref_lse = oracle.draft(hist, q[p].cpu(), [p] * B, S, W, 1.0)
                assert_close(f"fma draft D={D} G={G} S={S} W={W} p={p} ns={ns}", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D", [128, 256])
def test_fma_fused_step_matches_oracle_and_unfused(fma_math, D):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(600 + D)
    B, Hkv, G, S, W, n, steps = 2, 2, 8, 4, 700, 1500, 3
    hk, hv = rand_bf16((B, Hkv, n + steps, D), gen, dev), rand_bf16((B, Hkv, n + steps, D), gen, dev)
    lens = torch.tensor([n, n - 300], dtype=torch.int64, device=dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, lens))
    two = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(two, wm.KVCache(hk, hv, lens))
    ws = wm.step_workspace(ring, Hkv * G)
    hist = oracle_kv(hk, hv)
    for j in range(steps):
        pos = [n + j, n - 300 + j]
        kn = torch.stack([hk[b, :, pos[b]] for b in range(B)]).contiguous()
        vn = torch.stack([hv[b, :, pos[b]] for b in range(B)]).contiguous()
        q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
        out, lse = wm.draft_step(ring, kn, vn, q, D ** -0.5, ws)
        wm.ring_append(two, kn, vn)
        out2, lse2 = wm.draft_attn(two, q, D ** -0.5)
        ref, ref_lse = oracle.draft(hist, q.cpu(), pos, S, W, D ** -0.5)
        assert_close(f"fma fused step {j}", out, lse, ref, ref_lse)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16)) and torch.equal(lse, lse2)
    assert torch.equal(ring.pos_tag, two.pos_tag) and torch.equal(ring.n_seen, two.n_seen)
    assert wm.get_device_error() == 0


def test_fma_memory_slots_and_stale_nan(fma_math):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(700)
    B, Hkv, G, D, S, W, cap = 1, 2, 8, 128, 4, 200, 40
    n = 120  # fewer positions than slots: never-written slots hold NaN
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    ring.k.fill_(float("nan"))
    ring.v.fill_(float("nan"))
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.tensor([n], device=dev)))
    mem = wm.Mem.create(B, Hkv, D, cap, dev)
    mem.k.copy_(rand_bf16(mem.k.shape, gen, dev))
    mem.v.copy_(rand_bf16(mem.v.shape, gen, dev))
    mem.count.fill_(17)
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    out, lse = wm.draft_attn_mem(ring, mem, q, 1.0)
    ref, ref_lse = oracle.draft_mem(oracle_kv(hk, hv), oracle_kv(mem.k, mem.v), [17], q.cpu(), [n - 1], S, W, 1.0)
    assert_close("fma memory draft", out, lse, ref, ref_lse)
    out, lse = wm.draft_attn(ring, q, 1.0)
    ref, ref_lse = oracle.draft(oracle_kv(hk, hv), q.cpu(), [n - 1], S, W, 1.0)
    assert_close("fma draft over partly written ring", out, lse, ref, ref_lse)
    assert wm.get_device_error() == 0
