"""Ring buffer contents, tags and counters: bit-exact.

Expected contents come from the documented slot rule and from the textbook
StreamingLLM cache model (sink list + deque); K/V bytes are compared exactly.
"""
import pytest
import torch

from oracle.ring_model import StreamingCache
from speculative_decoding_attention_gb300 import wm

from parity import gpu

pytestmark = pytest.mark.gpu


def slot_rule(p, S, W):
    return p if p < S else S + (p - S) % W


def rand_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device).to(torch.bfloat16)


def check_ring_holds(ring, hk, hv, held_per_seq):
    tags = ring.pos_tag.cpu()
    for b, held in enumerate(held_per_seq):
        t = tags[b]
        assert sorted(int(x) for x in t[t >= 0]) == sorted(held)
        for s in torch.nonzero(t >= 0).flatten().tolist():
            p = int(t[s])
            assert s == slot_rule(p, ring.sink, ring.window)
            assert torch.equal(ring.k[b, :, s].view(torch.int16), hk[b, :, p].view(torch.int16))
            assert torch.equal(ring.v[b, :, s].view(torch.int16), hv[b, :, p].view(torch.int16))


@pytest.mark.parametrize("S,W", [(0, 1), (4, 5), (16, 37), (4, 256)])
def test_appends_bit_exact(S, W):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(10 + S + W)
    B, Hkv, D = 2, 3, 128
    n = 2 * (S + W) + 9
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    model = StreamingCache(S, W)
    for p in range(n):
        wm.ring_append(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous())
        model.append(p)
        if p in (0, S, S + W - 1, S + W, n - 1):
            check_ring_holds(ring, hk, hv, [model.held()] * B)
    assert ring.n_seen.tolist() == [n] * B
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S,W", [(0, 3), (4, 60), (16, 100)])
def test_fill_equals_sequential_appends(D, S, W):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(20 + D + S + W)
    B, Hkv = 3, 2
    cap = 500
    lens = [0, S // 2 + 1, 437]
    hk, hv = rand_bf16((B, Hkv, cap, D), gen, dev), rand_bf16((B, Hkv, cap, D), gen, dev)
    filled = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(filled, wm.KVCache(hk, hv, torch.tensor(lens, device=dev)))
    appended = wm.Ring.create(B, Hkv, D, S, W, dev)
    # one single-sequence ring per sequence, so each gets exactly lens[b] appends
    for b in range(B):
        one = wm.Ring.create(1, Hkv, D, S, W, dev)
        for p in range(lens[b]):
            wm.ring_append(one, hk[b:b + 1, :, p].contiguous(), hv[b:b + 1, :, p].contiguous())
        appended.k[b].copy_(one.k[0])
        appended.v[b].copy_(one.v[0])
        appended.pos_tag[b].copy_(one.pos_tag[0])
        appended.n_seen[b].copy_(one.n_seen[0])
    for name in ("k", "v"):
        assert torch.equal(getattr(filled, name).view(torch.int16), getattr(appended, name).view(torch.int16))
    assert torch.equal(filled.pos_tag, appended.pos_tag)
    assert torch.equal(filled.n_seen, appended.n_seen)
    from oracle.ring_model import held_after
    check_ring_holds(filled, hk, hv, [held_after(S, W, n) for n in lens])


def test_fill_from_paged_history():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(30)
    B, Hkv, D, ps, S, W = 2, 2, 128, 64, 4, 150
    lens = [333, 64]
    n_pages_b = [-(-n // ps) for n in lens]
    P = sum(n_pages_b)
    pool_k, pool_v = rand_bf16((P, Hkv, ps, D), gen, dev), rand_bf16((P, Hkv, ps, D), gen, dev)
    perm = torch.randperm(P, generator=gen, device=dev).to(torch.int32)
    bt = torch.full((B, max(n_pages_b)), -1, dtype=torch.int32, device=dev)
    bt[0, :n_pages_b[0]] = perm[:n_pages_b[0]]
    bt[1, :n_pages_b[1]] = perm[n_pages_b[0]:]
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(pool_k, pool_v, torch.tensor(lens, device=dev), bt))
    # logical view of the paged history
    hk = torch.zeros((B, Hkv, max(lens), D), dtype=torch.bfloat16, device=dev)
    hv = torch.zeros_like(hk)
    for b in range(B):
        for j in range(lens[b]):
            page = int(bt[b, j // ps])
            hk[b, :, j] = pool_k[page, :, j % ps]
            hv[b, :, j] = pool_v[page, :, j % ps]
    from oracle.ring_model import held_after
    check_ring_holds(ring, hk, hv, [held_after(S, W, n) for n in lens])


def test_twenty_thousand_appends_after_fill():
    """NoPE-workload pattern: bulk fill, then appends that wrap the window several times."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(40)
    B, Hkv, D, S, W = 2, 2, 128, 16, 2048
    n_fill, n_app = 3000, 5 * W + 11
    n = n_fill + n_app
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hv, torch.full((B,), n_fill, dtype=torch.int64, device=dev)))
    ks, vs = hk.permute(2, 0, 1, 3).contiguous(), hv.permute(2, 0, 1, 3).contiguous()
    for p in range(n_fill, n):
        wm.ring_append(ring, ks[p], vs[p])
    from oracle.ring_model import held_after
    check_ring_holds(ring, hk, hv, [held_after(S, W, n)] * B)


def test_rollback_matches_streaming_model():
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(50)
    B, Hkv, D, S, W = 1, 1, 64, 4, 16
    n = 60
    hk, hv = rand_bf16((B, Hkv, n, D), gen, dev), rand_bf16((B, Hkv, n, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    model = StreamingCache(S, W)
    p = 0
    for target, new_len in [(30, 27), (40, 2), (n, 50)]:
        while p < target:
            wm.ring_append(ring, hk[:, :, p].contiguous(), hv[:, :, p].contiguous())
            model.append(p)
            p += 1
        wm.ring_rollback(ring, torch.tensor([new_len], dtype=torch.int64, device=dev))
        model.rollback(new_len)
        p = new_len
        check_ring_holds(ring, hk, hv, [model.held()])
        assert int(ring.n_seen[0]) == new_len


def test_bad_page_sets_device_error():
    dev = gpu()
    B, Hkv, D, ps = 1, 1, 128, 64
    pool = torch.zeros((4, Hkv, ps, D), dtype=torch.bfloat16, device=dev)
    bt = torch.tensor([[0, 9, 1]], dtype=torch.int32, device=dev)   # page 9 is outside the pool
    ring = wm.Ring.create(B, Hkv, D, 4, 256, dev)
    wm.ring_fill(ring, wm.KVCache(pool, pool, torch.tensor([150], device=dev), bt))
    assert wm.get_device_error() == 2
    assert wm.get_device_error() == 0  # read clears it
    q = torch.zeros((B, 1, 2, D), dtype=torch.bfloat16, device=dev)
    wm.verify_attn(wm.KVCache(pool, pool, torch.tensor([150], device=dev), bt), q, 1.0)
    assert wm.get_device_error() == 2


def test_bad_length_sets_device_error():
    dev = gpu()
    k = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    q = torch.zeros((1, 1, 1, 64), dtype=torch.bfloat16, device=dev)
    wm.verify_attn(wm.KVCache(k, k, torch.tensor([129], device=dev)), q, 1.0)
    assert wm.get_device_error() == 1


@pytest.mark.parametrize("bad", [-1, 2 ** 31 - 1, 2 ** 33])
def test_append_past_int32_tags_is_refused(bad):
    """Tags are int32: an append at a position that does not fit one (or at a
    negative one) is recorded and leaves that sequence's ring untouched."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(31)
    B, Hkv, D, S, W = 2, 2, 64, 4, 16
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    hk = rand_bf16((B, Hkv, 40, D), gen, dev)
    wm.ring_fill(ring, wm.KVCache(hk, hk, torch.tensor([30, 30], device=dev)))
    before = (ring.k.clone(), ring.v.clone(), ring.pos_tag.clone())
    ring.n_seen[1] = bad
    kn, vn = rand_bf16((B, Hkv, D), gen, dev), rand_bf16((B, Hkv, D), gen, dev)
    wm.ring_append(ring, kn, vn)
    assert wm.get_device_error() == 1  # WM_DEVERR_BAD_LENGTH
    assert ring.n_seen.tolist() == [31, bad]
    for new, old in zip((ring.k, ring.v, ring.pos_tag), before):
        assert torch.equal(new[1], old[1])
    s = slot_rule(30, S, W)
    assert int(ring.pos_tag[0, s]) == 30 and torch.equal(ring.k[0, :, s], kn[0])
