"""Repeated graph replays of each attention path give the same bits every time.

A race on a pipeline barrier's phase, a staging slot or a partial buffer shows
up as a replay whose output differs from the others in the last bits, long
before it fails a tolerance.  Each case checks its first replay against the
fp64 oracle and then requires 300 further replays to reproduce it exactly."""
import math

import pytest
import torch

import oracle
from speculative_decoding_attention_gb300 import wm

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu

REPLAYS = 300


def rand_bf16(shape, gen, device, std=1.0):
    return (torch.randn(shape, generator=gen, device=device) * std).to(torch.bfloat16)


def capture(fn):
    fn()
    torch.cuda.synchronize()
    g, s = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def replays_identical(graph, outs, reset=None):
    """Replay REPLAYS times; every replay's outputs equal the first replay's."""
    if reset:
        reset()
    graph.replay()
    torch.cuda.synchronize()
    first = [t.clone() for t in outs]
    saved = [torch.empty((REPLAYS,) + t.shape, dtype=t.dtype, device=t.device) for t in outs]
    for i in range(REPLAYS):
        for t in outs:
            t.fill_(float("nan"))
        if reset:
            reset()
        graph.replay()
        for s, t in zip(saved, outs):
            s[i].copy_(t)
    torch.cuda.synchronize()
    bad = sum(not all(torch.equal(s[i], f) for s, f in zip(saved, first)) for i in range(REPLAYS))
    assert bad == 0, f"{bad} of {REPLAYS} replays differ from the first"
    return first


@pytest.mark.parametrize("D,G,T,page,n_split", [
    (256, 8, 4, 0, 24),    # the 1M hybrid shape on a short cache: 32 rows, several splits, merge
    (256, 8, 6, 0, 12),    # 48 rows: V staged in 64-key halves by its own producer warp
    (128, 4, 3, 64, 9),    # 16 rows, short staging ring, paged
    (64, 4, 3, 0, 5),      # head_dim 64: the mma.sync verify kernel
])
def test_verify_replays_are_bit_identical(D, G, T, page, n_split):
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(3000 + D + G + T + page)
    Hkv, n = 2, 5000
    q = rand_bf16((1, T, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    if page:
        n_pages = -(-n // page)
        bt = torch.randperm(n_pages, generator=torch.Generator().manual_seed(3001)).view(1, n_pages)
        bt = bt.to(torch.int32).to(dev)
        k, v = rand_bf16((n_pages, Hkv, page, D), gen, dev), rand_bf16((n_pages, Hkv, page, D), gen, dev)
    else:
        bt = None
        k, v = rand_bf16((1, Hkv, n, D), gen, dev), rand_bf16((1, Hkv, n, D), gen, dev)
    kv = wm.KVCache(k, v, torch.tensor([n - 3], dtype=torch.int64, device=dev), bt)
    need = wm.workspace_size(wm.WM_OP_VERIFY, 1, Hkv, Hkv * G, T, D, kv.capacity, n_split)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((1, T, Hkv * G, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, T, Hkv * G), dtype=torch.float32, device=dev)
    g = capture(lambda: wm.verify_attn(kv, q, 1.0, n_split=n_split, out=out, lse=lse, workspace=ws))
    first_out, first_lse = replays_identical(g, [out, lse])
    ref, ref_lse = oracle.verify(oracle_kv(k, v, bt), q.cpu(), [n - 3], 1.0)
    assert_close(f"verify D={D} rows={G * T}", first_out, first_lse, ref, ref_lse)
    assert wm.get_device_error() == 0


@pytest.mark.parametrize("D,G", [(256, 8), (128, 8), (64, 4), (128, 16)])
def test_fused_draft_step_replays_are_bit_identical(D, G):
    """The fused draft step (append + attention + merge), rolled back before
    every replay so that each replay appends and attends at the same position;
    8 rows per KV head run the keys-as-M kernel, 16 the row-major one."""
    dev = gpu()
    gen = torch.Generator(device=dev).manual_seed(3100 + D + G)
    B, Hkv, S, W, n = 2, 2, 4, 2000, 6000
    k, v = rand_bf16((B, Hkv, n + 1, D), gen, dev), rand_bf16((B, Hkv, n + 1, D), gen, dev)
    ring = wm.Ring.create(B, Hkv, D, S, W, dev)
    wm.ring_fill(ring, wm.KVCache(k, v, torch.tensor([n, n - 700], device=dev)))
    base = ring.n_seen.clone()
    ws = wm.step_workspace(ring, Hkv * G)
    q = rand_bf16((B, Hkv * G, D), gen, dev, 1 / math.sqrt(D))
    kn = torch.stack([k[0, :, n], k[1, :, n - 700]]).contiguous()
    vn = torch.stack([v[0, :, n], v[1, :, n - 700]]).contiguous()
    out = torch.empty((B, Hkv * G, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hkv * G), dtype=torch.float32, device=dev)
    g = capture(lambda: wm.draft_step(ring, kn, vn, q, 1.0, ws, out=out, lse=lse))
    first_out, first_lse = replays_identical(g, [out, lse], reset=lambda: wm.ring_rollback(ring, base))
    ref, ref_lse = oracle.draft(oracle_kv(k, v), q.cpu(), [n, n - 700], S, W, 1.0)
    assert_close(f"draft step D={D} G={G}", first_out, first_lse, ref, ref_lse)
    assert wm.get_device_error() == 0
