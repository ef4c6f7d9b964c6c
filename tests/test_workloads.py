"""Workload recipes against the figures the pages print, and the input generator."""
import json
import os

import pytest
import torch

from oracle.ring_model import held_after
from speculative_decoding_attention_gb300 import inputs, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")


def test_about_99_percent_of_draft_kv_dropped_at_1m():
    # Abstract: "dropping ~99% of KV entries at 1M" -- the held set of the
    # StreamingLLM cache model, as a share of the 1M context.
    fig = json.load(open(GOLDEN))["draft_kv_entries_dropped_at_1m"]
    for name in ("hybrid_1m_d256", "nope_1m_b2"):
        w = workloads.get(name)
        assert w.context == fig["context"]
        held = min(w.context, w.slots)
        dropped = 1 - held / w.context
        assert dropped >= fig["value"], (name, dropped)


def test_held_set_size_is_the_slot_count():
    w = workloads.get("tiny_4k")
    assert len(held_after(w.sink, w.window, w.context)) == w.slots == 260


def test_workload_shapes():
    for w in workloads.WORKLOADS.values():
        assert w.n_q_heads % w.n_kv_heads == 0
        assert w.head_dim in (64, 128, 256)
        assert w.window >= 1 and w.sink >= 0


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_inputs_are_seeded_and_laid_out(name):
    w = workloads.get(name)
    ctx = 600 if not w.ragged else 2048
    a = inputs.make_inputs(w, context=ctx)
    b = inputs.make_inputs(w, context=ctx)
    assert torch.equal(a.k, b.k) and torch.equal(a.q_verify, b.q_verify)
    d, T = a.depth, a.n_verify
    assert T == d + 1
    assert a.q_draft.shape == (d, w.batch, w.n_q_heads, w.head_dim)
    assert a.k_new.shape == (d, w.batch, w.n_kv_heads, w.head_dim)
    assert a.q_verify.shape == (w.batch, T, w.n_q_heads, w.head_dim)
    # the appended entries are the store's rows at positions N_b + j
    for j in range(d):
        kj, vj = a.position_rows([n + j for n in a.seq_lens_host])
        assert torch.equal(kj, a.k_new[j]) and torch.equal(vj, a.v_new[j])
    if w.page_size:
        used = a.block_table[a.block_table >= 0]
        assert used.unique().numel() == used.numel() == a.k.shape[0]


def test_peaked_keys_fraction():
    w = workloads.get("hybrid_1m_d256")
    a = inputs.make_inputs(w, depth=1, context=20000)
    big = (a.k[0, 0, :20000].float().abs().amax(-1) > 6).float().mean().item()
    assert 0.005 < big < 0.02
