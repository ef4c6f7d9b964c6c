"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

Each workload's step state is built exactly as the bench builds it (ring fill,
and for the NoPE workload 20,000 single appends that wrap the window), then:
every draft row of every draft step (fused and unfused) and every verify row
of the [batch, T, Hq] space is compared with the oracle element by element;
the ring's tags are compared with the StreamingLLM cache model.  The bench's
output buffers are filled with NaN before each run, so a row the kernels leave
unwritten fails.
"""
import pytest
import torch

import oracle
from oracle.ring_model import held_after

from parity import assert_close, gpu, oracle_kv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_4k", "gqa8_128k", "hybrid_1m_d256", "paged_ragged_b8", "nope_1m_b2"])
def test_full_size_step(name):
    dev = gpu()
    import bench
    from speculative_decoding_attention_gb300 import wm, workloads

    w = workloads.get(name)
    depth = workloads.BENCH_DEPTH if name == workloads.BENCH_WORKLOAD else w.max_depth
    st = bench.Step(w, depth, dev)
    inp = st.inp
    torch.cuda.synchronize()
    assert wm.get_device_error() == 0
    # ring after fill (+ appends): exactly the sinks and the last W positions
    tags = st.ring.pos_tag.cpu()
    for b, n in enumerate(inp.seq_lens_host):
        t = tags[b]
        assert sorted(int(x) for x in t[t >= 0]) == held_after(w.sink, w.window, n)

    hist = oracle_kv(inp.k, inp.v, inp.block_table)
    refs = [oracle.draft(hist, inp.q_draft[j].cpu(), [n + j for n in inp.seq_lens_host], w.sink, w.window,
                         w.scale) for j in range(depth)]
    # the unfused draft (append, attention, merge) first, then the fused step the bench times, each
    # from the ring as built (a rollback does not restore the window entries the appends overwrote)
    saved = [t.clone() for t in (st.ring.k, st.ring.v, st.ring.pos_tag, st.ring.n_seen)]
    for fused in (False, True):
        for t, c in zip((st.ring.k, st.ring.v, st.ring.pos_tag, st.ring.n_seen), saved):
            t.copy_(c)
        for t in (st.d_out, st.d_lse, st.v_out, st.v_lse):
            t.fill_(float("nan"))
        st.run(fused=fused)
        torch.cuda.synchronize()
        assert wm.get_device_error() == 0
        for j, (ref, ref_lse) in enumerate(refs):
            assert_close(f"{name} draft step {j} ({'fused' if fused else 'unfused'})", st.d_out[j], st.d_lse[j],
                         ref, ref_lse)
        assert st.ring.n_seen.tolist() == list(inp.seq_lens_host)  # rolled back

    # every verify row (the verify of the fused run above)
    ref, ref_lse = oracle.verify(hist, inp.q_verify.cpu(), inp.seq_lens_host, w.scale)
    assert_close(f"{name} verify (all {w.batch * st.T * w.n_q_heads} rows)", st.v_out, st.v_lse, ref, ref_lse)
