"""A multi-layer decode step captured in a CUDA graph (append -> decode ->
combine per layer, programmatic dependent launches inside the graph).

Every layer has its own seeded K/V, new tokens, page table and per-tensor
scales, so a replay that mixed up layers (one layer reading another's pool,
queries or partials) gives outputs that match the wrong layer.  Checked, for
the split-KV decode path and the tensor-core tile path:
  - replayed outputs equal eager execution, bit for bit;
  - each layer's replayed fp32 output matches the oracle computed over that
    layer's own pool and queries (max-abs <= 1e-2, mean-abs <= 5e-3), and the
    bf16 output of a bf16 replay is its round-to-nearest-even;
  - the layers' oracle outputs differ from each other by far more than the
    tolerance, so the check above fails if two layers are swapped.
"""
import numpy as np
import pytest
import torch

import oracle_path

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _oracle(w, s):
    """{(t, h): o} of layer session s over its own pool and roped queries."""
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    return {k: v[0] for k, v in oracle_path.attention(w, pool, q).items()}


@pytest.mark.parametrize("dtype,cached,qlen", [("nvfp4", [5000, 700], [1, 1]),
                                               ("bf16", [3000], [5]),
                                               ("int8", [2500, 900], [2, 1]),
                                               ("nvfp4", [2000], [40])])
def test_graph_replay_layers_match_oracle(dtype, cached, qlen):
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeStack
    ws = [workloads.build("graph %s layer %d" % (dtype, i), 31 + 1000 * i, dtype, cached, qlen)
          for i in range(3)]
    st = DecodeStack(ws)
    st.fill()
    eager = [o.clone() for o in st.step(out_fp32=True)]
    torch.cuda.synchronize()
    assert st.error_word() == 0
    st.capture(out_fp32=True)
    for o in st.outputs(out_fp32=True):
        o.zero_()
    for _ in range(2):
        st.replay()
        torch.cuda.synchronize()
        for a, b in zip(eager, st.outputs(out_fp32=True)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert st.error_word() == 0

    refs = [_oracle(w, s) for w, s in zip(ws, st.sessions)]
    outs = [o.cpu().numpy() for o in st.outputs(out_fp32=True)]
    for i, (ref, o) in enumerate(zip(refs, outs)):
        errs = np.concatenate([np.abs(o[t, h] - r) for (t, h), r in ref.items()])
        assert errs.max() <= MAX_ABS and errs.mean() <= MEAN_ABS, (i, errs.max(), errs.mean())
    # a swap of two layers would be caught: their true outputs differ widely
    for i in range(3):
        for j in range(i + 1, 3):
            d = max(np.abs(refs[i][k] - refs[j][k]).max() for k in refs[i])
            assert d > 100 * MAX_ABS, (i, j, d)


def test_graph_replay_bf16_output():
    """A replayed bf16-output step: each layer's bf16 output is the RNE of its
    replayed fp32 output (same pools, same inputs: the append is idempotent)."""
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeStack
    ws = [workloads.build("graph bf16-out layer %d" % i, 57 + 1000 * i, "nvfp4", [3000, 64], [1, 3])
          for i in range(2)]
    st = DecodeStack(ws)
    st.fill()
    f32 = [o.clone() for o in st.step(out_fp32=True)]
    st.capture(out_fp32=False)
    st.replay()
    torch.cuda.synchronize()
    assert st.error_word() == 0
    for a, b in zip(f32, st.outputs(out_fp32=False)):
        assert torch.equal(a.to(torch.bfloat16).view(torch.int16), b.view(torch.int16))
