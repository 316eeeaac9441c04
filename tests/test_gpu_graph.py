"""A multi-layer decode step captured in a CUDA graph (append -> decode ->
combine per layer, programmatic dependent launches inside the graph): replay
must give the same bits as eager execution, for the split-KV decode path and
for the tensor-core tile path."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("dtype,cached,qlen", [("nvfp4", [5000, 700], [1, 1]),
                                               ("bf16", [3000], [5]),
                                               ("nvfp4", [2000], [40])])
def test_graph_replay_equals_eager(dtype, cached, qlen):
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeStack
    w = workloads.build("graph " + dtype, 31, dtype, cached, qlen)
    st = DecodeStack(w, layers=3)
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
