"""GPU parity of the FP4-query prefill (paged_prefill_attention_fp4q): the
chunk's QK^T as a block-scaled FP4 x FP4 tensor-core product on the cache's
own codes, with the queries NVFP4-encoded under the decode scale g_Q.

The oracle's reading ("262,144 Tokens on One RTX 5090", section "Why NVFP4
KV changes the math"; ``oracle/fp4_prefill.py``): the logits are (q_hat .
k_hat) * sm_scale with q_hat the NVFP4 round trip of the roped bf16 query
under the cache's encoder, and everything after the logits is the plain
attention.  Checked on identical inputs (the GPU's roped queries and pool):
  - fp32 output vs the oracle's attention with q_hat: max-abs <= 1e-2,
    mean-abs <= 5e-3; LSE within 1e-3; bf16 output = RNE of the fp32 output;
  - repeated launches bitwise identical; the device error word stays 0;
  - the result really uses the encoded queries: it is much closer to the
    q_hat attention than to the plain-query attention, whose distance is
    printed beside it (the numerical price of FP4 queries).
"""
import numpy as np
import pytest
import torch

import oracle_path
from oracle import fp4_prefill as FP

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


CASES = {
    "fp4q-mixed": ([3000, 500, 77], [100, 37, 1]),
    "fp4q-long": ([40000], [300]),
    "fp4q-two-chunks": ([1500, 2200], [64, 17]),
    "fp4q-page-edges": ([16, 31, 2047], [12, 33, 15]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_fp4q_matches_oracle(case):
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    cached, qlen = CASES[case]
    w = workloads.build(case, 88, "nvfp4", cached, qlen)
    s = DecodeSession(w)
    s.fill()
    s.append()
    out32 = s.attend(out_fp32=True, q_scale=w.g_q).clone()
    lse = s.lse.clone()
    out16 = s.attend(out_fp32=False, q_scale=w.g_q).clone()
    again = s.attend(out_fp32=True, q_scale=w.g_q).clone()
    torch.cuda.synchronize()
    assert s.error_word() == 0
    assert torch.equal(again.view(torch.int32), out32.view(torch.int32))
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    q_hat = FP.dequantized_queries(q, w.g_q)
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    ref = oracle_path.attention(w, pool, q_hat)
    plain = oracle_path.attention(w, pool, q)
    o = out32.cpu().numpy()
    l = lse.cpu().numpy()
    errs, dplain = [], []
    for (t, h), (ro, rl) in ref.items():
        errs.append(np.abs(o[t, h] - ro))
        dplain.append(np.abs(o[t, h] - plain[(t, h)][0]))
        assert abs(l[t, h] - rl) < 1e-3 * max(1.0, abs(rl)), (t, h)
    errs, dplain = np.concatenate(errs), np.concatenate(dplain)
    assert errs.max() <= MAX_ABS, errs.max()
    assert errs.mean() <= MEAN_ABS, errs.mean()
    print("%s: vs FP4-query oracle max %.3g mean %.3g; vs plain-query attention max %.3g mean %.3g"
          % (case, errs.max(), errs.mean(), dplain.max(), dplain.mean()))
    assert dplain.mean() > 4 * errs.mean()
    want16 = torch.from_numpy(o).to(torch.bfloat16)
    assert torch.equal(out16.cpu().view(torch.int16), want16.view(torch.int16))


@pytest.mark.parametrize("dtype,qlen", [("nvfp4", 10), ("bf16", 20), ("fp8", 20), ("int8", 20)])
def test_fp4q_unsupported_requests(dtype, qlen):
    """Non-NVFP4 pools and requests with at most 64 rows per KV head (6 x 10
    here) are refused before anything runs."""
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = workloads.build("fp4q-refused", 5, dtype, [300], [qlen])
    s = DecodeSession(w)
    s.fill()
    s.append()
    with pytest.raises(RuntimeError, match="unsupported"):
        s.attend(out_fp32=True, q_scale=w.g_q)
    torch.cuda.synchronize()
    assert s.error_word() == 0
