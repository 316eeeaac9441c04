"""The allocation-free decode entry point, checked against the regular one.

paged_decode_attention_noalloc serves callers that cannot allocate device
memory for the split-KV partials (an engine that reserves all device memory
up front for its own allocator, a latency-critical loop where cudaMalloc
could synchronise the device, plain C code).  It keeps the partials in the
library's fixed scratch array instead.  It runs the same kernels with the
same work split as the regular decode + combine, so called through the C ABI
twice in a row its output and LSE must equal the regular entry point's bit
for bit (a scratch overlap that perturbed a few partials would show), on the
split-KV path and on the tensor-core tile path (more than 64 query rows per
KV head).  This file is collected last so that a stop at the first failure
has already run every other test.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,cached,qlen", [("nvfp4", [3000, 77, 1500], [1, 1, 1]),
                                               ("bf16", [900, 40], [5, 5]),
                                               ("nvfp4", [2500], [20])])
def test_noalloc_matches_regular_entry(dtype, cached, qlen):
    import __graft_entry__
    __graft_entry__.build()
    from paged_nvfp4_kv_gb300 import _lib, workloads
    from paged_nvfp4_kv_gb300.engine import DecodeSession

    w = workloads.build("noalloc " + dtype, 91, dtype, cached, qlen)
    s = DecodeSession(w)
    s.fill()
    s.append()
    want = s.attend(out_fp32=True).clone()
    want_lse = s.lse.clone()
    torch.cuda.synchronize()
    assert s.error_word() == 0

    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(want, float("nan"))
        lse = torch.full_like(want_lse, float("nan"))
        st = lib.paged_decode_attention_noalloc(
            ctypes.byref(s.cache.desc), ctypes.c_void_p(s.q_roped.data_ptr()),
            ctypes.c_void_p(s.qo_indptr.data_ptr()), ctypes.c_void_p(s.page_table.data_ptr()),
            s.page_table.shape[1], ctypes.c_void_p(s.seq_lens.data_ptr()), w.batch,
            w.num_q_heads, s.max_qlen, s.sm_scale, 1, s.total_q,
            ctypes.c_void_p(out.data_ptr()), 1, ctypes.c_void_p(lse.data_ptr()),
            ctypes.c_void_p(s.dev_err.data_ptr()), stream)
        assert st == 0, st
        torch.cuda.synchronize()
        assert s.error_word() == 0
        assert torch.equal(out.view(torch.int32), want.view(torch.int32)), call
        assert torch.equal(lse.view(torch.int32), want_lse.view(torch.int32)), call


def test_noalloc_rejects_requests_beyond_the_scratch():
    import __graft_entry__
    __graft_entry__.build()
    from paged_nvfp4_kv_gb300 import Cache, _lib
    cache = Cache(16, "nvfp4", k_scale=0.01, v_scale=0.01)
    lib = _lib.load()
    P = ctypes.c_void_p
    # 4,096 sequences x 4 heads x 48 rows x 257 floats is far beyond 8 MiB
    st = lib.paged_decode_attention_noalloc(ctypes.byref(cache.desc), P(256), P(256), P(256), 1,
                                            P(256), 4096, 24, 8, 0.0625, 1, 4096, P(256), 1, None,
                                            P(256), None)
    assert st == _lib.PNKV_ERR_INVALID_ARG
