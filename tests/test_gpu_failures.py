"""Device-side failure detection, driven from the host.

Each test corrupts one host-built input -- a page id outside the pool, a
position past the rope table, a sequence longer than its page-table row, a
decreasing qo_indptr, rows past total_q, a sequence index outside the batch
-- and checks that (1) the call returns and the matching PNKV_DEV_ERR_* bit
is set, (2) nothing faults: the context serves the next call, and (3) the
sequences the corruption does not touch still produce the oracle's attention
(and the same bits as an uncorrupted run).  The kernels check these inputs,
skip the offending page, token or sequence and flag it ("A 1,048,576-token
context on two RTX 5090s", section "Things that bit me": a negative control
past the staging bound must fail cleanly, not corrupt memory).

The timeout tests shorten the pipeline wait bound so that ordinary waits run
out, and check that PNKV_DEV_ERR_TIMEOUT is set, the kernel returns, and the
next call with the default bound is correct ("NInfer -- Windows 11 TP2 fork"
README: a bounded spin with an error word instead of a silent deadlock).
Nothing here makes a GPU fault, trap or hang.
"""
import numpy as np
import pytest
import torch

import oracle_path

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 5e-3
PAGE_ID, POSITION, SEQ_LEN, QO_INDPTR, TIMEOUT, SEQ_INDEX = 1, 2, 4, 8, 16, 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _session(dtype="nvfp4", cached=(900, 700, 1300), qlen=(1, 1, 1), seed=404):
    from paged_nvfp4_kv_gb300 import workloads
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = workloads.build("failure %s" % dtype, seed, dtype, list(cached), list(qlen))
    s = DecodeSession(w)
    s.fill()
    s.append()
    clean = s.attend(out_fp32=True).clone()
    clean_lse = s.lse.clone()
    torch.cuda.synchronize()
    assert s.error_word() == 0
    return w, s, clean, clean_lse


def _rows_of(w, seqs):
    return [t for b in seqs for t in range(int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))]


def _check_untouched(w, s, out, clean, seqs, bitwise=True):
    """Rows of sequences ``seqs``: within the oracle's tolerance over the GPU
    pool, and bitwise equal to the clean run where the corruption leaves the
    work split unchanged (skipping a whole sequence changes how stream-K cuts
    the remaining units into splits, and so the summation order)."""
    rows = _rows_of(w, seqs)
    o = out.cpu().numpy()
    if bitwise:
        assert np.array_equal(o[rows].view(np.int32), clean.cpu().numpy()[rows].view(np.int32))
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    want = oracle_path.attention(w, pool, q, rows={(t, h) for t in rows for h in range(w.num_q_heads)})
    errs = np.concatenate([np.abs(o[t, h] - r[0]) for (t, h), r in want.items()])
    assert errs.max() <= MAX_ABS and errs.mean() <= MEAN_ABS, (errs.max(), errs.mean())


def _reset(s):
    s.dev_err.zero_()
    torch.cuda.synchronize()


@pytest.mark.parametrize("bad", ["num_pages", "minus_one"])
@pytest.mark.parametrize("path", ["split-kv", "tile"])
def test_page_id_outside_pool(bad, path):
    qlen = (1, 1, 1) if path == "split-kv" else (20, 20, 20)  # 120 rows per KV head: the tile
    w, s, clean, _ = _session(qlen=qlen)
    pid = w.num_pages if bad == "num_pages" else -1
    s.page_table[1, 3] = pid
    _reset(s)
    out = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    assert s.error_word() & PAGE_ID
    _check_untouched(w, s, out, clean, [0, 2])
    # the context still serves a clean call
    s.page_table.copy_(torch.from_numpy(w.page_table).cuda())
    _reset(s)
    again = s.attend(out_fp32=True)
    torch.cuda.synchronize()
    assert s.error_word() == 0
    assert torch.equal(again.view(torch.int32), clean.view(torch.int32))


def test_position_past_rope_table():
    from paged_nvfp4_kv_gb300 import kv_append_nvfp4
    w, s, clean, _ = _session()
    pos = s.tok_pos.clone()
    pos[1] = s.cos.shape[0]  # one row past the table
    s.q_roped.zero_()
    pool_before = s.cache.pool.clone()
    _reset(s)
    kv_append_nvfp4(s.cache, s.page_table, w.batch, s.tok_seq, pos, s.q, s.q_roped, s.k, s.v,
                    s.cos, s.sin, s.rotary_dim, s.dev_err)
    torch.cuda.synchronize()
    assert s.error_word() & POSITION
    # the other tokens' roped queries are written; the flagged one (no rope
    # row to read) is not, and the pool is untouched (the others' K/V rewrite
    # identical bytes, the flagged token's are skipped)
    assert torch.count_nonzero(s.q_roped[1]) == 0
    assert torch.count_nonzero(s.q_roped[0]) > 0 and torch.count_nonzero(s.q_roped[2]) > 0
    assert torch.equal(s.cache.pool, pool_before)
    out = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    _check_untouched(w, s, out, clean, [0, 2])


def test_sequence_index_outside_batch():
    from paged_nvfp4_kv_gb300 import kv_append_nvfp4
    w, s, clean, _ = _session()
    seq = s.tok_seq.clone()
    seq[1] = w.batch
    pool_before = s.cache.pool.clone()
    _reset(s)
    kv_append_nvfp4(s.cache, s.page_table, w.batch, seq, s.tok_pos, s.q, s.q_roped, s.k, s.v,
                    s.cos, s.sin, s.rotary_dim, s.dev_err)
    torch.cuda.synchronize()
    assert s.error_word() & SEQ_INDEX
    # a query's rope needs only its position, so its roped row is still
    # written; the token's K/V (which needs the sequence's page table row) is
    # skipped, and the pool is untouched
    assert torch.equal(s.cache.pool, pool_before)
    out = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    _check_untouched(w, s, out, clean, [0, 2])


@pytest.mark.parametrize("path", ["split-kv", "tile"])
def test_sequence_longer_than_its_page_table_row(path):
    qlen = (1, 1, 1) if path == "split-kv" else (20, 20, 20)
    w, s, clean, _ = _session(qlen=qlen)
    s.seq_lens[1] = s.page_table.shape[1] * 16 + 1
    _reset(s)
    out = s.attend(out_fp32=True).clone()
    lse = s.lse.clone()
    torch.cuda.synchronize()
    assert s.error_word() & SEQ_LEN
    rows = _rows_of(w, [1])
    # the flagged sequence is skipped: no visible key, zero output, LSE -inf
    assert torch.count_nonzero(out[rows]) == 0
    assert torch.all(torch.isneginf(lse[rows]))
    _check_untouched(w, s, out, clean, [0, 2], bitwise=path == "tile")


@pytest.mark.parametrize("path", ["split-kv", "tile"])
def test_decreasing_qo_indptr(path):
    ql = 2 if path == "split-kv" else 20
    w, s, clean, _ = _session(qlen=(ql, ql, ql))
    bad = w.qo_indptr.astype(np.int32).copy()
    bad[2] = bad[1] - 1  # sequence 1 gets a negative row count, sequence 2 too many rows
    s.qo_indptr.copy_(torch.from_numpy(bad).cuda())
    _reset(s)
    out = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    assert s.error_word() & QO_INDPTR
    _check_untouched(w, s, out, clean, [0], bitwise=path == "tile")


def test_rows_past_total_q():
    """qo_indptr[batch] beyond the rows of q: the last sequence is skipped and
    flagged instead of being read past the end of q."""
    from paged_nvfp4_kv_gb300 import paged_decode_attention, split_kv_combine
    w, s, clean, _ = _session(qlen=(2, 2, 2))
    total = w.total_q - 1
    q = s.q_roped[:total]
    out = torch.full((total, w.num_q_heads, w.head_dim), float("nan"), device="cuda")
    _reset(s)
    paged_decode_attention(s.cache, q, s.qo_indptr, s.page_table, s.seq_lens, w.num_q_heads,
                           s.max_qlen, s.sm_scale, w.causal, s.o_part, s.lse_part, s.work_meta,
                           s.dev_err)
    split_kv_combine(s.o_part, s.lse_part, s.work_meta, s.qo_indptr, total, w.num_q_heads,
                     w.num_kv_heads, s.max_qlen, out)
    torch.cuda.synchronize()
    assert s.error_word() & QO_INDPTR
    assert torch.count_nonzero(out[total - 1]) == 0  # the skipped sequence's only row in range
    _check_untouched(w, s, out, clean[:total], [0, 1], bitwise=False)


@pytest.mark.parametrize("path", ["split-kv", "tile"])
def test_pipeline_wait_timeout(path):
    """A 1 us bound makes ordinary pipeline waits run out: the kernel flags
    the timeout and returns (its outputs are then unspecified); with the
    default bound restored the next call is exact again."""
    from paged_nvfp4_kv_gb300 import set_wait_limit_ns
    qlen = (1,) if path == "split-kv" else (40,)
    w, s, clean, clean_lse = _session(cached=(70000,), qlen=qlen)
    prev = set_wait_limit_ns(1000)
    try:
        seen = 0
        for _ in range(20):
            _reset(s)
            s.attend(out_fp32=True)
            torch.cuda.synchronize()
            seen = s.error_word()
            if seen & TIMEOUT:
                break
    finally:
        set_wait_limit_ns(prev)
    assert seen & TIMEOUT, seen
    assert (seen & ~TIMEOUT) == 0, seen  # nothing else was flagged
    _reset(s)
    again = s.attend(out_fp32=True)
    torch.cuda.synchronize()
    assert s.error_word() == 0
    assert torch.equal(again.view(torch.int32), clean.view(torch.int32))
    assert torch.equal(s.lse.view(torch.int32), clean_lse.view(torch.int32))
