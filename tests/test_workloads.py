"""Host-side checks of the seeded workload generator (no arithmetic of the
method lives there): determinism, sub-range draws equal slices of a full
draw, page tables are permutations, and the five workloads have the shapes
the method is measured on."""
import numpy as np

from paged_nvfp4_kv_gb300 import workloads as W


def test_draws_are_deterministic_and_sliceable():
    w = W.build("t", 77, "nvfp4", [70000, 100], [2, 1])
    a = w.k_rows(0, 0, 70002)
    b = W.build("t", 77, "nvfp4", [70000, 100], [2, 1]).k_rows(0, 65530, 65540)
    assert np.array_equal(a[65530:65540], b)
    assert np.array_equal(w.v_rows(1, 3, 9), w.v_rows(1, 0, 20)[3:9])
    assert a.dtype == np.float32
    assert np.array_equal(W.bf16_values(a), a)           # bf16-representable
    assert not np.array_equal(w.k_rows(1, 0, 10), w.k_rows(0, 0, 10)[:, :, :])


def test_page_table_is_a_permutation():
    w = W.build("t", 5, "bf16", [33, 16, 1], [1, 1, 5])
    used = w.page_table[w.page_table >= 0]
    assert sorted(used.tolist()) == list(range(w.num_pages))
    npg = (w.seq_lens + 15) // 16
    for b in range(3):
        assert np.all(w.page_table[b, :npg[b]] >= 0)
        assert np.all(w.page_table[b, npg[b]:] == -1)


def test_new_tokens_and_indptr():
    w = W.build("t", 5, "nvfp4", [10, 0, 7], [2, 3, 1])
    seq, pos = w.new_tokens()
    assert seq.tolist() == [0, 0, 1, 1, 1, 2]
    assert pos.tolist() == [10, 11, 0, 1, 2, 7]
    assert w.qo_indptr.tolist() == [0, 2, 5, 6]
    assert w.seq_lens.tolist() == [12, 3, 8]


def test_the_five_workloads():
    t = W.tiny_decode()
    assert t.seq_lens.tolist() == [4096] and t.kv_dtype == "bf16" and t.num_pages == 256
    n = W.native_window_decode()
    assert n.seq_lens.tolist() == [262144] and n.num_pages == 16384
    m = W.million_token_decode()
    assert m.seq_lens.tolist() == [1048576] and m.kv_dtype == "nvfp4" and m.num_pages == 65536
    v = W.multi_session_verify()
    assert v.batch == 16 and set(v.qlen.tolist()) == {5}
    assert v.cached.min() >= 8192 and v.cached.max() <= 524288
    p = W.chunked_prefill()
    assert p.cached.tolist() == [1040384] and p.qlen.tolist() == [8192]
    assert p.seq_lens.tolist() == [1048576]
    for w in (t, n, m, v, p):
        assert w.num_q_heads == 24 and w.num_kv_heads == 4 and w.head_dim == 256
        assert 0 < w.g_k < 1 and 0 < w.g_v < 1
