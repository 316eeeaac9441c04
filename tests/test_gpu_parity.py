"""GPU parity of the whole decode path against the CPU oracle, stage by stage
on identical inputs:

  1. YaRN table: GPU vs oracle within 2^-22 absolute, mismatching entries
     rare.  Both sides evaluate pow/cos/sin in double; the libraries may
     differ in the last double bit of an inverse frequency, which the
     position multiplies (p * 2^-52 relative) -- harmless in absolute terms
     but worth a few binary32 ulps where cos/sin is near zero.
  2. Roped queries and keys: bit-exact given the GPU table.
  3. Pool bytes (E2M1 codes, E4M3 scales, page placement; bf16 values):
     bit-exact given the GPU table.
  4. Attention: the fp32 output of split_kv_combine vs the oracle's float64
     attention over the same pool, max-abs <= 1e-2 and mean-abs <= 5e-3; the
     bf16 output is the round-to-nearest-even of that fp32 output, bit for
     bit; LSE within 1e-3.
  5. Repeated launches are bitwise identical; the device error word stays 0.
"""
import numpy as np
import pytest
import torch

import oracle_path
from oracle.formats import f32

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _session(w):
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    s = DecodeSession(w)
    s.fill()
    s.append()
    out32 = s.attend(out_fp32=True).clone()
    lse = s.lse.clone()
    out16 = s.attend(out_fp32=False).clone()
    torch.cuda.synchronize()
    return s, out32, out16, lse


def _workload(name, dtype, cached, qlen, seed=77, **kw):
    from paged_nvfp4_kv_gb300 import workloads as W
    return W.build(name, seed, dtype, cached, qlen, **kw)


CASES = {
    "ragged-nvfp4": ("nvfp4", [1000, 36, 4100], [1, 1, 1]),
    "ragged-bf16": ("bf16", [1000, 36, 4100], [1, 1, 1]),
    "verify5-nvfp4": ("nvfp4", [700, 50, 333, 2011], [5, 5, 5, 5]),
    "verify5-bf16": ("bf16", [700, 50, 333, 2011], [5, 5, 5, 5]),
    "qlen2-nvfp4": ("nvfp4", [517, 1200], [2, 2]),
    "qlen8-nvfp4": ("nvfp4", [300, 1800], [8, 3]),
    "qlen8-bf16": ("bf16", [300, 1800], [8, 3]),
    "page-edge-nvfp4": ("nvfp4", [16, 15, 17, 31, 32, 0], [1, 1, 1, 1, 1, 1]),
    # long sequences: every CTA takes many units and wraps its stage ring
    "long-bf16": ("bf16", [65535], [1]),
    "long-nvfp4": ("nvfp4", [70000, 7000], [1, 1]),
    "long-verify5-nvfp4": ("nvfp4", [40000, 23000], [5, 5]),
    "long-verify5-bf16": ("bf16", [30000], [5]),
    # FP8 (E4M3, per-tensor scale) pools through the same entry points
    "ragged-fp8": ("fp8", [1000, 36, 4100], [1, 1, 1]),
    "verify5-fp8": ("fp8", [700, 50, 333, 2011], [5, 5, 5, 5]),
    "qlen8-fp8": ("fp8", [300, 1800], [8, 3]),
    "page-edge-fp8": ("fp8", [16, 15, 17, 31, 32, 0], [1, 1, 1, 1, 1, 1]),
    "long-fp8": ("fp8", [70000, 7000], [1, 1]),
    # INT8 group-64 pools
    "ragged-int8": ("int8", [1000, 36, 4100], [1, 1, 1]),
    "verify5-int8": ("int8", [700, 50, 333, 2011], [5, 5, 5, 5]),
    "qlen8-int8": ("int8", [300, 1800], [8, 3]),
    "page-edge-int8": ("int8", [16, 15, 17, 31, 32, 0], [1, 1, 1, 1, 1, 1]),
    "long-int8": ("int8", [70000, 7000], [1, 1]),
    # more than 64 query rows per KV head: the tensor-core tile path
    "prefill-nvfp4": ("nvfp4", [3000, 500, 77], [100, 37, 1]),
    "prefill-long-nvfp4": ("nvfp4", [40000], [300]),
    # the verify tile's row range on NVFP4 pools at its two ends and without
    # the causal mask: 8 query heads per KV head x 4 tokens = all 32 rows of
    # the product's N; 3 x 3 = 9 rows, the fewest that take the tile
    "verify-32rows-nvfp4": ("nvfp4", [900, 130, 2500], [4, 4, 1], {"num_q_heads": 32, "num_kv_heads": 4}),
    "verify-9rows-nvfp4": ("nvfp4", [257, 1500, 64], [3, 1, 2], {"num_q_heads": 12, "num_kv_heads": 4}),
    "verify5-noncausal-nvfp4": ("nvfp4", [700, 333, 2011], [5, 5, 2], {"causal": False}),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def run(request):
    dtype, cached, qlen, *extra = CASES[request.param]
    w = _workload(request.param, dtype, cached, qlen, **(extra[0] if extra else {}))
    s, out32, out16, lse = _session(w)
    return w, s, out32, out16, lse


def test_table_close_to_oracle(run):
    w, s, *_ = run
    cos_o, sin_o = oracle_path.tables(w, s.max_pos)
    for got, want in ((s.cos, cos_o), (s.sin, sin_o)):
        g = got.cpu().numpy().astype(np.float64)
        d = np.abs(g - want)
        assert d.max() <= 2.0 ** -22, d.max()
        assert (d > 0).mean() < 1e-2, (d > 0).mean()


def test_roped_q_bit_exact(run):
    w, s, *_ = run
    cos_t, sin_t = s.cos.double().cpu().numpy(), s.sin.double().cpu().numpy()
    want = oracle_path.roped_new_q(w, cos_t, sin_t)
    assert np.array_equal(s.q_roped.float().cpu().numpy(), want)


def test_pool_bit_exact(run):
    w, s, *_ = run
    cos_t, sin_t = s.cos.double().cpu().numpy(), s.sin.double().cpu().numpy()
    want = oracle_path.pool(w, cos_t, sin_t)
    got = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    assert np.array_equal(got, want)


def test_attention_within_tolerance(run):
    w, s, out32, out16, lse = run
    cos_t, sin_t = s.cos.double().cpu().numpy(), s.sin.double().cpu().numpy()
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    ref = oracle_path.attention(w, pool, q)
    o = out32.cpu().numpy()
    l = lse.cpu().numpy()
    errs = []
    for (t, h), (ro, rl) in ref.items():
        errs.append(np.abs(o[t, h] - ro))
        assert abs(l[t, h] - rl) < 1e-3 * max(1.0, abs(rl)), (t, h)
    errs = np.concatenate(errs)
    assert errs.max() <= MAX_ABS, errs.max()
    assert errs.mean() <= MEAN_ABS, errs.mean()
    # bf16 output = RNE(bf16) of the fp32 output, bit for bit
    want16 = torch.from_numpy(o).to(torch.bfloat16)
    assert torch.equal(out16.cpu().view(torch.int16), want16.view(torch.int16))
    assert s.error_word() == 0


def test_repeat_is_bitwise_identical(run):
    w, s, out32, *_ = run
    again = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int32), out32.view(torch.int32))


def test_page_permutation_invariance():
    """A permutation of the pool's pages, with the page table permuted to
    match, leaves every output bit unchanged."""
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = _workload("perm", "nvfp4", [900, 130], [1, 5])
    s, out32, _, _ = _session(w)
    rng = np.random.default_rng(5)
    sigma = torch.from_numpy(rng.permutation(w.num_pages)).cuda()
    pool = s.cache.pool.view(w.num_pages, -1)
    new_pool = torch.empty_like(pool)
    new_pool[sigma] = pool
    pool.copy_(new_pool)
    pt = s.page_table
    s.page_table.copy_(torch.where(pt >= 0, sigma[pt.clamp(min=0).long()].int(), pt))
    again = s.attend(out_fp32=True).clone()
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int32), out32.view(torch.int32))


@pytest.mark.parametrize("dtype", ["fp8", "int8", "bf16"])
def test_prefill_chunk_needs_nvfp4(dtype):
    """More than 64 query rows per KV head run the tensor-core tile, built for
    NVFP4 pools only: other pools get PNKV_ERR_UNSUPPORTED, nothing runs."""
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = _workload("chunk-" + dtype, dtype, [500], [20])
    s = DecodeSession(w)
    s.fill()
    s.append()
    with pytest.raises(RuntimeError, match="unsupported"):
        s.attend(out_fp32=True)
    torch.cuda.synchronize()
    assert s.error_word() == 0
