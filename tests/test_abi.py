"""CPU checks of the C ABI: the library builds and loads, exports every
function include/pnkv.h declares, and rejects out-of-contract host arguments
before touching the GPU (no call here reaches a CUDA API)."""
import ctypes
import os
import re

import pytest

from paged_nvfp4_kv_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "pnkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[a-z0-9_]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"yarn_rope_tables", "kv_append_nvfp4", "paged_decode_attention",
            "split_kv_combine"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert {n for n, _, _ in _lib.SIGNATURES} == names


def test_version_and_status_text(lib):
    assert lib.pnkv_version() == 200
    assert lib.pnkv_status_string(-1) == b"invalid argument"


def test_wait_limit_setting(lib):
    """The pipeline wait bound is a host setting; out-of-range values are
    rejected and the previous bound is returned (no GPU involved)."""
    assert lib.pnkv_set_wait_limit_ns(999) == _lib.PNKV_ERR_INVALID_ARG
    assert lib.pnkv_set_wait_limit_ns(61 * 10**9) == _lib.PNKV_ERR_INVALID_ARG
    prev = lib.pnkv_set_wait_limit_ns(5000)
    assert prev == 2 * 10**9
    assert lib.pnkv_set_wait_limit_ns(prev) == 5000


def _yarn(**kw):
    p = dict(theta=1e7, factor=4.0, original_max=262144, beta_fast=32.0, beta_slow=1.0,
             rotary_dim=64, deployed_range=1)
    p.update(kw)
    return _lib.YarnParams(**p)


@pytest.mark.parametrize("kw", [dict(factor=65.0), dict(factor=0.5), dict(factor=float("nan")),
                                dict(original_max=262144 * 5), dict(factor=1.3, original_max=3),
                                dict(rotary_dim=48), dict(beta_fast=0.5), dict(theta=1.0),
                                dict(deployed_range=2)])
def test_yarn_validation(lib, kw):
    # rules of the README's "Usage" section: factor finite in [1, 64],
    # origin x factor a whole count <= 1,048,576
    st = lib.yarn_rope_tables(ctypes.byref(_yarn(**kw)), 10, ctypes.c_void_p(256),
                              ctypes.c_void_p(512), None)
    assert st == _lib.PNKV_ERR_INVALID_ARG


def test_yarn_bad_sizes(lib):
    p = _yarn()
    assert lib.yarn_rope_tables(ctypes.byref(p), 0, ctypes.c_void_p(256), ctypes.c_void_p(512),
                                None) == _lib.PNKV_ERR_INVALID_ARG
    assert lib.yarn_rope_tables(ctypes.byref(p), 10, None, ctypes.c_void_p(512),
                                None) == _lib.PNKV_ERR_INVALID_ARG


def _cache(**kw):
    d = dict(pool=1024, num_pages=10, page_size=16, num_kv_heads=4, head_dim=256, dtype=1,
             k_scale=0.01, v_scale=0.01)
    d.update(kw)
    return _lib.CacheDesc(**d)


def test_page_bytes(lib):
    out = ctypes.c_int64()
    assert lib.pnkv_page_bytes(ctypes.byref(_cache()), ctypes.byref(out)) == 0
    assert out.value == 18432
    assert lib.pnkv_page_bytes(ctypes.byref(_cache(dtype=0)), ctypes.byref(out)) == 0
    assert out.value == 65536
    assert lib.pnkv_page_bytes(ctypes.byref(_cache(dtype=2)), ctypes.byref(out)) == 0
    assert out.value == 32768
    assert lib.pnkv_page_bytes(ctypes.byref(_cache(dtype=2, k_scale=-1.0)), ctypes.byref(out)) == -1
    assert lib.pnkv_page_bytes(ctypes.byref(_cache(dtype=3, k_scale=0.0)), ctypes.byref(out)) == 0
    assert out.value == 33792
    for bad in (dict(page_size=32), dict(head_dim=128), dict(dtype=5), dict(pool=None),
                dict(pool=1000), dict(k_scale=0.0), dict(v_scale=float("inf")), dict(num_pages=0),
                dict(num_kv_heads=0)):
        assert lib.pnkv_page_bytes(ctypes.byref(_cache(**bad)), ctypes.byref(out)) == -1, bad


def test_append_validation(lib):
    c = _cache()
    P = ctypes.c_void_p
    ok = dict(pt=P(256), stride=4, batch=1, seq=P(256), pos=P(256), n=3, q=P(256), qo=P(512),
              hq=24, k=P(1024), v=P(2048), cos=P(4096), sin=P(8192), rows=100, R=64, err=P(256))

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.kv_append_nvfp4(ctypes.byref(c), a["pt"], a["stride"], a["batch"], a["seq"],
                                   a["pos"], a["n"], a["q"], a["qo"], a["hq"], a["k"], a["v"],
                                   a["cos"], a["sin"], a["rows"], a["R"], a["err"], None)

    for bad in (dict(R=48), dict(q=None), dict(k=P(1025)), dict(stride=0), dict(n=-1),
                dict(err=None), dict(hq=0), dict(batch=0)):
        assert call(**bad) == -1, bad
    assert call(n=0) == 0  # nothing to do, nothing launched
    tiny = _cache(k_scale=1e-35)
    assert lib.kv_append_nvfp4(ctypes.byref(tiny), P(256), 4, 1, P(256), P(256), 3, None, None, 0,
                               P(1024), P(2048), P(4096), P(8192), 100, 64, P(256), None) == -1


def test_decode_and_combine_validation(lib):
    c = _cache()
    P = ctypes.c_void_p
    args = [ctypes.byref(c), P(256), P(256), P(256), 4, P(256), 1, 1, 24, 1, 0.0625, 1, P(256),
            P(256), 1000, P(256), P(256), None]
    bad = list(args)
    bad[10] = float("nan")
    assert lib.paged_decode_attention(*bad) == -1
    bad = list(args)
    bad[8] = 25                      # not a multiple of the KV heads
    assert lib.paged_decode_attention(*bad) == -1
    bad = list(args)
    bad[1] = None
    assert lib.paged_decode_attention(*bad) == -1
    bad = list(args)
    bad[7] = -1                      # total_q
    assert lib.paged_decode_attention(*bad) == -1
    assert lib.pnkv_work_meta_ints(16, 4) == 4 + 2 * 64
    assert lib.pnkv_work_meta_ints(0, 4) == -1
    assert lib.split_kv_combine(P(256), P(256), P(256), P(256), 1, 1, 24, 4, 128, 1, P(256), 1,
                                None, None) == -1
    assert lib.split_kv_combine(P(256), P(256), P(256), P(256), 1, 0, 24, 4, 256, 1, P(256), 1,
                                None, None) == 0


def test_fp4q_prefill_validation(lib):
    """paged_prefill_attention_fp4q refuses out-of-contract arguments and
    requests it does not serve before touching the GPU."""
    c = _cache()
    P = ctypes.c_void_p

    def call(cache=c, hq=24, max_qlen=20, q_scale=0.01, sm=0.0625, q=P(256)):
        return lib.paged_prefill_attention_fp4q(ctypes.byref(cache), q, P(256), P(256), 4, P(256), 1, 20,
                                                hq, max_qlen, sm, 1, q_scale, P(256), P(256), 1000, P(256),
                                                P(256), None)

    for bad in (dict(q_scale=0.0), dict(q_scale=-1.0), dict(q_scale=float("inf")),
                dict(q_scale=float("nan")), dict(q_scale=2.0 ** -110), dict(q_scale=2.0 ** 110),
                dict(sm=0.0), dict(hq=25), dict(q=None), dict(max_qlen=0)):
        assert call(**bad) == _lib.PNKV_ERR_INVALID_ARG, bad
    # at most 64 rows per KV head (6 x 10) is a decode step, not a prefill chunk
    assert call(max_qlen=10) == _lib.PNKV_ERR_UNSUPPORTED
    # only NVFP4 pools hold codes the block-scaled product can read
    for dtype in (0, 2, 3):
        assert call(cache=_cache(dtype=dtype)) == _lib.PNKV_ERR_UNSUPPORTED, dtype
