"""Host-only checks of the C ABI: the library loads, exports what include/pa.h declares, and
rejects malformed arguments synchronously without touching a GPU."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as B

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_290_gb300 import build
    build.build()
    return B.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.pa_version() == 3


# --------------------------------------------------------------- hand-made descriptors (no GPU)

FAKE = 0x10000  # never dereferenced: every call below fails validation first


def T(dtype, shape, stride=None, data=FAKE):
    t = B.PATensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        t.shape[i] = s
        t.stride[i] = st
    return t


def call_attention(lib, q=None, kc=None, vc=None, bt=None, sl=None, qsl=None, out=None,
                   hint=(1, 100), ws=None, wsb=0, scale=0.125):
    n, hq, hkv, d, bs, nb, mb = 3, 8, 2, 64, 16, 40, 8
    q = q or T(B.PA_F16, [n, hq, d])
    kc = kc or T(B.PA_F16, [nb, hkv, bs, d])
    vc = vc or T(B.PA_F16, [nb, hkv, bs, d])
    bt = bt or T(B.PA_I32, [n, mb])
    sl = sl or T(B.PA_I32, [n])
    qsl = qsl or T(B.PA_I32, [n + 1])
    out = out or T(B.PA_F16, [n, hq, d])
    h = None if hint is None else ctypes.byref(B.PABatchHint(*hint))
    return lib.pa_attention(ctypes.byref(q), ctypes.byref(kc), ctypes.byref(vc), ctypes.byref(bt),
                            ctypes.byref(sl), ctypes.byref(qsl), ctypes.c_float(scale),
                            ctypes.byref(out), h, ws, wsb, None)


def msg(lib):
    return lib.pa_last_error().decode()


@pytest.mark.parametrize("kw, status, text", [
    (dict(q=T(B.PA_I32, [3, 8, 64])), B.PA_ERR_INVALID_ARG, "q must be float16"),
    (dict(q=T(B.PA_F16, [3, 8])), B.PA_ERR_INVALID_ARG, "rank"),
    (dict(kc=T(B.PA_F16, [40, 2, 16, 96]), vc=T(B.PA_F16, [40, 2, 16, 96]),
          q=T(B.PA_F16, [3, 8, 96]), out=T(B.PA_F16, [3, 8, 96])), B.PA_ERR_UNSUPPORTED, "head_dim"),
    (dict(kc=T(B.PA_F16, [40, 2, 8, 64]), vc=T(B.PA_F16, [40, 2, 8, 64])), B.PA_ERR_UNSUPPORTED,
     "block_size"),
    (dict(q=T(B.PA_F16, [3, 7, 64]), out=T(B.PA_F16, [3, 7, 64])), B.PA_ERR_INVALID_ARG, "multiple"),
    (dict(kc=T(B.PA_F16, [40, 1, 16, 64]), vc=T(B.PA_F16, [40, 1, 16, 64]),
          q=T(B.PA_F16, [3, 32, 64]), out=T(B.PA_F16, [3, 32, 64])), B.PA_ERR_UNSUPPORTED, "group"),
    (dict(out=T(B.PA_F16, [3, 8, 64], stride=[1024, 64, 1])), B.PA_ERR_INVALID_ARG, "contiguous"),
    (dict(kc=T(B.PA_F16, [40, 2, 16, 64], stride=[4096, 1024, 64, 1])), B.PA_ERR_INVALID_ARG,
     "contiguous"),
    (dict(vc=T(B.PA_F16, [41, 2, 16, 64])), B.PA_ERR_INVALID_ARG, "differ"),
    (dict(qsl=T(B.PA_I32, [3])), B.PA_ERR_INVALID_ARG, "query_start_loc"),
    (dict(bt=T(B.PA_I32, [2, 8])), B.PA_ERR_INVALID_ARG, "block_tables"),
    (dict(bt=T(B.PA_I64, [3, 8])), B.PA_ERR_INVALID_ARG, "int32"),
    (dict(q=T(B.PA_F16, [3, 8, 64], data=FAKE + 2)), B.PA_ERR_INVALID_ARG, "alignment"),
    (dict(kc=T(B.PA_F16, [40, 2, 16, 64], data=0)), B.PA_ERR_INVALID_ARG, "NULL"),
    (dict(hint=None), B.PA_ERR_INVALID_ARG, "hint"),
    (dict(hint=(-1, 10)), B.PA_ERR_INVALID_ARG, "non-negative"),
    (dict(hint=(1, 10, -2)), B.PA_ERR_INVALID_ARG, "non-negative"),
    (dict(hint=(20, 10)), B.PA_ERR_INVALID_ARG, "max_query_len"),
    (dict(hint=(1, 1000)), B.PA_ERR_WORKSPACE, "workspace"),
    (dict(hint=(1, 1000), ws=FAKE + 16, wsb=1 << 30), B.PA_ERR_WORKSPACE, "aligned"),
    (dict(scale=float("nan")), B.PA_ERR_INVALID_ARG, "NaN"),
])
def test_attention_rejects_bad_arguments(lib, kw, status, text):
    assert call_attention(lib, **kw) == status
    assert text in msg(lib), msg(lib)


@pytest.mark.parametrize("kw, status, text", [
    (dict(hint=(1, 1000, 0, -512)), B.PA_ERR_INVALID_ARG, "non-negative"),
    (dict(hint=(1, 1000, 0, 256)), B.PA_ERR_INVALID_ARG, "multiple of 512"),
    (dict(hint=(1, 512, 0, 512), bt=T(B.PA_I32, [3, 64])), B.PA_ERR_INVALID_ARG, "below max_seq_len"),
    (dict(hint=(1, 1000, 0, 512)), B.PA_ERR_INVALID_ARG, "within the block tables"),
    (dict(hint=(2, 1000, 0, 512), bt=T(B.PA_I32, [3, 64])), B.PA_ERR_UNSUPPORTED, "decode rows"),
])
def test_shared_prefix_hint_is_validated(lib, kw, status, text):
    assert call_attention(lib, **kw) == status
    assert text in msg(lib), msg(lib)


def test_shared_prefix_with_prefill_rows_refused_over_fp8(lib):
    n, hq, hkv, d, bs, nb, mb = 3, 8, 2, 128, 16, 40, 64
    args = [ctypes.byref(x) for x in (
        T(B.PA_F16, [n, hq, d]), T(B.PA_F8E4M3, [nb, hkv, bs, d]), T(B.PA_F8E4M3, [nb, hkv, bs, d]),
        T(B.PA_I32, [n, mb]), T(B.PA_I32, [n]), T(B.PA_I32, [n + 1]))]
    r = lib.pa_attention_fp8(*args, ctypes.c_float(0.1), ctypes.byref(T(B.PA_F16, [n, hq, d])),
                             ctypes.byref(B.PABatchHint(2, 1000, 0, 512)),
                             ctypes.byref(B.PAKVScales(0.5, 0.5)), None, 0, None)
    assert r == B.PA_ERR_UNSUPPORTED and "decode rows" in msg(lib)


def test_timing_hook_rejects_unknown_kernel(lib):
    assert lib.pa_set_timing_events(7, None, None) == B.PA_ERR_INVALID_ARG
    assert "PA_TIMED" in msg(lib)
    assert lib.pa_set_timing_events(1, None, None) == B.PA_OK
    assert lib.pa_set_timing_events(2, None, None) == B.PA_OK


def test_attention_null_tensor(lib):
    r = lib.pa_attention(None, None, None, None, None, None, ctypes.c_float(1.0), None, None, None,
                         0, None)
    assert r == B.PA_ERR_INVALID_ARG and "NULL" in msg(lib)


def test_empty_batch_is_a_no_op(lib):
    # zero query rows: valid, nothing to launch, no CUDA call needed
    assert call_attention(lib, q=T(B.PA_F16, [0, 8, 64]), out=T(B.PA_F16, [0, 8, 64]),
                          hint=(0, 0)) == B.PA_OK


def call_cache(lib, k=None, v=None, kc=None, vc=None, sm=None):
    t, hkv, d, bs, nb = 5, 2, 128, 32, 10
    k = k or T(B.PA_F16, [t, hkv, d])
    v = v or T(B.PA_F16, [t, hkv, d])
    kc = kc or T(B.PA_F16, [nb, hkv, bs, d])
    vc = vc or T(B.PA_F16, [nb, hkv, bs, d])
    sm = sm or T(B.PA_I64, [t])
    return lib.pa_reshape_and_cache(ctypes.byref(k), ctypes.byref(v), ctypes.byref(kc),
                                    ctypes.byref(vc), ctypes.byref(sm), None)


@pytest.mark.parametrize("kw, status, text", [
    (dict(sm=T(B.PA_I32, [5])), B.PA_ERR_INVALID_ARG, "int64"),
    (dict(sm=T(B.PA_I64, [4])), B.PA_ERR_INVALID_ARG, "slot_mapping"),
    (dict(k=T(B.PA_F16, [5, 3, 128])), B.PA_ERR_INVALID_ARG, "matching the pool"),
    (dict(v=T(B.PA_F16, [5, 2, 128], stride=[260, 128, 1])), B.PA_ERR_INVALID_ARG, "multiple of 8"),
    (dict(k=T(B.PA_F16, [5, 2, 128], stride=[128, 128, 1])), B.PA_ERR_INVALID_ARG, "token stride"),
    (dict(kc=T(B.PA_F16, [10, 2, 32, 80]), vc=T(B.PA_F16, [10, 2, 32, 80])), B.PA_ERR_UNSUPPORTED,
     "head_dim"),
    (dict(v=T(B.PA_F16, [5, 2, 128], data=FAKE + 8)), B.PA_ERR_INVALID_ARG, "alignment"),
])
def test_reshape_and_cache_rejects_bad_arguments(lib, kw, status, text):
    assert call_cache(lib, **kw) == status
    assert text in msg(lib), msg(lib)


def test_reshape_and_cache_empty_is_a_no_op(lib):
    assert call_cache(lib, k=T(B.PA_F16, [0, 2, 128]), v=T(B.PA_F16, [0, 2, 128]),
                      sm=T(B.PA_I64, [0])) == B.PA_OK


def test_workspace_size_formula(lib):
    # fp32 o[T][Hq][P][d] + m + l, each region rounded up to 256 B; 0 when one partition suffices
    assert pa.workspace_size(32, 64, 128, 512) == 0
    rows = 32 * 64 * 16
    up = lambda x: (x + 255) // 256 * 256
    assert pa.workspace_size(32, 64, 128, 8192) == up(rows * 128 * 4) + 2 * up(rows * 4)
    assert pa.workspace_size(3, 5, 64, 513) == up(30 * 64 * 4) + 2 * up(30 * 4)


def test_batch_descriptor_from_host():
    d = pa.BatchDescriptor.from_host([5, 40, 17], [5, 1, 2], [[3, 0, 0], [1, 2, 4], [7, 6, 0]],
                                     block_size=16, device="cpu")
    assert d.query_start_loc.tolist() == [0, 5, 6, 8]
    assert d.slot_mapping.tolist() == [48, 49, 50, 51, 52, 4 * 16 + 7, 7 * 16 + 15, 6 * 16 + 0]
    assert d.max_query_len == 5 and d.max_seq_len == 40 and d.num_prefill_seqs == 2


def test_step_slot_mapping_rejects_bad_descriptors(lib):
    with pytest.raises(B.PAError, match="query_len"):
        pa.BatchDescriptor.from_host([5, 4], [5, 5], [[0], [1]], block_size=16, device="cpu")
    with pytest.raises(B.PAError, match="too short"):
        pa.BatchDescriptor.from_host([17], [1], [[0]], block_size=16, device="cpu")
    i32 = lambda *x: (ctypes.c_int32 * max(1, len(x)))(*x)
    qsl, sm = i32(0, 0), (ctypes.c_int64 * 1)()
    assert lib.pa_step_slot_mapping(1, i32(3), i32(2), i32(9), 1, 1, 16, qsl, sm, 1) == \
        B.PA_ERR_INVALID_ARG
    assert "holds 1 entries, 2 needed" in msg(lib)
    assert list(qsl) == [0, 0]  # nothing written
    # an idle sequence (no new token) needs no table entry
    d = pa.BatchDescriptor.from_host([0, 3], [0, 1], [[0], [5]], block_size=16, device="cpu")
    assert d.query_start_loc.tolist() == [0, 0, 1] and d.slot_mapping.tolist() == [5 * 16 + 2]


def test_wait_limit_range(lib):
    assert lib.pa_set_wait_limit(0) == B.PA_ERR_INVALID_ARG
    assert "wait limit" in msg(lib)
    assert lib.pa_set_wait_limit(10**11) == B.PA_ERR_INVALID_ARG
    assert lib.pa_set_wait_limit(2 * 10**9) == B.PA_OK
    # the self-test hook refuses limits that would hold a GPU for long, before any CUDA call
    assert lib.pa_selftest_wait_timeout(10**9, None) == B.PA_ERR_INVALID_ARG
    assert lib.pa_selftest_wait_timeout(10, None) == B.PA_ERR_INVALID_ARG


# --------------------------------------------------------------- FP8 cache entry points

def call_attention_fp8(lib, k_scale=0.05, v_scale=0.02, hint=(1, 100), pool_dtype=B.PA_F8E4M3,
                       null_scales=False):
    n, hq, hkv, d, bs, nb, mb = 3, 8, 2, 128, 16, 40, 8
    q = T(B.PA_F16, [n, hq, d])
    kc = T(pool_dtype, [nb, hkv, bs, d])
    vc = T(pool_dtype, [nb, hkv, bs, d])
    out = T(B.PA_F16, [n, hq, d])
    sc = None if null_scales else ctypes.byref(B.PAKVScales(k_scale, v_scale))
    return lib.pa_attention_fp8(ctypes.byref(q), ctypes.byref(kc), ctypes.byref(vc),
                                ctypes.byref(T(B.PA_I32, [n, mb])), ctypes.byref(T(B.PA_I32, [n])),
                                ctypes.byref(T(B.PA_I32, [n + 1])), ctypes.c_float(0.1),
                                ctypes.byref(out), ctypes.byref(B.PABatchHint(*hint)), sc, None,
                                0, None)


@pytest.mark.parametrize("kw, status, text", [
    (dict(pool_dtype=B.PA_F16), B.PA_ERR_INVALID_ARG, "float8_e4m3"),
    (dict(k_scale=0.0), B.PA_ERR_INVALID_ARG, "finite and > 0"),
    (dict(v_scale=-1.0), B.PA_ERR_INVALID_ARG, "finite and > 0"),
    (dict(k_scale=float("nan")), B.PA_ERR_INVALID_ARG, "finite and > 0"),
    (dict(v_scale=float("inf")), B.PA_ERR_INVALID_ARG, "finite and > 0"),
    (dict(null_scales=True), B.PA_ERR_INVALID_ARG, "scales is NULL"),
])
def test_attention_fp8_rejects_bad_arguments(lib, kw, status, text):
    assert call_attention_fp8(lib, **kw) == status
    assert text in msg(lib), msg(lib)


def test_fp16_entry_rejects_an_fp8_pool(lib):
    kc = T(B.PA_F8E4M3, [40, 2, 16, 64])
    assert call_attention(lib, kc=kc, vc=T(B.PA_F8E4M3, [40, 2, 16, 64])) == B.PA_ERR_INVALID_ARG
    assert "float16" in msg(lib)


def test_reshape_fp8_checks_scales_and_dtype(lib):
    t, hkv, d, bs, nb = 5, 2, 128, 16, 10
    args = [ctypes.byref(x) for x in (T(B.PA_F16, [t, hkv, d]), T(B.PA_F16, [t, hkv, d]),
                                       T(B.PA_F8E4M3, [nb, hkv, bs, d]),
                                       T(B.PA_F8E4M3, [nb, hkv, bs, d]), T(B.PA_I64, [t]))]
    assert lib.pa_reshape_and_cache_fp8(*args, None, None) == B.PA_ERR_INVALID_ARG
    assert "scales" in msg(lib)
    bad = ctypes.byref(B.PAKVScales(1.0, 0.0))
    assert lib.pa_reshape_and_cache_fp8(*args, bad, None) == B.PA_ERR_INVALID_ARG
    empty = [ctypes.byref(x) for x in (T(B.PA_F16, [0, hkv, d]), T(B.PA_F16, [0, hkv, d]),
                                        T(B.PA_F8E4M3, [nb, hkv, bs, d]),
                                        T(B.PA_F8E4M3, [nb, hkv, bs, d]), T(B.PA_I64, [0]))]
    ok = ctypes.byref(B.PAKVScales(0.5, 0.25))
    assert lib.pa_reshape_and_cache_fp8(*empty, ok, None) == B.PA_OK


def test_stream_error_word_registry(lib):
    # fake stream handles and word addresses: registration touches no device memory
    words = [0x100000 + 16 * i for i in range(65)]
    try:
        for i in range(64):
            assert lib.pa_set_stream_error_word(0x5000 + i, words[i]) == B.PA_OK
        assert lib.pa_set_stream_error_word(0x5000 + 64, words[64]) == B.PA_ERR_INVALID_ARG
        assert "64 streams" in msg(lib)
        # re-registering a stream replaces its word; releasing one frees a place
        assert lib.pa_set_stream_error_word(0x5000 + 3, words[64]) == B.PA_OK
        assert lib.pa_set_stream_error_word(0x5000 + 7, None) == B.PA_OK
        assert lib.pa_set_stream_error_word(0x5000 + 64, words[7]) == B.PA_OK
        assert lib.pa_set_stream_error_word(0x6000, 0x100002) == B.PA_ERR_INVALID_ARG  # misaligned
        assert "aligned" in msg(lib)
    finally:
        for i in range(65):
            lib.pa_set_stream_error_word(0x5000 + i, None)
