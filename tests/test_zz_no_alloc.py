"""pa_attention_static_scratch: the allocation-free variant of pa_attention.

Some callers cannot allocate device memory (a plugin whose host program owns all device memory,
or a serving path where cudaMalloc/cudaFree would block or synchronise), so this entry point
takes its split-context scratch from a fixed array inside the library instead of a
caller-provided workspace.  The test calls it through the C ABI twice in a row on the same
inputs and checks both outputs against the existing pa_attention entry point, with the same
tolerance as the parity tests; it also checks that a batch needing more scratch than the array
holds is refused.  The file is named to be collected last, and it needs no state from other
tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as B
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_decode

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
MAX_REL_L2 = 1e-3
STATIC_SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_290_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = B.load_library()
    pa.get_device_error()
    return lib


def _static_call(lib, q, kc, vc, bt, sl, qsl, scale, out, max_q, max_s):
    descs = [B.describe(x) for x in (q, kc, vc, bt, sl, qsl)]
    hint = B.PABatchHint(max_q, max_s)
    return lib.pa_attention_static_scratch(*[ctypes.byref(d) for d in descs],
                                           ctypes.c_float(scale), ctypes.byref(B.describe(out)),
                                           ctypes.byref(hint),
                                           torch.cuda.current_stream().cuda_stream)


def _close(a, b):
    a = a.detach().cpu().double().numpy()
    b = b.detach().cpu().double().numpy()
    err = np.abs(a - b)
    assert np.isfinite(a).all()
    assert err.max() <= MAX_ABS
    assert np.linalg.norm(err) / max(np.linalg.norm(b), 1e-30) <= MAX_REL_L2


@pytest.mark.parametrize("make", [lambda: small_decode(seed=9700),
                                  lambda: W.llama70b_decode(8, keep_contiguous=False,
                                                            keep_pre=False)])
def test_static_scratch_matches_workspace_entry_point_twice(lib, make):
    b = make()
    dev = "cuda"
    q, kc, vc = b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev)
    bt, sl, qsl = b.block_tables.to(dev), b.seq_lens.to(dev), b.query_start_loc.to(dev)
    assert b.max_seq_len > 512  # several partitions, so the scratch is really used
    need = pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim, b.max_seq_len)
    assert 0 < need <= STATIC_SCRATCH_BYTES

    ref = torch.empty_like(q)
    pa.attention(q, kc, vc, bt, sl, qsl, b.scale, ref, b.max_query_len, b.max_seq_len)
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _static_call(lib, q, kc, vc, bt, sl, qsl, b.scale, out, b.max_query_len,
                          b.max_seq_len)
        assert rc == B.PA_OK, pa.last_error()
        st, bits = pa.get_device_error()
        assert st == 0, (st, bits)
        _close(out, ref)


def test_static_scratch_refuses_oversized_batch(lib):
    b = small_decode(seed=9701)
    dev = "cuda"
    q = b.q.to(dev)
    out = torch.zeros_like(q)
    big = 1 << 22  # a max_seq_len whose partials exceed the static array
    assert pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim, big) > STATIC_SCRATCH_BYTES
    rc = _static_call(lib, q, b.k_cache.to(dev), b.v_cache.to(dev), b.block_tables.to(dev),
                      b.seq_lens.to(dev), b.query_start_loc.to(dev), b.scale, out, 1, big)
    assert rc == B.PA_ERR_WORKSPACE
    assert "static array" in pa.last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing ran
