"""The bounded-wait failure path, driven to its end without a fault.

Every mbarrier wait in the kernels gives up after a limit, sets the timeout bit of the device
error word and returns, so a copy that never lands cannot hang the GPU.  Here the self-test hook
launches one warp that waits, with a 1 ms limit, on an mbarrier nothing ever arrives on (no copy
is issued, so nothing is in flight when it gives up).  The host must read PA_ERR_TIMEOUT with
bit 1, and an ordinary attention call on the same device afterwards must still match the fp64
oracle.  A short wait limit on real calls (pa_set_wait_limit) must not change their results:
legitimate waits last microseconds.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as B
from _cases import small_mixed

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
MAX_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_290_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    lib = B.load_library()
    pa.get_device_error()
    return lib


def _step_matches_oracle(b):
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev))
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.attention(q, kc, vc, b.block_tables.to(dev), b.seq_lens.to(dev),
                 b.query_start_loc.to(dev), b.scale, out, b.max_query_len, b.max_seq_len,
                 num_prefill_seqs=b.num_prefill_seqs)
    st, bits = pa.get_device_error()
    assert st == B.PA_OK, (st, bits, pa.last_error())
    o = out.cpu().double().numpy()
    ref = oracle.attention_batch(b)
    err = np.abs(o - ref)
    assert np.isfinite(o).all()
    assert err.max() <= MAX_ABS
    assert np.linalg.norm(err) / np.linalg.norm(ref) <= MAX_REL_L2


def test_wait_runs_out_and_reports_timeout(lib):
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    assert lib.pa_selftest_wait_timeout(1_000_000, stream.cuda_stream) == B.PA_OK, pa.last_error()
    st, bits = pa.get_device_error()
    elapsed = time.perf_counter() - t0
    assert st == B.PA_ERR_TIMEOUT, (st, bits)
    assert bits & 1, bits
    assert "timed out" in pa.last_error()
    assert elapsed < 5.0  # gave up after its own limit, far below the 2 s default
    # the word was cleared by the read, and the context is still usable
    assert pa.get_device_error() == (B.PA_OK, 0)
    _step_matches_oracle(small_mixed(seed=9811))


def test_short_wait_limit_leaves_real_calls_unchanged(lib):
    # 1 ms is three orders of magnitude above any legitimate wait of these kernels
    assert lib.pa_set_wait_limit(1_000_000) == B.PA_OK
    try:
        _step_matches_oracle(small_mixed(seed=9812))
    finally:
        assert lib.pa_set_wait_limit(B.PA_WAIT_LIMIT_DEFAULT_NS) == B.PA_OK
