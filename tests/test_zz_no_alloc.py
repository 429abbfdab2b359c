"""pa_attention_static_scratch: the allocation-free variant of pa_attention.

Some callers cannot allocate device memory (a plugin whose host program owns all device memory,
or a serving path where cudaMalloc/cudaFree would block or synchronise), so this entry point
takes its split-context scratch from a fixed array inside the library instead of a
caller-provided workspace.  It runs the same kernels on the same inputs as pa_attention, so the
test, calling it through the C ABI, asks for the same bits, not just the parity tolerance:
  - on two calls in a row on the same inputs;
  - on a chain of different batches, so that each call finds the array holding the previous
    call's partials (a larger batch first, then smaller ones): nothing in the array needs to
    start at zero;
  - on a mixed batch (prefill chunks beside decode rows).
A batch needing more scratch than the array holds must be refused before anything runs.  The
file is named to be collected last, and it needs no state from other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as B
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_decode, small_mixed

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


def _static_call(lib, q, kc, vc, bt, sl, qsl, scale, out, max_q, max_s, n_prefill=0):
    descs = [B.describe(x) for x in (q, kc, vc, bt, sl, qsl)]
    hint = B.PABatchHint(max_q, max_s, n_prefill, 0)
    return lib.pa_attention_static_scratch(*[ctypes.byref(d) for d in descs],
                                           ctypes.c_float(scale), ctypes.byref(B.describe(out)),
                                           ctypes.byref(hint),
                                           torch.cuda.current_stream().cuda_stream)


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


class _OnDevice:
    """A batch's tensors on the GPU, with its pa_attention (caller workspace) output."""

    def __init__(self, b, write=False):
        dev = "cuda"
        self.b = b
        self.q = b.q.to(dev)
        if write:  # the step's new tokens go through the scatter-write first
            self.kc, self.vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
            pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), self.kc, self.vc,
                                 b.slot_mapping.to(dev))
        else:
            self.kc, self.vc = b.k_cache.to(dev), b.v_cache.to(dev)
        self.bt, self.sl = b.block_tables.to(dev), b.seq_lens.to(dev)
        self.qsl = b.query_start_loc.to(dev)
        self.ref = torch.empty_like(self.q)
        pa.attention(self.q, self.kc, self.vc, self.bt, self.sl, self.qsl, b.scale, self.ref,
                     b.max_query_len, b.max_seq_len, num_prefill_seqs=b.num_prefill_seqs)
        st, bits = pa.get_device_error()
        assert st == 0, (st, bits)

    def static(self, lib):
        b = self.b
        out = torch.full_like(self.q, float("nan"))
        rc = _static_call(lib, self.q, self.kc, self.vc, self.bt, self.sl, self.qsl, b.scale, out,
                          b.max_query_len, b.max_seq_len, b.num_prefill_seqs)
        assert rc == B.PA_OK, pa.last_error()
        st, bits = pa.get_device_error()
        assert st == 0, (st, bits)
        return out


def _close_to_oracle(out, b):
    o = out.cpu().double().numpy()
    ref = oracle.attention_batch(b)
    err = np.abs(o - ref)
    assert np.isfinite(o).all()
    assert err.max() <= MAX_ABS
    assert np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30) <= MAX_REL_L2


@pytest.mark.parametrize("make", [lambda: small_decode(seed=9700),
                                  lambda: W.llama70b_decode(8, keep_contiguous=False,
                                                            keep_pre=False)])
def test_static_scratch_matches_workspace_entry_point_twice(lib, make):
    x = _OnDevice(make())
    b = x.b
    assert b.max_seq_len > 512  # several partitions, so the scratch is really used
    need = pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim, b.max_seq_len)
    assert 0 < need <= STATIC_SCRATCH_BYTES
    for _ in range(2):
        assert torch.equal(_bits(x.static(lib)), _bits(x.ref))


def test_static_scratch_keeps_no_state_between_batches(lib):
    # the 8 x 8k batch fills 16 partitions per row; the smaller batches after it find the array
    # holding its partials (and each other's), and must still give pa_attention's bits
    chain = [_OnDevice(W.llama70b_decode(8, keep_contiguous=False, keep_pre=False)),
             _OnDevice(small_decode(seed=9702)),
             _OnDevice(small_mixed(seed=9703), write=True),
             _OnDevice(small_decode(seed=9704, lens=(600, 2000, 1, 513)))]
    for x in chain:
        assert torch.equal(_bits(x.static(lib)), _bits(x.ref))
    _close_to_oracle(chain[-1].static(lib), chain[-1].b)


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
