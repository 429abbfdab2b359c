"""Device errors reported per stream (pa_set_stream_error_word).

A caller serving several streams registers a word of its own for each; a slot outside the pool
planted in one stream's scatter-write must show up in that stream's word only: the other
stream's word and the device's shared word stay clean, and reading a word clears it.
"""
import pytest
import torch

import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as B
from paged_kv_cache_290_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available()
    pa.get_device_error()


def test_errors_go_to_the_stream_that_made_them():
    b = W.tiny_decode()
    dev = "cuda"
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = torch.zeros(1, dtype=torch.int32, device=dev)
    w2 = torch.zeros(1, dtype=torch.int32, device=dev)
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    k_new, v_new = b.k_new.to(dev), b.v_new.to(dev)
    bad = b.slot_mapping.clone()
    bad[1] = b.num_blocks * b.block_size + 3  # past the pool: skipped and reported
    bad = bad.to(dev)
    good = b.slot_mapping.to(dev)
    torch.cuda.synchronize()
    B.set_stream_error_word(s1, w1)
    B.set_stream_error_word(s2, w2)
    try:
        with torch.cuda.stream(s1):
            pa.reshape_and_cache(k_new, v_new, kc, vc, bad, stream=s1)
        s1.synchronize()
        with torch.cuda.stream(s2):
            pa.reshape_and_cache(k_new, v_new, kc, vc, good, stream=s2)
        s2.synchronize()
        assert int(w1.item()) & 2 and int(w2.item()) == 0
        assert pa.get_device_error(s2) == (B.PA_OK, 0)
        assert pa.get_device_error() == (B.PA_OK, 0)  # the device's word saw nothing
        st, bits = pa.get_device_error(s1)
        assert st == B.PA_ERR_OUT_OF_RANGE and bits & 2
        assert int(w1.item()) == 0  # read and cleared
    finally:
        B.set_stream_error_word(s1, None)
        B.set_stream_error_word(s2, None)
    # unregistered again: the same planted slot now reports through the device's word
    with torch.cuda.stream(s1):
        pa.reshape_and_cache(k_new, v_new, kc, vc, bad, stream=s1)
    st, bits = pa.get_device_error(s1)
    assert st == B.PA_ERR_OUT_OF_RANGE and bits & 2 and int(w1.item()) == 0
