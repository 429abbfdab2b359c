"""GPU parity of the FP8 (E4M3) KV cache against the oracle.

The scatter-write must store exactly the oracle's codes (round to nearest even of x * (1/scale),
saturating at +-448), bit for bit over the whole pool.  Decode, verify and prefill attention over
the FP8 pool are compared with the oracle's fp64 attention over the dequantised cache, under the
same bar as the fp16 path.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as Bd
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_decode, small_long_chunks, small_mixed, small_spec

pytestmark = pytest.mark.gpu

MAX_ABS, MAX_REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available()
    pa.get_device_error()


def _u8(t):
    return t.detach().cpu().contiguous().numpy()


def run_fp8(b, write=True):
    dev = "cuda"
    kc = (b.k_cache_pre if write else b.k_cache).to(dev)
    vc = (b.v_cache_pre if write else b.v_cache).to(dev)
    if write:
        pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev),
                             k_scale=b.k_scale, v_scale=b.v_scale)
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.attention(q, kc, vc, b.block_tables.to(dev), b.seq_lens.to(dev),
                 b.query_start_loc.to(dev), b.scale, out, b.max_query_len, b.max_seq_len,
                 num_prefill_seqs=b.num_prefill_seqs, k_scale=b.k_scale, v_scale=b.v_scale)
    st, bits = pa.get_device_error()
    assert st == 0, (st, bits, pa.last_error())
    return kc, vc, out


def assert_close(out, ref, rows=None):
    o = out.detach().cpu().double().numpy()
    if rows is not None:
        o, ref = o[rows], ref[rows]
    assert np.isfinite(o).all(), "non-finite output"
    err = np.abs(o - ref)
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3e}"
    assert rel <= MAX_REL_L2, f"rel L2 err {rel:.3e}"


@pytest.mark.parametrize("d, bs, k_scale, v_scale", [(128, 16, 0.005, 1.0), (64, 32, 1 / 32, 0.5)])
def test_fp8_scatter_is_bit_exact(d, bs, k_scale, v_scale):
    """k_scale 0.005 pushes |x / scale| past 448 (saturation); v_scale 1 keeps small values in
    the subnormal range; a mixed batch has padding slots and many tokens per sequence."""
    b = W.to_fp8(small_mixed(d=d, bs=bs, hq=16, hkv=4, seed=9240 + d), k_scale, v_scale)
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev),
                         k_scale=b.k_scale, v_scale=b.v_scale)
    assert pa.get_device_error() == (0, 0)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk), "k_cache bytes differ"
    assert np.array_equal(_u8(vc), rv), "v_cache bytes differ"
    if k_scale < 0.01:
        assert (rk == 0x7E).any() and (rk == 0xFE).any(), "saturation not exercised"
    assert ((rv & 0x78) == 0).any(), "subnormals not exercised"


CASES = {
    "d128_bs16_g4": lambda: small_decode(),
    "d128_bs32_g8": lambda: small_decode(bs=32, hq=64, hkv=8, seed=9104),
    "d64_bs16_g1": lambda: small_decode(d=64, hq=4, hkv=4, seed=9105),
    "d64_bs32_g16": lambda: small_decode(d=64, bs=32, hq=32, hkv=2, seed=9106),
    "d128_bs16_g7": lambda: small_decode(hq=28, hkv=4, seed=9107),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_decode_matches_oracle(name):
    b = W.to_fp8(CASES[name](), k_scale=0.03, v_scale=0.02)
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


def test_fp8_full_70b_decode():
    """8 sequences of 8192 keys, 64 q / 8 kv heads, 16 partitions each: every row."""
    b = W.WORKLOADS["llama70b_8x8k_decode_fp8"]()
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


@pytest.mark.parametrize("name, make", [
    ("spec_d128_bs16_g4", lambda: small_spec(hq=16, hkv=4, seed=9242)),
    ("spec_d64_bs32_g2", lambda: small_spec(d=64, bs=32, hq=8, hkv=4, seed=9243)),
])
def test_fp8_verify_rows_match_oracle(name, make):
    """Speculative-verify rows (q_len x G <= 32) over an FP8 cache run on the decode kernel
    with a causal limit per query row."""
    b = W.to_fp8(make(), k_scale=0.03, v_scale=0.02)
    assert b.max_query_len * (b.num_q_heads // b.num_kv_heads) <= 32
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


def test_fp8_full_spec_verify():
    """64 sequences verifying 1-5 drafts over 512-4096 keys, 32 q / 8 kv heads: every row."""
    b = W.to_fp8(W.spec_verify())
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


PREFILL = {
    # chunks longer than one Q tile (two-tile kernel) next to decode rows
    "mixed_d128_bs16_g4": lambda: small_mixed(hq=16, hkv=4, seed=9241),
    "mixed_d64_bs32_g8": lambda: small_mixed(d=64, bs=32, hq=16, hkv=2, seed=9244),
    # verify rows past 32 columns (key-parity kernel)
    "spec_d128_bs16_g8": lambda: small_spec(seed=9245),
    # long contexts, chunks alone
    "long_alone_d128_bs16_g4": lambda: small_long_chunks(seed=9246, decode=False),
}


@pytest.mark.parametrize("name", list(PREFILL))
def test_fp8_prefill_matches_oracle(name):
    """Prefill chunks over an FP8 pool: the prefill kernels widen each K/V tile of codes into
    fp16 in shared memory (exact) and apply the scales; the bar is the fp16 one."""
    b = W.to_fp8(PREFILL[name](), k_scale=0.03, v_scale=0.02)
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


def test_fp8_full_mixed_step_sampled_rows():
    """The mixed step over an FP8 pool: every decode row and a seeded sample of each chunk's
    rows (with its first and last)."""
    b = W.to_fp8(W.mixed_step(16))
    kc, vc, out = run_fp8(b)
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    assert np.array_equal(_u8(kc), rk) and np.array_equal(_u8(vc), rv)
    g = torch.Generator().manual_seed(4244)
    mask = np.zeros(b.num_tokens, dtype=np.uint8)
    for s, spec in enumerate(b.seqs):
        r0 = int(b.query_start_loc[s])
        pick = torch.randperm(spec.query_len, generator=g)[:24].tolist()
        for i in set(pick) | {0, spec.query_len - 1}:
            mask[r0 + i] = 1
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale, row_mask=mask)
    assert_close(out, ref, np.nonzero(mask)[0])
