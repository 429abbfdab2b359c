"""GPU parity of the shared-prefix pass (hint shared_prefix_tokens > 0).

The prefix that every sequence shares is attended once for all decode rows, in 512-key
partitions, and merged with each sequence's own partitions by the log-sum-exp rule.  The result
is plain attention over each sequence's whole context, so the bar is the fp64 oracle's, as for
every other path; the output with and without the pass must agree to the same bar.  Sequences
whose table differs inside the prefix, or that end inside it, are reported, not computed.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as Bd
from paged_kv_cache_290_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MAX_REL_L2 = 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available()
    pa.get_device_error()


def shared_case(n, prefix, d, bs, hq, hkv, seed):
    """n decode rows behind a shared prefix; private continuations ragged around block and
    partition edges (1 key past the prefix, 511/512/513), the rest seeded in [1, 1400]."""
    edge = [1, 15, 16, 17, 511, 512, 513, 1100][:n]
    g = torch.Generator().manual_seed(seed)
    priv = edge + torch.randint(1, 1401, (n - len(edge),), generator=g).tolist()
    order = torch.randperm(n, generator=g).tolist()
    seqs = [W.SeqSpec(prefix + priv[i], 1) for i in order]
    return W.build_batch(f"shared_prefix_{n}x{prefix}_d{d}_bs{bs}_g{hq // hkv}", seqs,
                         num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                         seed_base=seed, shared_prefix_len=prefix)


def run(b, shared_prefix_tokens, tables=None, seq_lens=None):
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev))
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    bt = (b.block_tables if tables is None else tables).to(dev)
    sl = (b.seq_lens if seq_lens is None else seq_lens).to(dev)
    pa.attention(q, kc, vc, bt, sl, b.query_start_loc.to(dev), b.scale, out, b.max_query_len,
                 b.max_seq_len, shared_prefix_tokens=shared_prefix_tokens)
    return out, pa.get_device_error()


def assert_close(out, ref):
    o = out.detach().cpu().double().numpy()
    assert np.isfinite(o).all(), "non-finite output"
    err = np.abs(o - ref)
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3e}"
    assert rel <= MAX_REL_L2, f"rel L2 err {rel:.3e}"


def oracle_of(b):
    return oracle.attention_batch(b)


# (rows, prefix, d, bs, q heads, kv heads): Q tiles of 128 // G tokens, so each case spans
# several CTAs with a ragged last one; G = 12 leaves 8 padding rows in every tile.  Small grids
# run one Q tile per CTA; the last cases' grids (640 rows, 2 Q tiles of 16 per CTA, 8 kv heads:
# 160 CTAs) fill the GPU and run on the two-Q-tile kernel.  An even number of prefix partitions
# goes two per CTA (the merge skips the second's slot); an odd one, one per CTA.
CASES = {
    "g7_d128_bs16_p512": (40, 512, 128, 16, 28, 4),
    "g4_d128_bs32_p1024": (70, 1024, 128, 32, 32, 8),
    "g8_d64_bs16_p512": (20, 512, 64, 16, 16, 2),
    "g1_d64_bs32_p1536": (300, 1536, 64, 32, 4, 4),
    "g16_d128_bs16_p512": (12, 512, 128, 16, 32, 2),
    "g12_d128_bs32_p2048": (25, 2048, 128, 32, 24, 2),
    "pair_g8_d128_bs16_p512": (640, 512, 128, 16, 64, 8),
    "pair_g8_d128_bs16_p1024": (640, 1024, 128, 16, 64, 8),
}


@pytest.mark.parametrize("name", list(CASES))
def test_shared_prefix_pass_matches_oracle(name):
    n, prefix, d, bs, hq, hkv = CASES[name]
    b = shared_case(n, prefix, d, bs, hq, hkv, seed=9500 + sum(map(ord, name)))
    ref = oracle_of(b)
    out, (st, bits) = run(b, prefix)
    assert st == 0, (st, bits, pa.last_error())
    assert_close(out, ref)
    # a shorter declared prefix (fewer shared partitions) is just as valid
    if prefix > 512:
        out2, (st, bits) = run(b, 512)
        assert st == 0, (st, bits)
        assert_close(out2, ref)
    plain, (st, _) = run(b, 0)
    assert st == 0
    assert_close(plain, ref)


@pytest.mark.parametrize("name", ["g7_d128_bs16_p512", "g8_d64_bs16_p512", "g4_d128_bs32_p1024"])
def test_shared_prefix_pass_over_fp8(name):
    """Over an FP8 pool the pass widens the prefix's codes into fp16 in shared memory."""
    n, prefix, d, bs, hq, hkv = CASES[name]
    b = W.to_fp8(shared_case(n, prefix, d, bs, hq, hkv, seed=9700 + d), k_scale=0.03,
                 v_scale=0.02)
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev),
                         k_scale=b.k_scale, v_scale=b.v_scale)
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.attention(q, kc, vc, b.block_tables.to(dev), b.seq_lens.to(dev),
                 b.query_start_loc.to(dev), b.scale, out, b.max_query_len, b.max_seq_len,
                 shared_prefix_tokens=prefix, k_scale=b.k_scale, v_scale=b.v_scale)
    st, bits = pa.get_device_error()
    assert st == 0, (st, bits, pa.last_error())
    rk, rv = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    ref = oracle.attention_fp8(b.q, rk, rv, b.block_tables, b.seq_lens, b.query_start_loc,
                               b.scale, b.k_scale, b.v_scale)
    assert_close(out, ref)


def test_full_prefix_shared_decode_with_the_pass():
    """160 rows behind a 2048-key prefix (4 shared partitions), 28 q / 4 kv heads: every row."""
    b = W.WORKLOADS["prefix_shared_decode"]()
    out, (st, bits) = run(b, b.meta["shared_prefix_len"])
    assert st == 0, (st, bits, pa.last_error())
    assert_close(out, oracle_of(b))


def test_table_that_differs_in_the_prefix_is_reported():
    b = shared_case(20, 1024, 128, 16, 32, 8, seed=9561)
    bt = b.block_tables.clone()
    bt[7, 40] = b.nan_block       # a valid block id, but not the shared one
    _, (st, _) = run(b, 1024, tables=bt)
    assert st == Bd.PA_ERR_DESCRIPTOR
    _, (st, _) = run(b, 1024)      # the error word was cleared; the intact batch runs clean
    assert st == 0


def test_sequence_ending_inside_the_prefix_is_reported():
    b = shared_case(20, 1024, 128, 16, 32, 8, seed=9562)
    sl = b.seq_lens.clone()
    sl[3] = 1024                   # no key of its own past the declared prefix
    _, (st, _) = run(b, 1024, seq_lens=sl)
    assert st == Bd.PA_ERR_DESCRIPTOR
