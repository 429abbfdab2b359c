"""GPU parity of the bfloat16 path (q, new tokens, pools and out all bf16) against the oracle.

The scatter-write is a bit copy, compared over the whole pool.  Attention is compared with the
fp64 oracle run on the same bf16 values.  The bar is the fp16 bar scaled by 8: bfloat16 keeps 7
fraction bits where binary16 keeps 10, so each rounding the kernels make (P as an MMA operand,
the output) is 2^3 times coarser, and nothing else in the arithmetic changes (fp32
accumulation, the same exp2 and merge).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_decode, small_long_chunks, small_mixed, small_spec

pytestmark = pytest.mark.gpu

MAX_ABS, MAX_REL_L2 = 8 * 2e-3, 8 * 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available()
    pa.get_device_error()


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run(b, shared_prefix_tokens=0):
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev))
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.attention(q, kc, vc, b.block_tables.to(dev), b.seq_lens.to(dev),
                 b.query_start_loc.to(dev), b.scale, out, b.max_query_len, b.max_seq_len,
                 num_prefill_seqs=b.num_prefill_seqs, shared_prefix_tokens=shared_prefix_tokens)
    st, bits = pa.get_device_error()
    assert st == 0, (st, bits, pa.last_error())
    assert out.dtype == torch.bfloat16
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


def check_cache(b, kc, vc):
    rk, rv = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                      b.slot_mapping)
    assert np.array_equal(_u16(kc), rk), "k_cache bits differ"
    assert np.array_equal(_u16(vc), rv), "v_cache bits differ"


def shared(n=30, prefix=1024, d=128, bs=16, hq=28, hkv=4, seed=9600):
    g = torch.Generator().manual_seed(seed)
    priv = [1, 16, 513] + torch.randint(1, 900, (n - 3,), generator=g).tolist()
    return W.build_batch("bf16_shared", [W.SeqSpec(prefix + p, 1) for p in priv],
                         num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                         seed_base=seed, shared_prefix_len=prefix)


CASES = {
    # decode kernel (one and two head groups of 8 per warp), merge, single-partition rows
    "decode_d128_bs16_g4": (lambda: small_decode(), 0),
    "decode_d64_bs32_g16": (lambda: small_decode(d=64, bs=32, hq=32, hkv=2, seed=9106), 0),
    "decode_d128_bs32_g7": (lambda: small_decode(bs=32, hq=28, hkv=4, seed=9107), 0),
    "decode_d64_bs16_g1": (lambda: small_decode(d=64, hq=4, hkv=4, seed=9105), 0),
    # prefill chunks longer than one Q tile (two-tile kernel) next to decode rows
    "mixed_d128_bs16_g4": (lambda: small_mixed(), 0),
    "mixed_d64_bs32_g8": (lambda: small_mixed(d=64, bs=32, hq=16, hkv=2, seed=9207), 0),
    # verify rows that fit one Q tile (key-parity kernel)
    "spec_d128_bs16_g8": (lambda: small_spec(), 0),
    "spec_d64_bs32_g4": (lambda: small_spec(d=64, bs=32, hq=16, hkv=4, seed=9401), 0),
    # the shared-prefix pass
    "shared_d128_bs16_g7": (lambda: shared(), 1024),
    "shared_d64_bs32_g8": (lambda: shared(d=64, bs=32, hq=64, hkv=8, seed=9601), 512),
    # long contexts, beside decode rows and alone
    "long_d128_bs16_g4": (lambda: small_long_chunks(seed=9502), 0),
    "long_alone_d128_bs16_g4": (lambda: small_long_chunks(seed=9505, decode=False), 0),
    # verify rows of at most q_len x G = 8 columns: the decode kernel with causal limits
    "verify_d128_bs16_g2": (lambda: W.build_batch(
        "bf16_verify", [W.SeqSpec(L, q) for L, q in [(3, 3), (600, 4), (1030, 2), (77, 1),
                                                     (4, 4), (2000, 3)]],
        num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=16, seed_base=9606), 0),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bf16_matches_oracle(name):
    make, sp = CASES[name]
    b = W.to_bf16(make())
    kc, vc, out = run(b, sp)
    check_cache(b, kc, vc)
    assert_close(out, oracle.attention_batch(b))


def test_bf16_full_70b_decode():
    """8 sequences of 8192 keys, 64 q / 8 kv heads: every row."""
    b = W.to_bf16(W.llama70b_decode(8))
    kc, vc, out = run(b)
    check_cache(b, kc, vc)
    assert_close(out, oracle.attention_batch(b))


def test_bf16_full_mixed_step_sampled_rows():
    """The 4 x 512-row chunks and 128 decode rows of the mixed step: every decode row and a
    seeded sample of each chunk's rows (with its first and last)."""
    b = W.WORKLOADS["mixed_step_bs16_bf16"]()
    kc, vc, out = run(b)
    check_cache(b, kc, vc)
    g = torch.Generator().manual_seed(4243)
    mask = np.zeros(b.num_tokens, dtype=np.uint8)
    for s, spec in enumerate(b.seqs):
        r0 = int(b.query_start_loc[s])
        pick = torch.randperm(spec.query_len, generator=g)[:24].tolist()
        for i in set(pick) | {0, spec.query_len - 1}:
            mask[r0 + i] = 1
    ref = oracle.attention_batch(b, row_mask=mask)
    assert_close(out, ref, np.nonzero(mask)[0])
