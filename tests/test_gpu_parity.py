"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on seeded inputs.

Bars: reshape_and_cache is bit-exact over the whole pool (NaN sentinels and untouched bytes
included); fp16 attention output has max |err| <= 2e-3 and ||err||_2 / ||ref||_2 <= 1e-3
against the fp64 oracle.  Invariants that hold exactly on the GPU too: re-permuting physical
blocks and un-aliasing a shared prefix give bit-identical outputs, and a 1-token context returns
V exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_decode, small_long_chunks, small_mixed, small_prefix, small_spec

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-3
MAX_REL_L2 = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.init()
    pa.get_device_error()  # start from a clear device error word


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_step(b, write=True, pool=None):
    """reshape_and_cache (pre-step pool + new tokens) then attention, like one serving step."""
    dev = "cuda"
    if pool is None:
        kc = (b.k_cache_pre if write else b.k_cache).to(dev)
        vc = (b.v_cache_pre if write else b.v_cache).to(dev)
    else:
        kc, vc = pool
    if write:
        pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, b.slot_mapping.to(dev))
    q = b.q.to(dev)
    out = torch.full_like(q, float("nan"))
    pa.attention(q, kc, vc, b.block_tables.to(dev), b.seq_lens.to(dev),
                 b.query_start_loc.to(dev), b.scale, out, b.max_query_len, b.max_seq_len,
                 num_prefill_seqs=b.num_prefill_seqs)
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
    return err.max(), rel


SMALL = {
    "tiny_decode": W.tiny_decode,
    "decode_d128_bs16_g4": lambda: small_decode(),
    "decode_d128_bs32_g8": lambda: small_decode(bs=32, hq=64, hkv=8, seed=9104),
    "decode_d64_bs16_g1": lambda: small_decode(d=64, hq=4, hkv=4, seed=9105),
    "decode_d64_bs32_g16": lambda: small_decode(d=64, bs=32, hq=32, hkv=2, seed=9106),
    "decode_d128_bs16_g7": lambda: small_decode(hq=28, hkv=4, seed=9107),
    "decode_d128_bs16_g12": lambda: small_decode(hq=24, hkv=2, seed=9108),
    "mixed_d128_bs16_g4": lambda: small_mixed(),
    "mixed_d128_bs32_g8": lambda: small_mixed(bs=32, hq=16, hkv=2, seed=9207),
    "mixed_d64_bs16_g7": lambda: small_mixed(d=64, hq=28, hkv=4, seed=9208),
    "mixed_d64_bs32_g1": lambda: small_mixed(d=64, bs=32, hq=4, hkv=4, seed=9209),
    "mixed_d128_bs16_g16": lambda: small_mixed(hq=32, hkv=2, seed=9210),
    "prefix_d128_bs16": lambda: small_prefix(),
    "spec_d128_bs16_g8": lambda: small_spec(),
    "spec_d64_bs32_g4": lambda: small_spec(d=64, bs=32, hq=16, hkv=4, seed=9401),
    "spec_d128_bs32_g16": lambda: small_spec(bs=32, hq=32, hkv=2, seed=9402),
    # group sizes that do not divide 128: a Q tile holds 128 // G whole tokens
    "mixed_d64_bs16_g3": lambda: small_mixed(d=64, hq=6, hkv=2, seed=9211),
    # 84 tokens per CTA (two tiles of 42): a 170-row chunk needs 3 CTAs, not ceil(170 / 85)
    "chunk170_d64_bs16_g3": lambda: W.build_batch(
        "chunk170_g3", [W.SeqSpec(200, 170), W.SeqSpec(90, 1), W.SeqSpec(300, 40)],
        num_q_heads=6, num_kv_heads=2, head_dim=64, block_size=16, seed_base=9213),
    "mixed_d128_bs32_g6": lambda: small_mixed(bs=32, hq=12, hkv=2, seed=9212),
    # long contexts, beside decode rows (launch slices) and alone
    "long_d128_bs16_g4": lambda: small_long_chunks(),
    "long_d64_bs32_g8": lambda: small_long_chunks(d=64, bs=32, hq=16, hkv=2, seed=9501),
    "long_alone_d128_bs16_g4": lambda: small_long_chunks(seed=9503, decode=False),
    "long_alone_d64_bs32_g8": lambda: small_long_chunks(d=64, bs=32, hq=16, hkv=2, seed=9504,
                                                        decode=False),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases_match_oracle(name):
    b = SMALL[name]()
    kc, vc, out = gpu_step(b)
    rk, rv = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                      b.slot_mapping)
    assert np.array_equal(_u16(kc), rk), "k_cache bytes differ"
    assert np.array_equal(_u16(vc), rv), "v_cache bytes differ"
    ref = oracle.attention_batch(b)
    assert_close(out, ref)


@pytest.mark.parametrize("sign", [0.0, -1.0])
@pytest.mark.parametrize("d", [128, 64])
def test_zero_and_negative_scale_match_oracle(sign, d):
    """The prefill softmax folds a positive scale into the exponent and pre-scales otherwise;
    scale 0 turns every visible key's weight into 1 (the mean of V), scale -1/sqrt(d) flips
    which key dominates.  Both, on decode and prefill rows, must agree with the oracle.  (Much
    larger |scale| makes single keys dominate, and the fp16 rounding of outputs of magnitude 2-4
    alone then reaches the 2e-3 bar.)"""
    b = small_mixed(d=d, hq=16, hkv=4, seed=9230 + d)
    b.scale = sign / float(np.sqrt(d))
    _, _, out = gpu_step(b)
    assert_close(out, oracle.attention_batch(b))


@pytest.mark.parametrize("d, bs, hq, hkv", [(128, 16, 32, 4), (64, 32, 16, 4), (128, 32, 32, 2)])
def test_both_prefill_kernels_match_oracle(d, bs, hq, hkv):
    """Verify rows take one of three paths by the hint's max_query_len: the decode kernel when
    q_len x G <= 8 (max_query_len 2, G = 4), the key-parity prefill kernel while a chunk fits
    one 128-row Q tile, and the two-Q-tile kernel beyond (an upper bound is allowed).  All must
    agree with the oracle."""
    b = small_spec(d=d, bs=bs, hq=hq, hkv=hkv, seed=9410 + d + bs)
    if hq // hkv == 4:  # at most 2 rows per sequence: 8 columns, the decode kernel's share
        b = W.build_batch("spec2", [W.SeqSpec(L, q) for L, q in
                                    [(2, 2), (37, 2), (515, 2), (130, 1), (17, 2), (96, 2),
                                     (1, 1), (1100, 2)]],
                          num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                          seed_base=9415 + d)
    dev = "cuda"
    ref = oracle.attention_batch(b)
    args = [x.to(dev) for x in (b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                b.query_start_loc)]
    for max_q in (b.max_query_len, 16, 200):
        out = torch.full_like(args[0], float("nan"))
        pa.attention(*args, b.scale, out, max_q, b.max_seq_len,
                     num_prefill_seqs=b.num_prefill_seqs)
        assert pa.get_device_error() == (0, 0)
        assert_close(out, ref)


@pytest.mark.parametrize("case", ["many_sequences", "many_pairs"])
def test_prefill_many_sequences_and_tiles(case):
    """A batch of 140 short verify chunks (the scan spans two rounds of the CTA's threads) and
    one of nine 512-row chunks at 16 rows per CTA (288 CTAs per head): both must give the
    oracle's result."""
    g = torch.Generator().manual_seed(9500)
    if case == "many_sequences":   # 140 short verify chunks
        ctx = torch.randint(1, 41, (140,), generator=g).tolist()
        ql = torch.randint(2, 5, (140,), generator=g).tolist()
        b = W.build_batch("plan_seqs", [W.SeqSpec(c + q, q) for c, q in zip(ctx, ql)],
                          num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                          seed_base=9501)
    else:                          # 9 chunks of 512 rows, 16 rows per CTA: 288 pairs
        ctx = torch.randint(0, 101, (9,), generator=g).tolist()
        b = W.build_batch("plan_pairs", [W.SeqSpec(c + 512, 512) for c in ctx],
                          num_q_heads=32, num_kv_heads=2, head_dim=64, block_size=16,
                          seed_base=9502)
    _, _, out = gpu_step(b, write=False)
    assert_close(out, oracle.attention_batch(b))


@pytest.mark.parametrize("name", ["decode_d128_bs16_g4", "mixed_d128_bs32_g8", "prefix_d128_bs16"])
def test_block_placement_is_bit_invariant(name):
    b = SMALL[name]()
    _, _, o1 = gpu_step(b, write=False)
    _, _, o2 = gpu_step(W.repermute(b, seed=5), write=False)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_aliased_prefix_equals_private_copies_bitwise():
    b = small_prefix()
    _, _, o1 = gpu_step(b, write=False)
    _, _, o2 = gpu_step(W.unalias_prefix(b), write=False)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_one_token_context_returns_v_exactly():
    for d, bs, hq, hkv in [(64, 16, 8, 2), (128, 32, 64, 8), (128, 16, 28, 4)]:
        b = W.build_batch("one", [W.SeqSpec(1, 1)] * 5, num_q_heads=hq, num_kv_heads=hkv,
                          head_dim=d, block_size=bs, seed_base=9600 + d + bs)
        _, _, out = gpu_step(b)
        want = b.v_new.repeat_interleave(hq // hkv, dim=1)
        assert torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))


def test_padding_slots_and_reuse_of_output_buffer():
    """Padding tokens (slot -1) write nothing; rows of idle sequences (q_len 0) are untouched."""
    b = small_mixed(seed=9211)
    kc, vc, out = gpu_step(b)
    assert np.isfinite(out.cpu().double().numpy()).all()
    rk, _ = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                     b.slot_mapping)
    assert np.array_equal(_u16(kc), rk)


def test_bad_block_id_is_skipped_and_reported():
    """A block id outside the pool is caught by the kernels' own bounds check before any copy:
    the work item is skipped and the device error word reports it."""
    b = small_mixed(seed=9212)
    bt = b.block_tables.clone()
    s = next(i for i, x in enumerate(b.seqs) if x.query_len == 1)
    bt[s, 0] = b.num_blocks + 7
    dev = "cuda"
    kc, vc = b.k_cache.to(dev), b.v_cache.to(dev)
    out = torch.zeros_like(b.q, device=dev)
    pa.attention(b.q.to(dev), kc, vc, bt.to(dev), b.seq_lens.to(dev), b.query_start_loc.to(dev),
                 b.scale, out, b.max_query_len, b.max_seq_len)
    st, bits = pa.get_device_error()
    assert st == pa.binding.PA_ERR_OUT_OF_RANGE and bits & 4
    st, bits = pa.get_device_error()
    assert st == 0 and bits == 0


def test_slot_past_pool_is_skipped_and_reported():
    b = W.tiny_decode()
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    sm = b.slot_mapping.clone()
    sm[1] = b.num_blocks * b.block_size + 3
    pa.reshape_and_cache(b.k_new.to(dev), b.v_new.to(dev), kc, vc, sm.to(dev))
    st, bits = pa.get_device_error()
    assert st == pa.binding.PA_ERR_OUT_OF_RANGE and bits & 2
    rk, _ = oracle.reshape_and_cache(b.k_new[[0, 2, 3]], b.v_new[[0, 2, 3]], b.k_cache_pre,
                                     b.v_cache_pre, b.slot_mapping[[0, 2, 3]])
    assert np.array_equal(_u16(kc), rk)


def test_hint_too_small_is_reported():
    b = small_decode(seed=9109)
    dev = "cuda"
    out = torch.zeros_like(b.q, device=dev)
    need = pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim, 600)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    pa.attention(b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev), b.block_tables.to(dev),
                 b.seq_lens.to(dev), b.query_start_loc.to(dev), b.scale, out, 1, 600,
                 workspace=ws)
    st, bits = pa.get_device_error()
    assert st == pa.binding.PA_ERR_DESCRIPTOR and bits & 16


def test_workspace_reused_and_never_cleared():
    """Every partial is written before it is read: a workspace full of random bytes, reused by
    three calls in a row, gives the oracle's result every time."""
    b = small_decode(seed=9110)
    dev = "cuda"
    need = pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim, b.max_seq_len)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device=dev)
    ref = oracle.attention_batch(b)
    args = [x.to(dev) for x in (b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                b.query_start_loc)]
    for _ in range(3):
        out = torch.full_like(args[0], float("nan"))
        pa.attention(*args, b.scale, out, b.max_query_len, b.max_seq_len, workspace=ws)
        st, bits = pa.get_device_error()
        assert st == 0, (st, bits)
        assert_close(out, ref)


def test_prefill_longer_than_hint_is_reported():
    """A prefill chunk with more rows than the hint's max_query_len is skipped and reported."""
    b = small_mixed(seed=9213)
    dev = "cuda"
    out = torch.zeros_like(b.q, device=dev)
    pa.attention(b.q.to(dev), b.k_cache.to(dev), b.v_cache.to(dev), b.block_tables.to(dev),
                 b.seq_lens.to(dev), b.query_start_loc.to(dev), b.scale, out, 16, b.max_seq_len)
    st, bits = pa.get_device_error()
    assert st == pa.binding.PA_ERR_DESCRIPTOR and bits & 16


def test_prefill_sequence_count_hint():
    """num_prefill_seqs = 0 (not known) covers every sequence; the exact count gives the same
    bits; a count below the batch's is reported, and the chunks it covers are still exact."""
    b = small_mixed(seed=9214)
    dev = "cuda"
    assert b.num_prefill_seqs == 4
    args = [x.to(dev) for x in (b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                b.query_start_loc)]
    outs = {}
    for n in (0, 4, 2, 8):
        out = torch.full_like(args[0], float("nan"))
        pa.attention(*args, b.scale, out, b.max_query_len, b.max_seq_len, num_prefill_seqs=n)
        outs[n] = (out, pa.get_device_error())
    assert outs[0][1] == (0, 0) and outs[4][1] == (0, 0)
    assert torch.equal(outs[0][0], outs[4][0])
    assert_close(outs[4][0], oracle.attention_batch(b))
    st, bits = outs[2][1]
    assert st == pa.binding.PA_ERR_DESCRIPTOR and bits & 16
    # the first two prefill chunks (in batch order) and every decode row are still computed
    covered = [s for s, spec in enumerate(b.seqs) if spec.query_len > 1][:2]
    rows = [r for s, spec in enumerate(b.seqs) if spec.query_len == 1 or s in covered
            for r in range(int(b.query_start_loc[s]), int(b.query_start_loc[s + 1]))]
    assert torch.equal(outs[2][0][rows], outs[4][0][rows])
    # a count equal to the number of sequences skips the decode launches: the batch's one-row
    # sequences are then reported, and every prefill row is still exact
    st, bits = outs[8][1]
    assert st == pa.binding.PA_ERR_DESCRIPTOR and bits & 16
    rows = [r for s, spec in enumerate(b.seqs) if spec.query_len > 1
            for r in range(int(b.query_start_loc[s]), int(b.query_start_loc[s + 1]))]
    assert torch.equal(outs[8][0][rows], outs[4][0][rows])


# ------------------------------------------------------------------ the five full-size workloads

def _full(name, sample_prefill_rows=None, whole_longest_chunk=False):
    """One full-size step against the oracle.  With ``sample_prefill_rows`` the prefill chunks
    are sampled (first, last and a seeded sample of rows); ``whole_longest_chunk`` adds every
    row of the chunk with the longest context (all its 128-row tiles at full size)."""
    b = W.WORKLOADS[name]()
    kc, vc, out = gpu_step(b)
    rk, rv = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                      b.slot_mapping)
    assert np.array_equal(_u16(kc), rk)
    assert np.array_equal(_u16(vc), rv)
    mask = None
    if sample_prefill_rows:
        # every decode row, plus the first, last and a seeded sample of each prefill chunk's rows
        g = torch.Generator().manual_seed(4242)
        mask = np.zeros(b.num_tokens, dtype=np.uint8)
        for s, spec in enumerate(b.seqs):
            r0 = int(b.query_start_loc[s])
            if spec.query_len == 1:
                mask[r0] = 1
            elif spec.query_len > 1:
                pick = torch.randperm(spec.query_len, generator=g)[:sample_prefill_rows].tolist()
                for i in set(pick) | {0, spec.query_len - 1}:
                    mask[r0 + i] = 1
        if whole_longest_chunk:
            s = max((s for s, spec in enumerate(b.seqs) if spec.query_len > 1),
                    key=lambda s: b.seqs[s].seq_len)
            mask[int(b.query_start_loc[s]):int(b.query_start_loc[s + 1])] = 1
    ref = oracle.attention_batch(b, row_mask=mask)
    rows = None if mask is None else np.nonzero(mask)[0]
    return assert_close(out, ref, rows)


def test_full_tiny_decode():
    _full("tiny_decode")


def test_full_llama8b_decode():
    _full("llama8b_decode")


def test_full_llama70b_32x8k_decode():
    _full("llama70b_32x8k_decode")


def test_full_prefix_shared_decode():
    _full("prefix_shared_decode")


@pytest.mark.parametrize("bs", [16, 32])
def test_full_mixed_step(bs):
    _full(f"mixed_step_bs{bs}", sample_prefill_rows=24, whole_longest_chunk=bs == 16)


def test_full_spec_verify():
    _full("spec_verify")
