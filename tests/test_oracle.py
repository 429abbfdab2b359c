"""CPU pins for the fp64 oracle: each test ties it to something other than itself.

Pins (no GPU): the pages' KV-sizing arithmetic, the binary16 definition, closed forms,
invariants the pages state for paging (placement does not matter, aliased prefix pages equal
private copies, paged equals contiguous), a float64 library attention (torch SDPA) and an
independent NumPy brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_290_gb300 import workloads as W
from _brute import brute_attention
from _cases import small_decode, small_mixed, small_prefix, small_spec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- pages' arithmetic (golden)

def test_kv_sizing_matches_pages():
    """Llama-3-70B KV per token, per 8k session, and for 32 sessions, as the deck prints."""
    g = json.load(open(os.path.join(GOLDEN, "kv_sizing.json")))
    f = g["factors"]
    per_tok = f["k_and_v"] * f["layers"] * f["kv_dims"] * f["bytes_per_elem"]
    assert per_tok == g["bytes_per_token_all_layers"] == 320 * 1024
    assert g["kv_heads_times_head_dim"][0] * g["kv_heads_times_head_dim"][1] == f["kv_dims"]
    assert per_tok // f["layers"] == g["bytes_per_token_per_layer"]
    assert per_tok * g["session_tokens"] == g["session_bytes_all_layers"]
    assert g["session_bytes_all_layers"] / 2**30 == g["session_gib_all_layers"]
    assert g["sessions"] * g["session_bytes_all_layers"] / 2**30 == g["all_sessions_gib_all_layers"]
    assert (g["sessions"] * g["session_tokens"] * g["bytes_per_token_per_layer"]
            == g["all_sessions_bytes_one_layer"])


def test_70b_workload_is_one_gib_of_kv_per_layer():
    """The 32 x 8k decode workload holds exactly the 80 GB / 80 layers the deck sizes."""
    g = json.load(open(os.path.join(GOLDEN, "kv_sizing.json")))
    b = W.llama70b_decode(keep_contiguous=False, keep_pre=False)
    used = b.num_unique_blocks
    per_block = b.num_kv_heads * b.block_size * b.head_dim * 2
    assert 2 * used * per_block == g["all_sessions_bytes_one_layer"]
    assert b.num_kv_heads * b.head_dim == g["factors"]["kv_dims"]
    assert b.num_blocks == used + 64
    assert sum(s.seq_len for s in b.seqs) == 32 * 8192


# ---------------------------------------------------------------- binary16 decoding

def test_half_to_double_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # a few hand-checked values of the format
    assert oracle.half_to_double([0x3C00])[0] == 1.0
    assert oracle.half_to_double([0xC000])[0] == -2.0
    assert oracle.half_to_double([0x0001])[0] == 2.0 ** -24
    assert oracle.half_to_double([0x7BFF])[0] == 65504.0


# ---------------------------------------------------------------- reshape_and_cache

@pytest.mark.parametrize("make", [W.tiny_decode, small_mixed,
                                  lambda: small_mixed(d=64, bs=32, hq=8, hkv=8, seed=9201)])
def test_reshape_and_cache_places_new_tokens(make):
    """Writing the step's tokens into the pre-step pool reproduces the generator's placement of
    every token (an independent torch-indexing scatter), bit for bit; padding slots (-1) and all
    other bytes, NaN sentinels included, are untouched."""
    b = make()
    kc, vc = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                      b.slot_mapping)
    assert np.array_equal(kc, _bits(b.k_cache))
    assert np.array_equal(vc, _bits(b.v_cache))
    assert (b.slot_mapping < 0).sum() == (3 if "mixed" in b.name else 0)


def test_copy_blocks_moves_whole_blocks_only():
    """Block-level closed form: each destination equals its source as it was before the call,
    every other block keeps its bytes, an out-of-pool pair is skipped, and copying a block to
    a scratch block and back restores the pool."""
    g = torch.Generator().manual_seed(77)
    kc = torch.randint(0, 1 << 16, (9, 2, 16, 64), generator=g, dtype=torch.int32).to(torch.int16)
    vc = torch.randint(0, 1 << 16, (9, 2, 16, 64), generator=g, dtype=torch.int32).to(torch.int16)
    k0 = kc.numpy().view(np.uint16)
    v0 = vc.numpy().view(np.uint16)
    pairs = torch.tensor([[3, 7], [7, 1], [2, 99], [0, 5]], dtype=torch.int32)
    k1, v1 = oracle.copy_blocks(kc, vc, pairs)
    for blk in range(9):
        src = {7: 3, 1: 7, 5: 0}.get(blk, blk)  # [7, 1] copies block 7's old contents
        assert np.array_equal(k1[blk], k0[src]) and np.array_equal(v1[blk], v0[src])
    k2, v2 = oracle.copy_blocks(torch.from_numpy(k1.view(np.int16)),
                                torch.from_numpy(v1.view(np.int16)),
                                torch.tensor([[1, 3]], dtype=torch.int32))
    assert np.array_equal(k2[3], k0[7]) and np.array_equal(v2[3], v0[7])


def test_reshape_and_cache_rejects_out_of_range_slot():
    b = W.tiny_decode()
    sm = b.slot_mapping.clone()
    sm[0] = b.num_blocks * b.block_size
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre, sm)


# ---------------------------------------------------------------- closed forms

def _hand_case(scale):
    """Three keys in two blocks of size 2 (physical blocks 3 then 1, the rest NaN), d = 2.
    A 2-row chunk over a 1-token context: row 0 sits at position 1, row 1 at position 2."""
    nan = float("nan")
    kc = torch.full((4, 1, 2, 2), nan, dtype=torch.float16)
    vc = torch.full((4, 1, 2, 2), nan, dtype=torch.float16)
    K = [(0, 0), (1, 0), (0, 1)]
    V = [(1, 0), (0, 1), (1, 1)]
    place = [(3, 0), (3, 1), (1, 0)]
    for (blk, off), kk, vv in zip(place, K, V):
        kc[blk, 0, off] = torch.tensor(kk, dtype=torch.float16)
        vc[blk, 0, off] = torch.tensor(vv, dtype=torch.float16)
    q = torch.tensor([[[1, 0], [-1, 0]], [[0, 2], [0, 2]]], dtype=torch.float16)  # [T=2,Hq=2,d]
    bt = torch.tensor([[3, 1]], dtype=torch.int32)
    return oracle.attention(q, kc, vc, bt, torch.tensor([3], dtype=torch.int32),
                            torch.tensor([0, 2], dtype=torch.int32), scale)


def test_worked_example_closed_form():
    """Hand-derived softmax weights: row 0 sees keys 0, 1 only (causal, bottom-right), row 1
    sees all three; both query heads share the single KV head (GQA group of 2)."""
    e = math.e
    for scale in (1.0, 0.5):
        o = _hand_case(scale)
        a = math.exp(scale)                      # row 0 head 0: scores (0, scale)
        assert np.allclose(o[0, 0], [1 / (1 + a), a / (1 + a)], rtol=0, atol=1e-15)
        b_ = math.exp(-scale)                    # row 0 head 1: scores (0, -scale)
        assert np.allclose(o[0, 1], [1 / (1 + b_), b_ / (1 + b_)], rtol=0, atol=1e-15)
        c = math.exp(2 * scale)                  # row 1: scores (0, 0, 2*scale)
        want = (1 + c) / (2 + c)
        assert np.allclose(o[1, 0], [want, want], rtol=0, atol=1e-15)
        assert np.allclose(o[1, 1], [want, want], rtol=0, atol=1e-15)
    assert e > 2  # keeps the closed form honest about which constant it uses


def test_one_token_context_returns_v_exactly():
    """seq_len 1: the single weight is exp(0)/exp(0) = 1, so the output is that token's V,
    per query head through its GQA group (head h reads kv head h // G)."""
    b = W.build_batch("one", [W.SeqSpec(1, 1)] * 3, num_q_heads=8, num_kv_heads=2,
                      head_dim=64, block_size=16, seed_base=9400)
    o = oracle.attention_batch(b)
    vnew = b.v_new.double().numpy()                  # [3, Hkv, d]
    for h in range(8):
        assert np.array_equal(o[:, h], vnew[:, h // 4])


def test_identical_keys_give_mean_of_v():
    """All keys equal (or scale 0): every weight is equal, so the output is the mean of the
    visible V rows."""
    b = small_mixed(d=64, bs=16, hq=8, hkv=2, seed=9401)
    for scale in (0.0, None):
        kc = b.k_cache.clone()
        if scale is None:
            kc[~torch.isnan(kc)] = 0.75
        o = oracle.attention(b.q, kc, b.v_cache, b.block_tables, b.seq_lens, b.query_start_loc,
                             0.0 if scale == 0.0 else b.scale)
        v = b.v_contig.double().numpy()
        for s, spec in enumerate(b.seqs):
            base = int(b.kv_start[s])
            for i in range(spec.query_len):
                row = int(b.query_start_loc[s]) + i
                vis = spec.seq_len - spec.query_len + i + 1
                for h in range(8):
                    want = v[base:base + vis, h // 4].mean(0)
                    assert np.allclose(o[row, h], want, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- invariants of paging

CASES = [W.tiny_decode, small_mixed, lambda: small_mixed(d=64, bs=32, hq=28, hkv=4, seed=9202),
         small_prefix, lambda: small_decode(d=64, bs=32, hq=16, hkv=2, seed=9102),
         lambda: small_spec(d=64, bs=32, hq=16, hkv=2, seed=9403)]


@pytest.mark.parametrize("make", CASES)
def test_paged_equals_contiguous_bitwise(make):
    """De-paging through the block table reproduces each sequence's contiguous K/V exactly:
    the paged result is bit-identical to the same attention on one contiguous region per
    sequence (the layout the pages contrast paging with)."""
    b = make()
    o_paged = oracle.attention_batch(b)
    o_contig = oracle.attention_contiguous(b.q, b.k_contig, b.v_contig, b.kv_start, b.seq_lens,
                                           b.query_start_loc, b.scale)
    assert np.array_equal(o_paged, o_contig, equal_nan=True)
    assert np.isfinite(o_paged).all()


@pytest.mark.parametrize("make", CASES)
def test_physical_placement_does_not_matter(make):
    """Logical pages may sit anywhere in physical memory: re-permuting every block gives a
    bit-identical result."""
    b = make()
    o1 = oracle.attention_batch(b)
    o2 = oracle.attention_batch(W.repermute(b, seed=77))
    assert np.array_equal(o1, o2)


def test_aliased_prefix_equals_private_copies():
    """Sequences that start the same way share prefix pages; the result equals giving each
    sequence its own copy of those pages."""
    b = small_prefix()
    assert (b.block_tables[:, :4] == b.block_tables[0, :4]).all()
    u = W.unalias_prefix(b)
    assert len(set(u.block_tables[:, 0].tolist())) == b.num_seqs
    assert np.array_equal(oracle.attention_batch(b), oracle.attention_batch(u))


def test_nan_sentinels_never_reach_the_output():
    """Spare blocks, block tails and table padding are NaN, yet every output is finite: the
    oracle reads only positions below seq_len."""
    b = small_mixed(seed=9203)
    bt = b.block_tables
    assert torch.isnan(b.k_cache[b.nan_block]).all()
    o = oracle.attention_batch(b)
    assert np.isfinite(o).all()
    tails = 0
    for s, spec in enumerate(b.seqs):
        nb = -(-spec.seq_len // b.block_size)
        assert (bt[s, nb:] == b.nan_block).all()
        if spec.seq_len % b.block_size:
            last = int(bt[s, nb - 1])
            assert torch.isnan(b.k_cache[last, :, spec.seq_len % b.block_size:]).all()
            tails += 1
    assert tails > 0


# ---------------------------------------------------------------- independent references

@pytest.mark.parametrize("make", CASES)
def test_matches_numpy_brute_force(make):
    b = make()
    o = oracle.attention_batch(b)
    ref = brute_attention(b.q, b.k_contig, b.v_contig, b.kv_start, b.seq_lens,
                          b.query_start_loc, b.scale)
    assert np.allclose(o, ref, rtol=0, atol=1e-12, equal_nan=True)


def test_matches_torch_sdpa_float64():
    """Library special cases: a decode row attends to all L keys (no mask); a chunk with no
    prior context is ordinary causal self-attention.  KV heads are expanded to query heads
    with repeat_interleave(G), i.e. head h reads kv head h // G."""
    sdpa = torch.nn.functional.scaled_dot_product_attention
    seqs = [W.SeqSpec(200, 1), W.SeqSpec(37, 37), W.SeqSpec(1, 1), W.SeqSpec(96, 96)]
    b = W.build_batch("sdpa", seqs, num_q_heads=28, num_kv_heads=4, head_dim=128,
                      block_size=16, seed_base=9500)
    o = oracle.attention_batch(b)
    g = 7
    for s, spec in enumerate(b.seqs):
        r0 = int(b.query_start_loc[s])
        base = int(b.kv_start[s])
        q = b.q[r0:r0 + spec.query_len].double().permute(1, 0, 2)[None]
        k = b.k_contig[base:base + spec.seq_len].double().permute(1, 0, 2)[None]
        v = b.v_contig[base:base + spec.seq_len].double().permute(1, 0, 2)[None]
        k, v = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)
        causal = spec.query_len > 1
        assert not causal or spec.query_len == spec.seq_len
        ref = sdpa(q, k, v, is_causal=causal, scale=b.scale)[0].permute(1, 0, 2).numpy()
        assert np.allclose(o[r0:r0 + spec.query_len], ref, rtol=0, atol=1e-12)


def test_chunk_row_equals_decode_at_its_position():
    """Row i of a prefill chunk sees exactly what a decode step at the same position sees:
    the first seq_len - q_len + i + 1 keys."""
    b = small_mixed(seed=9204)
    o = oracle.attention_batch(b)
    for s, spec in enumerate(b.seqs):
        if spec.query_len < 2:
            continue
        for i in (0, spec.query_len // 2, spec.query_len - 1):
            pos = spec.seq_len - spec.query_len + i
            row = int(b.query_start_loc[s]) + i
            sl = torch.tensor([pos + 1], dtype=torch.int32)
            qsl = torch.tensor([0, 1], dtype=torch.int32)
            od = oracle.attention(b.q[row:row + 1], b.k_cache, b.v_cache,
                                  b.block_tables[s:s + 1], sl, qsl, b.scale)
            assert np.array_equal(od[0], o[row])


# ---------------------------------------------------------------- split-context merge

@pytest.mark.parametrize("part", [512, 16, 7])
def test_split_context_merge_equals_unsplit(part):
    """Partitions combined with the log-sum-exp rule equal unsplit softmax attention."""
    b = small_decode(d=64, bs=16, hq=16, hkv=4, seed=9103)
    o = oracle.attention_batch(b)
    os_ = oracle.attention_batch(b, partition_size=part)
    assert np.allclose(o, os_, rtol=0, atol=1e-12)
    bm = small_mixed(seed=9205)
    assert np.allclose(oracle.attention_batch(bm), oracle.attention_batch(bm, partition_size=part),
                       rtol=0, atol=1e-12)


# ---------------------------------------------------------------- descriptor handling

def test_row_mask_limits_rows():
    b = small_mixed(seed=9206)
    mask = np.zeros(b.num_tokens, dtype=np.uint8)
    mask[[0, 5, b.num_tokens - 1]] = 1
    o = oracle.attention_batch(b, row_mask=mask)
    full = oracle.attention_batch(b)
    assert np.array_equal(o[mask == 1], full[mask == 1])
    assert np.isnan(o[mask == 0]).all()


def test_descriptor_errors():
    b = W.tiny_decode()
    bad = b.seq_lens.clone()
    bad[0] = 0                                   # query_len 1 > seq_len 0
    with pytest.raises(oracle.OracleError):
        oracle.attention(b.q, b.k_cache, b.v_cache, b.block_tables, bad, b.query_start_loc,
                         b.scale)
    bt = b.block_tables.clone()
    bt[0, 0] = b.num_blocks                       # block id past the pool
    with pytest.raises(oracle.OracleError):
        oracle.attention(b.q, b.k_cache, b.v_cache, bt, b.seq_lens, b.query_start_loc, b.scale)


# ---------------------------------------------------------------- FP8 (E4M3) KV cache

def test_e4m3_decode_known_values():
    """Values the E4M3 format fixes: zero, smallest subnormal 2^-9, largest subnormal 7 * 2^-9,
    smallest normal 2^-6, one, two, the largest finite 448, negative zero and one, and the two
    NaN codes."""
    c = [0x00, 0x01, 0x07, 0x08, 0x38, 0x40, 0x7E, 0x80, 0xB8]
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 2.0, 448.0, -0.0, -1.0]
    got = oracle.e4m3_decode(c)
    assert got.tolist() == want and np.signbit(got[7])
    assert np.isnan(oracle.e4m3_decode([0x7F, 0xFF])).all()


def test_e4m3_table_is_monotone_symmetric_and_exact_in_fp16():
    pos = oracle.e4m3_decode(np.arange(0x7F))
    assert (np.diff(pos) > 0).all()
    assert np.array_equal(oracle.e4m3_decode(np.arange(0x7F) | 0x80), -pos)
    assert np.array_equal(pos.astype(np.float16).astype(np.float64), pos)


def test_e4m3_encode_matches_torch_in_range():
    """Round to nearest, ties to even, against torch's float8_e4m3fn conversion: random values
    inside +-448 and every exact midpoint between neighbouring codes."""
    pos = oracle.e4m3_decode(np.arange(0x7F))
    g = np.random.default_rng(290)
    mids = (pos[1:] + pos[:-1]) / 2
    x = np.concatenate([g.normal(0, 30, 20000), g.uniform(-447.9, 447.9, 20000), mids, -mids,
                        pos, -pos, [2.0 ** -11, -2.0 ** -11]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)
    assert np.array_equal(oracle.e4m3_encode(pos), np.arange(0x7F))  # round trip


def test_e4m3_encode_saturates_and_keeps_sign_and_nan():
    x = np.array([448.0, 463.9, 464.0, 500.0, 1e30, np.inf, -500.0, -np.inf, np.nan, -0.0],
                 dtype=np.float32)
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 6 + [0xFE, 0xFE, 0x7F, 0x80]


def test_fp8_scatter_writes_codes_of_scaled_tokens():
    """Each new token lands at its slot as the code of x * (1/scale) (float32 product, torch's
    conversion as the independent encoder); every other byte of the pool is unchanged."""
    b = W.to_fp8(small_mixed(d=64, hq=8, hkv=2, seed=9231), k_scale=0.05, v_scale=0.02)
    kc, vc = oracle.reshape_and_cache_fp8(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                          b.slot_mapping, b.k_scale, b.v_scale)
    bs = b.block_size
    for new, pool, pre, scale in ((b.k_new, kc, b.k_cache_pre, b.k_scale),
                                  (b.v_new, vc, b.v_cache_pre, b.v_scale)):
        inv = torch.tensor(1.0 / scale, dtype=torch.float32)
        want = (new.float() * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        touched = np.zeros(pool.shape, dtype=bool)
        for t, slot in enumerate(b.slot_mapping.tolist()):
            if slot >= 0:
                assert np.array_equal(pool[slot // bs, :, slot % bs, :], want[t])
                touched[slot // bs, :, slot % bs, :] = True
        assert np.array_equal(pool[~touched], pre.numpy()[~touched])


@pytest.mark.parametrize("make", [lambda: small_decode(d=64, hq=8, hkv=2, seed=9105),
                                  lambda: small_mixed(d=64, bs=32, hq=8, hkv=4, seed=9232)])
def test_fp8_attention_matches_brute_force_on_dequantised_kv(make):
    """The FP8 attention equals a NumPy brute force over K = k_scale * value(code) and
    V = v_scale * value(code), the codes taken from the contiguous K/V by torch's conversion."""
    b = W.to_fp8(make(), k_scale=0.04, v_scale=0.03)
    o = oracle.attention_fp8(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                             b.query_start_loc, b.scale, b.k_scale, b.v_scale)

    def deq(x, scale):
        inv = torch.tensor(1.0 / scale, dtype=torch.float32)
        codes = (x.float() * inv).to(torch.float8_e4m3fn)
        return codes.to(torch.float64) * scale

    ref = brute_attention(b.q, deq(b.k_contig, b.k_scale), deq(b.v_contig, b.v_scale),
                          b.kv_start, b.seq_lens, b.query_start_loc, b.scale)
    assert np.allclose(o, ref, rtol=0, atol=1e-12, equal_nan=True)


# ---------------------------------------------------------------- bfloat16 KV cache

def test_bf16_to_double_all_patterns():
    """The oracle's bfloat16 decoder against torch's bfloat16 -> float64 conversion, every bit
    pattern, plus values the format fixes by hand."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    mine = oracle.bf16_to_double(bits.numpy().view(np.uint16))
    ref = bits.view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert oracle.bf16_to_double([0x3F80])[0] == 1.0
    assert oracle.bf16_to_double([0xC000])[0] == -2.0
    assert oracle.bf16_to_double([0x0001])[0] == 2.0 ** -133
    assert oracle.bf16_to_double([0x7F7F])[0] == (2 - 2.0 ** -7) * 2.0 ** 127


@pytest.mark.parametrize("make", [small_decode, small_mixed, small_spec,
                                  lambda: small_decode(d=64, bs=32, hq=32, hkv=2, seed=9106)])
def test_bf16_attention_matches_numpy_brute_force(make):
    b = W.to_bf16(make())
    assert b.q.dtype == b.k_cache.dtype == torch.bfloat16
    o = oracle.attention_batch(b)
    ref = brute_attention(b.q, b.k_contig, b.v_contig, b.kv_start, b.seq_lens,
                          b.query_start_loc, b.scale)
    assert np.allclose(o, ref, rtol=0, atol=1e-12, equal_nan=True)


def test_bf16_and_fp16_patterns_of_the_same_values_agree_bitwise():
    """Values exact in both formats (multiples of 1/64 in [-4, 4]) give bit-identical fp64
    attention whichever 16-bit format carries them: the format only changes the widening."""
    b = small_mixed(d=64, hq=8, hkv=2, seed=9233)
    snap = lambda t: (t.float() * 64).round().clamp(-256, 256).div(64).half()
    for f in ("q", "k_cache", "v_cache"):
        t = getattr(b, f)
        setattr(b, f, torch.where(torch.isnan(t), t, snap(t)))
    h = oracle.attention_batch(b)
    bb = W.to_bf16(b)
    assert torch.equal(bb.q.float(), b.q.float())                  # conversion was exact
    assert np.array_equal(oracle.attention_batch(bb), h, equal_nan=True)
    with pytest.raises(ValueError):
        oracle.attention(b.q, bb.k_cache, bb.v_cache, b.block_tables, b.seq_lens,
                         b.query_start_loc, b.scale)

