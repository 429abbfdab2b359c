"""Seeded synthetic batches for paged attention (inputs only).

This module draws the random tensors and chooses the physical block placement of a paged KV
cache; it computes no attention.  Both sides of every parity check consume what it returns:
the CUDA path through the C ABI and the fp64 CPU oracle.  Nothing here imports either side.

Shapes and conventions (the pages fix none of them; these are the readings used throughout):

* KV pool ``k_cache``/``v_cache``: fp16 ``[num_blocks, num_kv_heads, block_size, head_dim]``.
  One (block, kv-head) pair is a contiguous ``block_size x head_dim`` tile.  The pages describe
  the cache as fixed-size physical blocks reached through a per-sequence block table
  ("Local_LLM_03_vLLM_Architecture", paged-KV slide; "vLLM: LLM Inference That Doesn't Waste
  Your GPU", section "PagedAttention: virtual memory for KV").
* ``block_tables``: int32 ``[num_seqs, max_blocks]``; entry ``j`` of row ``s`` is the physical
  block holding logical positions ``j*block_size .. (j+1)*block_size-1`` of sequence ``s``.
  Entries past a sequence's last block hold the id of a NaN-filled spare block, so that a read
  past the end of a sequence shows up as NaN.
* ``seq_lens``: int32 ``[num_seqs]``; keys visible to a sequence after this step's tokens have
  been written to the cache, query tokens included.
* ``query_start_loc``: int32 ``[num_seqs + 1]``; sequence ``s`` owns query rows
  ``query_start_loc[s] .. query_start_loc[s+1]-1``.  One row is a decode step; more rows are a
  prefill chunk whose row ``i`` sits at absolute position ``seq_len - query_len + i``.
* ``q``: fp16 ``[num_tokens, num_q_heads, head_dim]``; ``k_new``/``v_new``: fp16
  ``[num_tokens(+pad), num_kv_heads, head_dim]``, the K/V of this step's tokens;
  ``slot_mapping``: int64, ``block * block_size + offset`` of each new token, ``-1`` = padding.
* Every pool element that no sequence maps (spare blocks, block tails past ``seq_len``) is the
  fp16 quiet NaN ``0x7E00``.

Seeds: workload ``c`` draws from ``torch.Generator`` streams seeded ``290_000 + 100*c + k`` with
``k`` = 0 lengths, 1 block permutation, 2 q, 3 k, 4 v, 5 order/prefix.  Values are N(0, 1)
drawn in fp32 and rounded to fp16 (round-to-nearest-even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

NAN_F16_BITS = 0x7E00


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _randn_f16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.float16)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass(frozen=True)
class SeqSpec:
    """One sequence of a step: ``seq_len`` keys in total, the last ``query_len`` are new."""

    seq_len: int
    query_len: int


@dataclass
class PagedBatch:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    seqs: List[SeqSpec]
    seq_lens: torch.Tensor          # int32 [N]
    query_start_loc: torch.Tensor   # int32 [N+1]
    block_tables: torch.Tensor      # int32 [N, MB]
    q: torch.Tensor                 # fp16 [T, Hq, d]
    k_new: torch.Tensor             # fp16 [T(+pad), Hkv, d]
    v_new: torch.Tensor             # fp16 [T(+pad), Hkv, d]
    slot_mapping: torch.Tensor      # int64 [T(+pad)]
    k_cache_pre: Optional[torch.Tensor]   # pool before this step's write (new slots NaN)
    v_cache_pre: Optional[torch.Tensor]
    k_cache: torch.Tensor           # pool with every position of every sequence in place
    v_cache: torch.Tensor
    nan_block: int                  # id of a spare block that is all NaN
    num_unique_blocks: int          # physical blocks referenced by at least one table
    k_contig: Optional[torch.Tensor] = None   # fp16 [sum L, Hkv, d], sequence after sequence
    v_contig: Optional[torch.Tensor] = None
    kv_start: Optional[torch.Tensor] = None   # int64 [N], row of k_contig where seq s starts
    meta: dict = field(default_factory=dict)
    # "f16"; "bf16": q, the new tokens and the pools are bfloat16; or "e4m3": the pools hold
    # E4M3 codes (uint8) standing for k_scale * value (v_scale)
    kv_dtype: str = "f16"
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_seqs(self) -> int:
        return len(self.seqs)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_seq_len(self) -> int:
        return max((s.seq_len for s in self.seqs), default=0)

    @property
    def max_query_len(self) -> int:
        return max((s.query_len for s in self.seqs), default=0)

    @property
    def num_prefill_seqs(self) -> int:
        return sum(1 for s in self.seqs if s.query_len > 1)


def build_batch(
    name: str,
    seqs: Sequence[SeqSpec],
    *,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int,
    seed_base: int,
    scale: Optional[float] = None,
    pool_blocks: Optional[int] = None,
    spare_frac: float = 0.10,
    min_spare: int = 1,
    shared_prefix_len: int = 0,
    keep_contiguous: bool = True,
    keep_pre: bool = True,
    num_pad_slots: int = 0,
    table_pad: int = 0,
) -> PagedBatch:
    """Draw one seeded batch and place its K/V in a randomly permuted block pool.

    ``shared_prefix_len`` (a multiple of ``block_size``) makes every sequence start with the
    same tokens, stored once and aliased in every block table, as prefix sharing does
    ("Scaling inference with vLLM": requests that start the same way share their pages).
    """
    seqs = list(seqs)
    n = len(seqs)
    bs = block_size
    for s in seqs:
        if not (0 <= s.query_len <= s.seq_len):
            raise ValueError(f"need 0 <= query_len <= seq_len, got {s}")
    if shared_prefix_len % bs:
        raise ValueError("shared prefix must cover whole blocks")
    p0 = shared_prefix_len // bs
    for s in seqs:
        if shared_prefix_len and s.seq_len - s.query_len < shared_prefix_len:
            raise ValueError("query tokens may not fall inside the shared prefix")

    nblk = [_cdiv(s.seq_len, bs) for s in seqs]
    priv = [b - p0 for b in nblk]
    used = p0 + sum(priv)
    if pool_blocks is None:
        pool_blocks = used + max(min_spare, math.ceil(spare_frac * used))
    if pool_blocks < used + 1:
        raise ValueError("pool needs at least one spare (NaN) block")

    perm = torch.randperm(pool_blocks, generator=_gen(seed_base + 1))
    prefix_ids = perm[:p0]
    cursor = p0
    max_blocks = max(nblk, default=0) + table_pad
    max_blocks = max(max_blocks, 1)
    nan_block = int(perm[used])
    tables = torch.full((n, max_blocks), nan_block, dtype=torch.int32)
    for i in range(n):
        tables[i, :p0] = prefix_ids.to(torch.int32)
        tables[i, p0:nblk[i]] = perm[cursor:cursor + priv[i]].to(torch.int32)
        cursor += priv[i]

    hkv, d = num_kv_heads, head_dim
    gk, gv = _gen(seed_base + 3), _gen(seed_base + 4)
    uniq_len = shared_prefix_len + sum(s.seq_len - shared_prefix_len for s in seqs)
    k_uniq = _randn_f16((uniq_len, hkv, d), gk)
    v_uniq = _randn_f16((uniq_len, hkv, d), gv)

    # token -> (row in the unique value arrays, physical block, offset) for every position
    src_rows, blk_ids, offs, is_new = [], [], [], []
    row = shared_prefix_len
    for i, s in enumerate(seqs):
        pos = torch.arange(s.seq_len, dtype=torch.int64)
        src = torch.where(pos < shared_prefix_len, pos,
                          row + pos - shared_prefix_len)
        row += s.seq_len - shared_prefix_len
        src_rows.append(src)
        blk_ids.append(tables[i].to(torch.int64)[pos // bs])
        offs.append(pos % bs)
        is_new.append(pos >= s.seq_len - s.query_len)
    src_rows = torch.cat(src_rows) if src_rows else torch.zeros(0, dtype=torch.int64)
    blk_ids = torch.cat(blk_ids) if blk_ids else torch.zeros(0, dtype=torch.int64)
    offs = torch.cat(offs) if offs else torch.zeros(0, dtype=torch.int64)
    is_new = torch.cat(is_new) if is_new else torch.zeros(0, dtype=torch.bool)

    def place(mask: Optional[torch.Tensor]):
        kc = torch.full((pool_blocks, hkv, bs, d), float("nan"), dtype=torch.float16)
        vc = torch.full((pool_blocks, hkv, bs, d), float("nan"), dtype=torch.float16)
        sr, bl, of = src_rows, blk_ids, offs
        if mask is not None:
            sr, bl, of = sr[mask], bl[mask], of[mask]
        kc[bl, :, of, :] = k_uniq[sr]
        vc[bl, :, of, :] = v_uniq[sr]
        return kc, vc

    k_cache, v_cache = place(None)
    k_pre = v_pre = None
    if keep_pre:
        k_pre, v_pre = place(~is_new)

    new_rows = src_rows[is_new]
    k_new = k_uniq[new_rows]
    v_new = v_uniq[new_rows]
    slot_mapping = blk_ids[is_new] * bs + offs[is_new]
    if num_pad_slots:
        gp = _gen(seed_base + 5)
        k_new = torch.cat([k_new, _randn_f16((num_pad_slots, hkv, d), gp)])
        v_new = torch.cat([v_new, _randn_f16((num_pad_slots, hkv, d), gp)])
        slot_mapping = torch.cat([slot_mapping,
                                  torch.full((num_pad_slots,), -1, dtype=torch.int64)])

    qlens = torch.tensor([s.query_len for s in seqs], dtype=torch.int64)
    qsl = torch.zeros(n + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(qlens, 0).to(torch.int32)
    t = int(qsl[-1])
    q = _randn_f16((t, num_q_heads, d), _gen(seed_base + 2))

    k_contig = v_contig = kv_start = None
    if keep_contiguous:
        k_contig = k_uniq[src_rows]
        v_contig = v_uniq[src_rows]
        lens = torch.tensor([s.seq_len for s in seqs], dtype=torch.int64)
        kv_start = torch.zeros(n, dtype=torch.int64)
        if n > 1:
            kv_start[1:] = torch.cumsum(lens, 0)[:-1]

    return PagedBatch(
        name=name, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=bs, scale=float(1.0 / math.sqrt(head_dim) if scale is None else scale),
        seqs=seqs,
        seq_lens=torch.tensor([s.seq_len for s in seqs], dtype=torch.int32),
        query_start_loc=qsl, block_tables=tables, q=q, k_new=k_new, v_new=v_new,
        slot_mapping=slot_mapping, k_cache_pre=k_pre, v_cache_pre=v_pre,
        k_cache=k_cache, v_cache=v_cache, nan_block=nan_block,
        num_unique_blocks=used, k_contig=k_contig, v_contig=v_contig, kv_start=kv_start,
        meta={"seed_base": seed_base, "shared_prefix_len": shared_prefix_len},
    )


def unalias_prefix(b: PagedBatch) -> PagedBatch:
    """Give every sequence private copies of the aliased prefix blocks (same values).

    The result is the "no sharing" placement of the same logical K/V, used to check that
    aliased prefix blocks and private copies give identical attention.
    """
    p0 = b.meta["shared_prefix_len"] // b.block_size
    if p0 == 0:
        return b
    n = b.num_seqs
    nb = b.num_blocks
    shared = b.block_tables[0, :p0].to(torch.int64)
    extra = n * p0
    k = torch.cat([b.k_cache, b.k_cache[shared].repeat(n, 1, 1, 1)])
    v = torch.cat([b.v_cache, b.v_cache[shared].repeat(n, 1, 1, 1)])
    tables = b.block_tables.clone()
    tables[:, :p0] = (nb + torch.arange(extra, dtype=torch.int32)).view(n, p0)
    out = PagedBatch(**{**b.__dict__})
    out.name = b.name + "_unaliased"
    out.k_cache, out.v_cache, out.block_tables = k, v, tables
    out.k_cache_pre = out.v_cache_pre = None
    out.num_unique_blocks = b.num_unique_blocks + extra - p0
    out.meta = {**b.meta, "shared_prefix_len": 0}
    return out


def repermute(b: PagedBatch, seed: int) -> PagedBatch:
    """Move every physical block to a new seeded random slot (same logical K/V).

    Block ids in the tables, the slot mapping and the pool are relabelled together.
    """
    nb = b.num_blocks
    new_of_old = torch.randperm(nb, generator=_gen(seed))
    k = torch.empty_like(b.k_cache)
    v = torch.empty_like(b.v_cache)
    k[new_of_old] = b.k_cache
    v[new_of_old] = b.v_cache
    out = PagedBatch(**{**b.__dict__})
    out.name = b.name + f"_perm{seed}"
    out.k_cache, out.v_cache = k, v
    if b.k_cache_pre is not None:
        kp = torch.empty_like(b.k_cache_pre)
        vp = torch.empty_like(b.v_cache_pre)
        kp[new_of_old] = b.k_cache_pre
        vp[new_of_old] = b.v_cache_pre
        out.k_cache_pre, out.v_cache_pre = kp, vp
    out.block_tables = new_of_old[b.block_tables.to(torch.int64)].to(torch.int32)
    sm = b.slot_mapping
    valid = sm >= 0
    new_sm = sm.clone()
    new_sm[valid] = new_of_old[sm[valid] // b.block_size] * b.block_size + sm[valid] % b.block_size
    out.slot_mapping = new_sm
    out.nan_block = int(new_of_old[b.nan_block])
    return out


def to_fp8(b: PagedBatch, k_scale: float = 1.0 / 32, v_scale: float = 1.0 / 32) -> PagedBatch:
    """The same batch over an FP8 (E4M3) cache with per-tensor scales: every pool value x becomes
    the E4M3 code of x * (1 / scale) (float32), by torch's float8_e4m3fn conversion (round to
    nearest even; the scales keep N(0,1) data far inside +-448).  NaN sentinels stay NaN (0x7F).
    The new tokens stay fp16: the scatter-write quantises them."""
    def q8(pool, scale):
        if pool is None:
            return None
        inv = torch.tensor(1.0 / scale, dtype=torch.float32)
        return (pool.float() * inv).to(torch.float8_e4m3fn).view(torch.uint8)
    out = PagedBatch(**{**b.__dict__})
    out.name = b.name + "_fp8"
    out.k_cache, out.v_cache = q8(b.k_cache, k_scale), q8(b.v_cache, v_scale)
    out.k_cache_pre, out.v_cache_pre = q8(b.k_cache_pre, k_scale), q8(b.v_cache_pre, v_scale)
    out.kv_dtype, out.k_scale, out.v_scale = "e4m3", float(k_scale), float(v_scale)
    return out


def to_bf16(b: PagedBatch) -> PagedBatch:
    """The same batch in bfloat16: q, the new tokens, the pools and the contiguous copies are
    rounded from fp16 to bfloat16 (torch's conversion, round to nearest even).  Rounding the
    pool and the new tokens the same way keeps the pool's new slots equal to what the
    scatter-write stores; NaN sentinels stay NaN."""
    def bf(t):
        return None if t is None else t.to(torch.bfloat16)
    out = PagedBatch(**{**b.__dict__})
    out.name = b.name + "_bf16"
    for f in ("q", "k_new", "v_new", "k_cache_pre", "v_cache_pre", "k_cache", "v_cache",
              "k_contig", "v_contig"):
        setattr(out, f, bf(getattr(b, f)))
    out.kv_dtype = "bf16"
    return out


# ---------------------------------------------------------------------------------------------
# The five workloads.  Model names only fix head counts and head_dim.


def _seed(c: int) -> int:
    return 290_000 + 100 * c


def tiny_decode(**kw) -> PagedBatch:
    """4 decode sequences, lengths uniform in [1, 64], 4 q / 2 kv heads, d 64, bs 16, pool 64."""
    s = _seed(1)
    lens = torch.randint(1, 65, (4,), generator=_gen(s + 0)).tolist()
    return build_batch("tiny_decode", [SeqSpec(L, 1) for L in lens], num_q_heads=4,
                       num_kv_heads=2, head_dim=64, block_size=16, seed_base=s,
                       scale=1.0 / 8.0, pool_blocks=64, **kw)


def llama8b_decode(**kw) -> PagedBatch:
    """64 decode sequences, lengths uniform in [512, 4096], 32 q / 8 kv heads, d 128, bs 16."""
    s = _seed(2)
    lens = torch.randint(512, 4097, (64,), generator=_gen(s + 0)).tolist()
    return build_batch("llama8b_decode", [SeqSpec(L, 1) for L in lens], num_q_heads=32,
                       num_kv_heads=8, head_dim=128, block_size=16, seed_base=s,
                       spare_frac=0.10, **kw)


def llama70b_decode(num_seqs: int = 32, **kw) -> PagedBatch:
    """32 decode sequences of 8192 keys, 64 q / 8 kv heads, d 128, bs 16, 64 spare blocks.
    ``num_seqs`` shrinks the batch (same shapes) for profiler captures."""
    s = _seed(3)
    n, L, bs = num_seqs, 8192, 16
    return build_batch(f"llama70b_{n}x8k_decode", [SeqSpec(L, 1)] * n, num_q_heads=64,
                       num_kv_heads=8, head_dim=128, block_size=bs, seed_base=s,
                       pool_blocks=n * L // bs + 64, **kw)


def prefix_shared_decode(**kw) -> PagedBatch:
    """160 decode sequences sharing a 2048-token prefix (128 aliased blocks) plus a private
    continuation uniform in [16, 1024]; 28 q / 4 kv heads, d 128, bs 16."""
    s = _seed(4)
    priv = torch.randint(16, 1025, (160,), generator=_gen(s + 0)).tolist()
    return build_batch("prefix_shared_decode", [SeqSpec(2048 + p, 1) for p in priv],
                       num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                       seed_base=s, shared_prefix_len=2048, spare_frac=0.10, **kw)


def mixed_step(block_size: int = 16, num_decode: int = 128, **kw) -> PagedBatch:
    """4 prefill chunks of 512 queries over a paged context uniform in [0, 7488] plus 128 decode
    sequences with lengths uniform in [256, 8000], in one seeded order; 32 q / 8 kv, d 128.
    ``num_decode`` keeps only the first decode sequences (for profiler captures)."""
    s = _seed(5)
    g = _gen(s + 0)
    ctx = torch.randint(0, 7489, (4,), generator=g).tolist()
    dec = torch.randint(256, 8001, (128,), generator=g).tolist()[:num_decode]
    seqs = [SeqSpec(c + 512, 512) for c in ctx] + [SeqSpec(L, 1) for L in dec]
    order = torch.randperm(len(seqs), generator=_gen(s + 5)).tolist()
    seqs = [seqs[i] for i in order]
    name = f"mixed_step_bs{block_size}" + ("" if num_decode == 128 else f"_{num_decode}dec")
    return build_batch(name, seqs, num_q_heads=32, num_kv_heads=8,
                       head_dim=128, block_size=block_size, seed_base=s, spare_frac=0.10, **kw)


def spec_verify(**kw) -> PagedBatch:
    """64 sequences each verifying k speculative draft tokens in one pass (k uniform in [1, 5],
    so q_len = k + 1 in [2, 6] rows, causal among themselves), after a context uniform in
    [512, 4096]; 32 q / 8 kv heads, d 128, bs 16.  ("Local_LLM_03_vLLM_Architecture",
    speculative-decoding slide: the target model checks all drafted tokens in one forward pass,
    and acceptance runs from 2 to 4 of 5 drafts.)"""
    s = _seed(6)
    ctx = torch.randint(512, 4097, (64,), generator=_gen(s + 0)).tolist()
    k = torch.randint(1, 6, (64,), generator=_gen(s + 6)).tolist()
    seqs = [SeqSpec(c + kk + 1, kk + 1) for c, kk in zip(ctx, k)]
    return build_batch("spec_verify", seqs, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       block_size=16, seed_base=s, spare_frac=0.10, **kw)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "llama8b_decode": llama8b_decode,
    "llama70b_32x8k_decode": llama70b_decode,
    "llama70b_8x8k_decode": lambda **kw: llama70b_decode(8, **kw),
    "prefix_shared_decode": prefix_shared_decode,
    "mixed_step_bs16": lambda **kw: mixed_step(16, **kw),
    "mixed_step_bs32": lambda **kw: mixed_step(32, **kw),
    "mixed_step_bs16_8dec": lambda **kw: mixed_step(16, num_decode=8, **kw),
    "mixed_step_bs16_0dec": lambda **kw: mixed_step(16, num_decode=0, **kw),
    "spec_verify": spec_verify,
    "llama70b_32x8k_decode_fp8": lambda **kw: to_fp8(llama70b_decode(**kw)),
    "llama70b_32x8k_decode_bf16": lambda **kw: to_bf16(llama70b_decode(**kw)),
    "mixed_step_bs16_bf16": lambda **kw: to_bf16(mixed_step(16, **kw)),
    "llama70b_8x8k_decode_fp8": lambda **kw: to_fp8(llama70b_decode(8, **kw)),
    "llama70b_8x8k_decode_bf16": lambda **kw: to_bf16(llama70b_decode(8, **kw)),
    "spec_verify_fp8": lambda **kw: to_fp8(spec_verify(**kw)),
    "mixed_step_bs16_fp8": lambda **kw: to_fp8(mixed_step(16, **kw)),
    "prefix_shared_decode_fp8": lambda **kw: to_fp8(prefix_shared_decode(**kw)),
    "mixed_step_bs16_0dec_fp8": lambda **kw: to_fp8(mixed_step(16, num_decode=0, **kw)),
}
