"""Small seeded batches shared by the oracle pins and the GPU parity tests.

They are scaled-down versions of the five workloads: the oracle finishes each in well under a
second, yet they span several key blocks, several 512-token partitions, ragged prefill chunks
(query lengths that are not multiples of any tile), block tails, GQA groups of 1, 2, 4, 7 and 8
and both block sizes.
"""
import torch

from paged_kv_cache_290_gb300.workloads import SeqSpec, build_batch


def small_decode(d=128, bs=16, hq=32, hkv=8, seed=9100, lens=(1, 15, 16, 17, 300, 511, 512, 513,
                                                                 1029, 1600)):
    return build_batch(f"small_decode_d{d}_bs{bs}_g{hq // hkv}", [SeqSpec(L, 1) for L in lens],
                       num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                       seed_base=seed)


def small_mixed(d=128, bs=16, hq=32, hkv=8, seed=9200):
    seqs = [
        SeqSpec(70, 40),      # chunk over a 30-token context, ragged
        SeqSpec(1, 1),        # first token of a sequence
        SeqSpec(533, 1),      # decode over two partitions
        SeqSpec(150, 17),     # short ragged chunk
        SeqSpec(64, 64),      # whole prompt, no context (plain causal)
        SeqSpec(5, 0),        # idle sequence in the batch: no rows
        SeqSpec(700, 129),    # chunk whose keys cross a partition boundary
        SeqSpec(48, 1),
    ]
    return build_batch(f"small_mixed_d{d}_bs{bs}_g{hq // hkv}", seqs, num_q_heads=hq,
                       num_kv_heads=hkv, head_dim=d, block_size=bs, seed_base=seed,
                       num_pad_slots=3)


def small_prefix(seed=9300, n=6, prefix=64, d=128, bs=16):
    lens = [prefix + 1 + 37 * i for i in range(n)]
    return build_batch("small_prefix", [SeqSpec(L, 1) for L in lens], num_q_heads=28,
                       num_kv_heads=4, head_dim=d, block_size=bs, seed_base=seed,
                       shared_prefix_len=prefix)


def small_shared(seed=9600, n=24, prefix=1024, d=128, bs=16, hq=28, hkv=4):
    """n decode rows behind a shared prefix of `prefix` keys (two 512-key partitions, attended
    once by the shared-prefix pass), private continuations of 1 to 700 keys."""
    g = torch.Generator().manual_seed(seed)
    priv = torch.randint(1, 701, (n,), generator=g).tolist()
    return build_batch(f"small_shared_{n}x{prefix}", [SeqSpec(prefix + p, 1) for p in priv],
                       num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                       seed_base=seed, shared_prefix_len=prefix)


def small_spec(d=128, bs=16, hq=32, hkv=4, seed=9400):
    """Speculative-verify rows: q_len = k + 1 in [2, 6] over short ragged contexts (one with a
    context shorter than its drafts, one crossing a 512-key boundary)."""
    seqs = [SeqSpec(2, 2), SeqSpec(37, 3), SeqSpec(515, 6), SeqSpec(130, 4), SeqSpec(17, 5),
            SeqSpec(96, 2), SeqSpec(1, 1), SeqSpec(260, 6)]
    return build_batch(f"small_spec_d{d}_bs{bs}_g{hq // hkv}", seqs, num_q_heads=hq,
                       num_kv_heads=hkv, head_dim=d, block_size=bs, seed_base=seed)


def small_long_chunks(d=128, bs=16, hq=8, hkv=2, seed=9500, decode=True):
    """Chunks over contexts past 4096 and 8192 keys, a short chunk, and (``decode``) decode rows
    in the same batch: with decode rows the two-tile prefill kernel runs beside the decode
    kernel in launch slices; without, alone on the caller's stream."""
    seqs = [SeqSpec(4096 + 40, 100), SeqSpec(8192 + 20, 150), SeqSpec(5000, 64),
            SeqSpec(300, 33)] + ([SeqSpec(9000, 1), SeqSpec(6000, 1)] if decode else [])
    return build_batch(f"long_chunks_d{d}_bs{bs}_g{hq // hkv}", seqs, num_q_heads=hq,
                       num_kv_heads=hkv, head_dim=d, block_size=bs, seed_base=seed)

