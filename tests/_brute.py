"""Independent NumPy fp64 brute-force attention over contiguous K/V (a pin for the oracle).

Written separately from the oracle: it never sees the paged pool, it works from the
per-sequence contiguous K/V the input generator kept before placing blocks, and it uses
NumPy's vectorised float64 arithmetic rather than the oracle's scalar loops.
"""
import numpy as np


def _f64(t):
    return t.detach().cpu().double().numpy()  # exact for fp16, bfloat16 and float64


def brute_attention(q, k_contig, v_contig, kv_start, seq_lens, query_start_loc, scale):
    q, k, v = _f64(q), _f64(k_contig), _f64(v_contig)
    kv_start = kv_start.numpy()
    lens = seq_lens.numpy()
    qsl = query_start_loc.numpy()
    t, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    out = np.full((t, hq, d), np.nan)
    for s in range(len(lens)):
        q_len = int(qsl[s + 1] - qsl[s])
        L = int(lens[s])
        base = int(kv_start[s])
        for i in range(q_len):
            row = int(qsl[s]) + i
            visible = L - q_len + i + 1          # bottom-right causal
            for h in range(hq):
                kk = k[base:base + visible, h // group, :]
                vv = v[base:base + visible, h // group, :]
                logits = scale * (kk @ q[row, h])
                w = np.exp(logits - logits.max())
                out[row, h] = (w[:, None] * vv).sum(0) / w.sum()
    return out
