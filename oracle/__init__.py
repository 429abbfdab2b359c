"""fp64 CPU oracle for paged attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library and its Python binding never do, and the two share no
code.  The arithmetic lives in ``pa_oracle.c`` (plain C, fp64, OpenMP); this module compiles it
with gcc and marshals arrays through ctypes.

Every oracle function is pinned by CPU tests against something other than itself: the pages'
worked arithmetic, closed forms, invariants of paging (placement, aliasing, contiguous vs
paged), a float64 library attention and an independent NumPy brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "_pa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp); returns the shared-object path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32p, u16p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            p = ctypes.c_void_p
            lib.pa_oracle_half_to_double.restype = ctypes.c_double
            lib.pa_oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.pa_oracle_bf16_to_double.restype = ctypes.c_double
            lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.pa_oracle_set_threads.argtypes = [ctypes.c_int]
            lib.pa_oracle_get_threads.restype = ctypes.c_int
            lib.pa_oracle_reshape_and_cache.restype = ctypes.c_int
            lib.pa_oracle_reshape_and_cache.argtypes = [u16p, u16p, u16p, u16p, p, i64, i64,
                                                        i64, i64, i64]
            common = [u16p, u16p, u16p, i32p, i64, i32p, i32p, i64, i64, i64, i64, i64, i64,
                      ctypes.c_double, i64]
            lib.pa_oracle_attention.restype = ctypes.c_int
            lib.pa_oracle_attention.argtypes = common + [p, p]
            lib.pa_oracle_attention_split.restype = ctypes.c_int
            lib.pa_oracle_attention_split.argtypes = common + [i64, p, p]
            lib.pa_oracle_attention_contiguous.restype = ctypes.c_int
            lib.pa_oracle_attention_contiguous.argtypes = [u16p, u16p, u16p, p, i32p, i32p,
                                                           i64, i64, i64, i64,
                                                           ctypes.c_double, i64, p, p]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _np(x, dtype):
    """CPU numpy view (C-contiguous) of a torch tensor or array, reinterpreted as ``dtype``."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype in (torch.float16, torch.bfloat16):
                x = x.view(torch.int16)
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize == np.dtype(dtype).itemsize and x.dtype != dtype:
        x = x.view(dtype)
    elif x.dtype != dtype:
        x = x.astype(dtype)
    return x


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().pa_oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().pa_oracle_get_threads())


def half_to_double(bits) -> np.ndarray:
    """Widen raw binary16 bit patterns to float64 through the oracle's own decoder."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.pa_oracle_half_to_double(int(x)) for x in b], dtype=np.float64)


def bf16_to_double(bits) -> np.ndarray:
    """Widen raw bfloat16 bit patterns to float64 through the oracle's own decoder."""
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.pa_oracle_bf16_to_double(int(x)) for x in b], dtype=np.float64)


FMT_F16, FMT_BF16 = 0, 1


def _fmt(*tensors) -> int:
    """The 16-bit format of q and the pools: bfloat16 when they are torch bfloat16 tensors,
    else binary16 (torch float16, or raw uint16 patterns, which are read as binary16)."""
    try:
        import torch
        kinds = {isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16 for t in tensors}
    except ImportError:  # pragma: no cover
        kinds = {False}
    if len(kinds) != 1:
        raise ValueError("q and the pools must all be bfloat16 or all be binary16")
    return FMT_BF16 if kinds.pop() else FMT_F16


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping):
    """Return (k_cache', v_cache') as uint16 arrays: copies of the pools with each new token's
    K/V rows written at block slot//bs, offset slot%bs; negative slots are skipped."""
    lib = _load()
    k16, v16 = _np(k, np.uint16), _np(v, np.uint16)
    kc = _np(k_cache, np.uint16).copy()
    vc = _np(v_cache, np.uint16).copy()
    sm = _np(slot_mapping, np.int64)
    t, hkv, d = k16.shape
    nb, hkv2, bs, d2 = kc.shape
    if hkv2 != hkv or d2 != d or sm.shape[0] != t or v16.shape != k16.shape:
        raise ValueError("shape mismatch")
    rc = lib.pa_oracle_reshape_and_cache(_ptr(k16), _ptr(v16), _ptr(kc), _ptr(vc), _ptr(sm),
                                         t, hkv, d, nb, bs)
    if rc:
        raise OracleError(f"reshape_and_cache: code {rc}")
    return kc, vc


def copy_blocks(k_cache, v_cache, pairs):
    """Return (k_cache', v_cache') as uint16 arrays: copies of the pools in which block
    pairs[i][1] holds what block pairs[i][0] held before (all kv heads, K and V); pairs with an
    id outside the pool are skipped.  Plain NumPy indexing."""
    kc0, vc0 = _np(k_cache, np.uint16), _np(v_cache, np.uint16)
    kc, vc = kc0.copy(), vc0.copy()
    nb = kc.shape[0]
    for src, dst in _np(pairs, np.int32).reshape(-1, 2).tolist():
        if 0 <= src < nb and 0 <= dst < nb:
            kc[dst] = kc0[src]
            vc[dst] = vc0[src]
    return kc, vc


# ------------------------------------------------------------------ FP8 (E4M3) KV cache
# E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities; S.1111.111 is NaN,
# so the largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the subnormals
# m * 2^-9.  A stored code c of a cache with scale s stands for s * value(c).


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (NaN for 0x7F / 0xFF), from the format's definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


_E4M3_POS = None


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code of each float: the nearest finite code (ties to the even code), magnitudes at or
    beyond 448 (and infinities) saturate to +-448, NaN -> 0x7F; the sign is kept, zero
    included.  Found by search over the table of the 127 non-negative finite codes."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_decode(np.arange(0x7F))  # codes 0x00 .. 0x7E, strictly increasing
    xv = np.asarray(x, dtype=np.float64)
    mag = np.abs(xv)
    tab = _E4M3_POS
    hi = np.clip(np.searchsorted(tab, mag, side="left"), 0, len(tab) - 1)
    lo = np.clip(hi - 1, 0, len(tab) - 1)
    d_lo, d_hi = np.abs(mag - tab[lo]), np.abs(tab[hi] - mag)
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(mag >= tab[-1], 0x7E, code)
    code = code | np.where(np.signbit(xv), 0x80, 0)
    code = np.where(np.isnan(xv), 0x7F, code)
    return code.astype(np.uint8)


def reshape_and_cache_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float):
    """FP8 scatter-write: (k_cache', v_cache') as uint8 arrays, copies of the pools with each new
    token's rows stored as e4m3_encode(x * (1/scale)), the product taken in float32 (1/scale
    too), slots < 0 skipped."""
    kc = _np(k_cache, np.uint8).copy()
    vc = _np(v_cache, np.uint8).copy()
    sm = _np(slot_mapping, np.int64)
    nb, hkv, bs, d = kc.shape
    for x, pool, scale in ((k, kc, k_scale), (v, vc, v_scale)):
        inv = np.float32(1.0) / np.float32(scale)
        vals = half_bits_to_float32(_np(x, np.uint16)) * inv   # float32 * float32
        codes = e4m3_encode(vals)
        for t, slot in enumerate(sm.tolist()):
            if 0 <= slot < nb * bs:
                pool[slot // bs, :, slot % bs, :] = codes[t]
    return kc, vc


_HALF_LUT = None


def half_bits_to_float32(bits) -> np.ndarray:
    """binary16 bit patterns -> float32 (exact) through the oracle's own decoder."""
    global _HALF_LUT
    if _HALF_LUT is None:
        _HALF_LUT = half_to_double(np.arange(1 << 16, dtype=np.uint16)).astype(np.float32)
    return _HALF_LUT[np.asarray(bits, dtype=np.uint16)]


def attention_fp8(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
                  k_scale: float, v_scale: float, row_mask=None) -> np.ndarray:
    """fp64 attention over an E4M3 cache: K = k_scale * value(code), V = v_scale * value(code).
    Every E4M3 value is exact in binary16, so this is the fp16-pool attention of the decoded
    codes with the score scale multiplied by k_scale (exact in fp64) and the output by
    v_scale."""
    kc, vc = _np(k_cache, np.uint8), _np(v_cache, np.uint8)
    to16 = e4m3_decode(np.arange(256)).astype(np.float16).view(np.uint16)  # exact, per code
    k16, v16 = to16[kc], to16[vc]
    out = attention(q, k16, v16, block_tables, seq_lens, query_start_loc,
                    float(scale) * float(k_scale), row_mask=row_mask)
    return out * float(v_scale)


def _attn_args(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc):
    q16 = _np(q, np.uint16)
    kc, vc = _np(k_cache, np.uint16), _np(v_cache, np.uint16)
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    t, hq, d = q16.shape
    nb, hkv, bs, d2 = kc.shape
    if d2 != d or vc.shape != kc.shape or qsl.shape[0] != sl.shape[0] + 1:
        raise ValueError("shape mismatch")
    if bt.ndim != 2 or bt.shape[0] != sl.shape[0]:
        raise ValueError("block table shape")
    return q16, kc, vc, bt, sl, qsl, (t, hq, hkv, d, bs, nb)


def _mask(row_mask, t):
    if row_mask is None:
        return None
    m = np.ascontiguousarray(np.asarray(row_mask, dtype=np.uint8))
    if m.shape != (t,):
        raise ValueError("row_mask must be [T]")
    return m


def attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale,
              row_mask=None, partition_size: int = 0, fmt=None) -> np.ndarray:
    """fp64 attention over the paged cache, [T, Hq, d].  ``partition_size > 0`` computes it
    split-context with a log-sum-exp merge instead.  Rows outside ``row_mask`` are NaN.
    q and the pools are binary16 or bfloat16 (``fmt`` None: from the torch dtypes)."""
    lib = _load()
    fmt = _fmt(q, k_cache, v_cache) if fmt is None else int(fmt)
    q16, kc, vc, bt, sl, qsl, (t, hq, hkv, d, bs, nb) = _attn_args(
        q, k_cache, v_cache, block_tables, seq_lens, query_start_loc)
    out = np.full((t, hq, d), np.nan, dtype=np.float64)
    m = _mask(row_mask, t)
    mp = _ptr(m) if m is not None else None
    args = [_ptr(q16), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(sl), _ptr(qsl),
            sl.shape[0], hq, hkv, d, bs, nb, float(scale), fmt]
    if partition_size > 0:
        rc = lib.pa_oracle_attention_split(*args, int(partition_size), mp, _ptr(out))
    else:
        rc = lib.pa_oracle_attention(*args, mp, _ptr(out))
    if rc:
        raise OracleError(f"attention: code {rc}")
    return out


def attention_contiguous(q, k, v, kv_start, seq_lens, query_start_loc, scale,
                         row_mask=None, fmt=None) -> np.ndarray:
    """fp64 attention over contiguous per-sequence K/V ``[sum L, Hkv, d]``."""
    lib = _load()
    fmt = _fmt(q, k, v) if fmt is None else int(fmt)
    q16 = _np(q, np.uint16)
    k16, v16 = _np(k, np.uint16), _np(v, np.uint16)
    ks = _np(kv_start, np.int64)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    t, hq, d = q16.shape
    hkv = k16.shape[1]
    out = np.full((t, hq, d), np.nan, dtype=np.float64)
    m = _mask(row_mask, t)
    rc = lib.pa_oracle_attention_contiguous(_ptr(q16), _ptr(k16), _ptr(v16), _ptr(ks), _ptr(sl),
                                            _ptr(qsl), sl.shape[0], hq, hkv, d, float(scale), fmt,
                                            _ptr(m) if m is not None else None, _ptr(out))
    if rc:
        raise OracleError(f"attention_contiguous: code {rc}")
    return out


def attention_batch(b, row_mask=None, partition_size: int = 0):
    """Convenience: oracle attention of a ``workloads.PagedBatch`` (full pool)."""
    return attention(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.query_start_loc,
                     b.scale, row_mask=row_mask, partition_size=partition_size)
