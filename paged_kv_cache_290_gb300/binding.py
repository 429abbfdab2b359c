"""Thin ctypes binding over the C ABI in ``include/pa.h`` and ``include/pa_block_manager.h``
(argument marshalling only).

Every computation runs in the sm_103a kernels of ``libpa_gb300.so``; this module turns torch
tensors into ``pa_tensor`` descriptors, passes the current CUDA stream and raises on a non-OK
status.  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_gb300.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_TIMEOUT = 4
PA_ERR_OUT_OF_RANGE = 5
PA_ERR_WORKSPACE = 6
PA_ERR_DESCRIPTOR = 7
PA_ERR_NO_BLOCKS = 8
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
                4: "PA_ERR_TIMEOUT", 5: "PA_ERR_OUT_OF_RANGE", 6: "PA_ERR_WORKSPACE",
                7: "PA_ERR_DESCRIPTOR", 8: "PA_ERR_NO_BLOCKS"}
PA_F16, PA_I32, PA_I64, PA_F8E4M3, PA_BF16 = 0, 1, 2, 3, 4
PA_WAIT_LIMIT_DEFAULT_NS = 2_000_000_000
PARTITION_TOKENS = 512
EXPORTED = ("pa_reshape_and_cache", "pa_attention_workspace_size", "pa_attention",
            "pa_last_error", "pa_get_device_error", "pa_set_timing_events", "pa_version",
            "pa_attention_static_scratch", "pa_copy_blocks", "pa_reshape_and_cache_fp8",
            "pa_attention_fp8",
            "pa_bm_create", "pa_bm_destroy", "pa_bm_add_sequence", "pa_bm_append",
            "pa_bm_truncate", "pa_bm_fork", "pa_bm_free", "pa_bm_stats", "pa_bm_sequence",
            "pa_bm_step_descriptor", "pa_step_slot_mapping", "pa_set_wait_limit",
            "pa_selftest_wait_timeout", "pa_set_stream_error_word")

# Byte tensors are E4M3 codes (the only one-byte type of the ABI).
_DTYPES = {torch.float16: PA_F16, torch.int32: PA_I32, torch.int64: PA_I64,
           torch.uint8: PA_F8E4M3, torch.float8_e4m3fn: PA_F8E4M3, torch.bfloat16: PA_BF16}


class PATensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class PABatchHint(ctypes.Structure):
    _fields_ = [("max_query_len", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("num_prefill_seqs", ctypes.c_int32), ("shared_prefix_tokens", ctypes.c_int32)]


class PAKVScales(ctypes.Structure):
    _fields_ = [("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class PAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_290_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(PATensor)
        lib.pa_reshape_and_cache.restype = ctypes.c_int
        lib.pa_reshape_and_cache.argtypes = [P, P, P, P, P, ctypes.c_void_p]
        lib.pa_attention_workspace_size.restype = ctypes.c_size_t
        lib.pa_attention_workspace_size.argtypes = [ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_int64, ctypes.c_int32]
        lib.pa_attention.restype = ctypes.c_int
        lib.pa_attention.argtypes = [P, P, P, P, P, P, ctypes.c_float, P,
                                     ctypes.POINTER(PABatchHint), ctypes.c_void_p, ctypes.c_size_t,
                                     ctypes.c_void_p]
        lib.pa_last_error.restype = ctypes.c_char_p
        lib.pa_get_device_error.restype = ctypes.c_int
        lib.pa_get_device_error.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
        lib.pa_version.restype = ctypes.c_int
        lib.pa_attention_static_scratch.restype = ctypes.c_int
        lib.pa_attention_static_scratch.argtypes = [P, P, P, P, P, P, ctypes.c_float, P,
                                                    ctypes.POINTER(PABatchHint), ctypes.c_void_p]
        lib.pa_set_wait_limit.restype = ctypes.c_int
        lib.pa_set_wait_limit.argtypes = [ctypes.c_uint64]
        lib.pa_set_stream_error_word.restype = ctypes.c_int
        lib.pa_set_stream_error_word.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.pa_selftest_wait_timeout.restype = ctypes.c_int
        lib.pa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
        lib.pa_set_timing_events.restype = ctypes.c_int
        lib.pa_set_timing_events.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.pa_copy_blocks.restype = ctypes.c_int
        lib.pa_copy_blocks.argtypes = [P, P, P, ctypes.c_void_p]
        S = ctypes.POINTER(PAKVScales)
        lib.pa_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.pa_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, S, ctypes.c_void_p]
        lib.pa_attention_fp8.restype = ctypes.c_int
        lib.pa_attention_fp8.argtypes = [P, P, P, P, P, P, ctypes.c_float, P,
                                         ctypes.POINTER(PABatchHint), S, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]
        I32, I64, VP = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        PI32, PI64 = ctypes.POINTER(I32), ctypes.POINTER(I64)
        for name, res, args in (
                ("pa_bm_create", VP, [I32, I32, I32]),
                ("pa_bm_destroy", None, [VP]),
                ("pa_bm_add_sequence", ctypes.c_int, [VP, I64, PI32, I32, I64, PI32]),
                ("pa_bm_append", ctypes.c_int, [VP, I64, PI32, I32, PI32, PI32]),
                ("pa_bm_truncate", ctypes.c_int, [VP, I64, I32]),
                ("pa_bm_fork", ctypes.c_int, [VP, I64, I64]),
                ("pa_bm_free", ctypes.c_int, [VP, I64]),
                ("pa_bm_stats", ctypes.c_int, [VP, PI32, PI32, PI32, PI32]),
                ("pa_bm_sequence", ctypes.c_int, [VP, I64, PI32, PI32, I32, PI32]),
                ("pa_bm_step_descriptor", ctypes.c_int,
                 [VP, PI64, PI32, I32, I32, I32, PI32, PI32, PI32, PI64]),
                ("pa_step_slot_mapping", ctypes.c_int,
                 [I32, PI32, PI32, PI32, I64, I32, I32, PI32, PI64, I64])):
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def describe(t: torch.Tensor) -> PATensor:
    """pa_tensor view of a torch tensor (no copy; strides in elements)."""
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() > 5:
        raise ValueError("rank above 5")
    d = PATensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status: int) -> None:
    if status != PA_OK:
        msg = load_library().pa_last_error()
        raise PAError(status, msg.decode() if msg else "")


def last_error() -> str:
    return load_library().pa_last_error().decode()


def version() -> int:
    return load_library().pa_version()


def _is_fp8(pool) -> bool:
    return pool.dtype in (torch.uint8, torch.float8_e4m3fn)


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None, k_scale=None,
                      v_scale=None) -> None:
    """``pa_reshape_and_cache``: write new K/V tokens [T, Hkv, d] into pool slots (in place).
    A byte pool is an FP8 (E4M3) cache: ``pa_reshape_and_cache_fp8`` with the two scales."""
    lib = load_library()
    args = [ctypes.byref(describe(x)) for x in (k, v, k_cache, v_cache, slot_mapping)]
    if _is_fp8(k_cache):
        sc = PAKVScales(float(k_scale), float(v_scale))
        _check(lib.pa_reshape_and_cache_fp8(*args, ctypes.byref(sc), _stream_handle(stream)))
    else:
        _check(lib.pa_reshape_and_cache(*args, _stream_handle(stream)))


def workspace_size(num_tokens: int, num_q_heads: int, head_dim: int, max_seq_len: int) -> int:
    return int(load_library().pa_attention_workspace_size(num_tokens, num_q_heads, head_dim,
                                                          max_seq_len))


def attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale: float, out,
              max_query_len: int, max_seq_len: int, workspace: Optional[torch.Tensor] = None,
              stream=None, num_prefill_seqs: int = 0, k_scale=None, v_scale=None,
              shared_prefix_tokens: int = 0) -> torch.Tensor:
    """``pa_attention`` for one mixed batch; writes ``out`` [T, Hq, d] and returns it.  A byte
    pool is an FP8 (E4M3) cache: ``pa_attention_fp8`` with the two scales (decode rows only).

    ``workspace`` is a caller-owned uint8 device tensor of at least ``workspace_size(...)``
    bytes (allocated here when omitted).  ``num_prefill_seqs`` is the count of sequences with
    more than one query row (0 = not known).  ``shared_prefix_tokens`` (a multiple of 512 and
    of the block size, decode rows only) says that every sequence's first keys are the same
    blocks: they are attended once for all rows and merged with each sequence's own keys."""
    lib = load_library()
    need = workspace_size(q.shape[0], q.shape[1], q.shape[2], max_seq_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = workspace.data_ptr() if workspace is not None and workspace.numel() else None
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    hint = PABatchHint(int(max_query_len), int(max_seq_len), int(num_prefill_seqs),
                       int(shared_prefix_tokens))
    descs = [describe(x) for x in (q, k_cache, v_cache, block_tables, seq_lens, query_start_loc)]
    if _is_fp8(k_cache):
        sc = PAKVScales(float(k_scale), float(v_scale))
        _check(lib.pa_attention_fp8(*[ctypes.byref(d) for d in descs], ctypes.c_float(scale),
                                    ctypes.byref(describe(out)), ctypes.byref(hint),
                                    ctypes.byref(sc), wptr, wbytes, _stream_handle(stream)))
    else:
        _check(lib.pa_attention(*[ctypes.byref(d) for d in descs], ctypes.c_float(scale),
                                ctypes.byref(describe(out)), ctypes.byref(hint), wptr, wbytes,
                                _stream_handle(stream)))
    return out


TIMED_KERNELS = {"decode": 0, "prefill": 1, "shared_prefix": 2}


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """``pa_copy_blocks``: copy K and V of block ``pairs[i, 0]`` to block ``pairs[i, 1]``
    (int32 [n, 2] device tensor), e.g. the copy-on-write pairs of the block manager."""
    lib = load_library()
    _check(lib.pa_copy_blocks(ctypes.byref(describe(k_cache)), ctypes.byref(describe(v_cache)),
                              ctypes.byref(describe(pairs.contiguous())), _stream_handle(stream)))


def set_timing_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event],
                      kernel: str = "decode"):
    """Record ``start``/``stop`` around every later launch of ``kernel`` ("decode": the
    decode-partition kernel, "prefill": the chunked-prefill kernel, "shared_prefix": the
    shared-prefix pass) on this thread
    (``None, None`` turns that hook off).  Measurement only; no work changes."""
    lib = load_library()
    if start is None or stop is None:
        _check(lib.pa_set_timing_events(TIMED_KERNELS[kernel], None, None))
    else:
        _check(lib.pa_set_timing_events(TIMED_KERNELS[kernel], start.cuda_event, stop.cuda_event))


def set_wait_limit(limit_ns: int) -> None:
    """``pa_set_wait_limit``: how long any wait inside later attention kernels of this thread
    may last before it gives up and reports PA_ERR_TIMEOUT (default 2 s)."""
    _check(load_library().pa_set_wait_limit(int(limit_ns)))


def set_stream_error_word(stream, word: Optional[torch.Tensor]) -> None:
    """``pa_set_stream_error_word``: later calls on ``stream`` report device errors into ``word``
    (a zeroed one-element int32 device tensor the caller keeps alive), read back by
    ``get_device_error(stream)``; ``None`` returns the stream to the device's shared word."""
    if word is not None and (word.dtype != torch.int32 or word.numel() < 1 or not word.is_cuda):
        raise ValueError("the error word must be a one-element int32 device tensor")
    _check(load_library().pa_set_stream_error_word(
        _stream_handle(stream), word.data_ptr() if word is not None else None))


def get_device_error(stream=None):
    """Synchronise the stream and return (status, bits) of the device error word (cleared)."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    st = lib.pa_get_device_error(_stream_handle(stream), ctypes.byref(bits))
    return st, int(bits.value)


@dataclass
class BatchDescriptor:
    """The scheduler-facing description of one continuous-batching step, on the device.

    Sequences may mix prefill chunks (several query rows) and decode steps (one row) in any
    order ("vLLM: LLM Inference That Doesn't Waste Your GPU", "Continuous batching").
    ``slot_mapping`` addresses the cache slots of this step's new tokens; ``max_query_len``,
    ``max_seq_len`` and ``num_prefill_seqs`` are the host-side hint the launch is planned from.
    """

    query_start_loc: torch.Tensor
    seq_lens: torch.Tensor
    block_tables: torch.Tensor
    slot_mapping: torch.Tensor
    max_query_len: int
    max_seq_len: int
    num_prefill_seqs: int = 0

    @classmethod
    def from_host(cls, seq_lens, query_lens, block_tables, block_size: int, device="cuda",
                  non_blocking: bool = False) -> "BatchDescriptor":
        """Build from host lists: ``seq_lens[s]`` keys after the step, ``query_lens[s]`` new
        rows (the last ones of the sequence), ``block_tables`` int32 [N, MB]."""
        sl = torch.as_tensor(seq_lens, dtype=torch.int32).contiguous()
        ql = torch.as_tensor(query_lens, dtype=torch.int32).contiguous()
        bt = torch.as_tensor(block_tables, dtype=torch.int32)
        if bt.dim() != 2 or bt.shape[0] != sl.shape[0] or ql.shape != sl.shape:
            raise ValueError("block_tables must be [N, MB] with N = len(seq_lens) = len(query_lens)")
        if bt.stride(1) != 1:
            bt = bt.contiguous()
        n = int(sl.shape[0])
        qsl = torch.empty(n + 1, dtype=torch.int32)
        cap = int(ql.to(torch.int64).clamp(min=0).sum())
        sm = torch.empty(cap, dtype=torch.int64)
        ptr = lambda t, c: ctypes.cast(t.data_ptr(), ctypes.POINTER(c)) if t.numel() else None
        _check(load_library().pa_step_slot_mapping(
            n, ptr(sl, ctypes.c_int32), ptr(ql, ctypes.c_int32), ptr(bt, ctypes.c_int32),
            bt.stride(0) if n else 0, int(bt.shape[1]), int(block_size),
            ptr(qsl, ctypes.c_int32), ptr(sm, ctypes.c_int64), cap))
        dev = lambda x: x.to(device, non_blocking=non_blocking)
        return cls(dev(qsl), dev(sl), dev(bt), dev(sm), int(ql.max()) if n else 0,
                   int(sl.max()) if n else 0, int((ql > 1).sum()))
