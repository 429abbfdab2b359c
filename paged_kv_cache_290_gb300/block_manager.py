"""Python face of the native block manager (``include/pa_block_manager.h``): marshalling only.

The allocator, the prefix cache, copy-on-write and the step descriptor all live in the C++
library; this class turns lists into arrays and statuses into exceptions.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import torch

from .binding import BatchDescriptor, _check, load_library


@dataclass
class Stats:
    free_blocks: int
    evictable_blocks: int
    cached_blocks: int
    num_seqs: int


def _i32(xs: Sequence[int]):
    arr = (ctypes.c_int32 * max(1, len(xs)))(*xs)
    return arr


class BlockManager:
    """Ref-counted physical blocks of one paged pool, with prefix caching.

    ``add(seq_id, tokens, salt)`` returns how many leading tokens already have K/V in reused
    blocks; ``append`` returns the copy-on-write pairs (src, dst) the caller must run through
    ``copy_blocks`` before the step's scatter-write; ``descriptor`` builds the batch
    descriptor of a step."""

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self._lib = load_library()
        self._h = self._lib.pa_bm_create(int(num_blocks), int(block_size), int(prefix_caching))
        if not self._h:
            raise ValueError("pa_bm_create failed (sizes must be >= 1)")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            self._lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, seq_id: int, tokens: Sequence[int], salt: int = 0) -> int:
        cached = ctypes.c_int32(0)
        _check(self._lib.pa_bm_add_sequence(self._h, int(seq_id), _i32(tokens), len(tokens),
                                            int(salt), ctypes.byref(cached)))
        return cached.value

    def append(self, seq_id: int, tokens: Sequence[int]) -> List[Tuple[int, int]]:
        copies = (ctypes.c_int32 * 2)()
        n = ctypes.c_int32(0)
        _check(self._lib.pa_bm_append(self._h, int(seq_id), _i32(tokens), len(tokens), copies,
                                      ctypes.byref(n)))
        return [(copies[0], copies[1])] if n.value else []

    def truncate(self, seq_id: int, new_len: int) -> None:
        _check(self._lib.pa_bm_truncate(self._h, int(seq_id), int(new_len)))

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_bm_fork(self._h, int(parent), int(child)))

    def free(self, seq_id: int) -> None:
        _check(self._lib.pa_bm_free(self._h, int(seq_id)))

    def stats(self) -> Stats:
        v = [ctypes.c_int32(0) for _ in range(4)]
        _check(self._lib.pa_bm_stats(self._h, *[ctypes.byref(x) for x in v]))
        return Stats(*[x.value for x in v])

    def sequence(self, seq_id: int) -> Tuple[int, List[int]]:
        """(length, block table) of a sequence."""
        length, nb = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(self._lib.pa_bm_sequence(self._h, int(seq_id), ctypes.byref(length), None, 0,
                                        ctypes.byref(nb)))
        out = (ctypes.c_int32 * max(1, nb.value))()
        _check(self._lib.pa_bm_sequence(self._h, int(seq_id), None, out, nb.value, None))
        return length.value, list(out[:nb.value])

    def descriptor(self, seq_ids: Sequence[int], query_lens: Sequence[int], max_blocks: int,
                   pad_block: int = 0, device: Optional[str] = None) -> BatchDescriptor:
        """The step's block tables, lengths, query offsets and slot mapping (new tokens =
        the last ``query_lens[i]`` tokens of each sequence), on ``device`` (host when None)."""
        n = len(seq_ids)
        bt = torch.empty((n, max_blocks), dtype=torch.int32)
        sl = torch.empty(n, dtype=torch.int32)
        qsl = torch.empty(n + 1, dtype=torch.int32)
        sm = torch.empty(max(1, sum(int(q) for q in query_lens)), dtype=torch.int64)
        p32 = lambda t: ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_int32))
        ids = (ctypes.c_int64 * max(1, n))(*seq_ids)
        _check(self._lib.pa_bm_step_descriptor(
            self._h, ids, _i32(query_lens), n, int(max_blocks), int(pad_block), p32(bt), p32(sl),
            p32(qsl), ctypes.cast(sm.data_ptr(), ctypes.POINTER(ctypes.c_int64))))
        sm = sm[:int(qsl[-1])]
        dev = (lambda x: x) if device is None else (lambda x: x.to(device))
        ql = [int(q) for q in query_lens]
        return BatchDescriptor(dev(qsl), dev(sl), dev(bt), dev(sm), max(ql, default=0),
                               int(sl.max()) if n else 0, sum(1 for q in ql if q > 1))
