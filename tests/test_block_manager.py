"""The native block manager (include/pa_block_manager.h) on the CPU: prefix sharing, cache salt,
eviction, copy-on-write, truncation, capacity errors and the step descriptor.

The central check is a content model independent of allocation policy: what a slot holds is
identified with the token prefix whose K/V it stores (K/V at position p depend on tokens 0..p).
An engine driven by the manager computes K/V only for tokens past the reused prefix and runs
the copy-on-write copies it is given; after every operation, every live sequence must find at
each position p exactly its own prefix tokens[0..p].  A wrong cache hit, a missed copy or a
block reused while still referenced breaks that.
"""
import random

import pytest

from paged_kv_cache_290_gb300 import binding as B
from paged_kv_cache_290_gb300.block_manager import BlockManager


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_290_gb300 import build
    build.build()
    B.load_library()


class Engine:
    """Drives a BlockManager like a serving loop and keeps the content of every slot."""

    def __init__(self, nb, bs, caching=True):
        self.bm = BlockManager(nb, bs, caching)
        self.nb, self.bs = nb, bs
        self.slots = {}   # slot -> prefix tuple whose K/V it holds
        self.toks = {}    # seq id -> tokens
        self.reused = 0

    def _write(self, sid, start):
        length, table = self.bm.sequence(sid)
        t = self.toks[sid]
        assert length == len(t)
        for p in range(start, length):
            self.slots[table[p // self.bs] * self.bs + p % self.bs] = tuple(t[:p + 1])

    def add(self, sid, tokens, salt=0):
        cached = self.bm.add(sid, tokens, salt)
        assert cached % self.bs == 0 and 0 <= cached < len(tokens)
        self.reused += cached
        self.toks[sid] = list(tokens)
        self._write(sid, cached)
        return cached

    def append(self, sid, tokens):
        copies = self.bm.append(sid, tokens)
        for src, dst in copies:
            for off in range(self.bs):
                if src * self.bs + off in self.slots:
                    self.slots[dst * self.bs + off] = self.slots[src * self.bs + off]
        start = len(self.toks[sid])
        self.toks[sid] += list(tokens)
        self._write(sid, start)
        return copies

    def truncate(self, sid, n):
        self.bm.truncate(sid, n)
        self.toks[sid] = self.toks[sid][:n]

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.toks[child] = list(self.toks[parent])

    def free(self, sid):
        self.bm.free(sid)
        del self.toks[sid]

    def check(self):
        used = set()
        for sid, t in self.toks.items():
            length, table = self.bm.sequence(sid)
            assert length == len(t) and len(table) == (len(t) + self.bs - 1) // self.bs
            used.update(table)
            for p in range(len(t)):
                got = self.slots.get(table[p // self.bs] * self.bs + p % self.bs)
                assert got == tuple(t[:p + 1]), (sid, p)
        st = self.bm.stats()
        assert st.num_seqs == len(self.toks)
        assert len(used) + st.free_blocks + st.evictable_blocks == self.nb
        assert st.evictable_blocks <= st.cached_blocks


def test_shared_prompt_reuses_full_blocks_only():
    e = Engine(64, 4)
    sys_prompt = list(range(100, 110))          # 2.5 blocks
    assert e.add(1, sys_prompt + [1, 2]) == 0
    assert e.add(2, sys_prompt + [7]) == 8      # both full blocks of the shared prefix
    t1, t2 = e.bm.sequence(1)[1], e.bm.sequence(2)[1]
    assert t1[:2] == t2[:2] and t1[2] != t2[2]  # third (partial) block is private
    e.check()


def test_last_token_block_is_always_recomputed():
    e = Engine(64, 4)
    e.add(1, list(range(8)))
    assert e.add(2, list(range(8))) == 4        # block holding token 7 is not reused
    e.check()


def test_salt_and_prefix_chain_decide_sharing():
    e = Engine(64, 4)
    e.add(1, [1, 2, 3, 4, 5, 6, 7, 8, 9])
    assert e.add(2, [1, 2, 3, 4, 5, 6, 7, 8, 9], salt=7) == 0      # another tenant
    assert e.add(3, [0, 2, 3, 4, 5, 6, 7, 8, 9]) == 0              # first block differs
    assert e.add(4, [1, 2, 3, 4, 0, 6, 7, 8, 9]) == 4              # second differs
    # the same second block behind a different first block is not a hit (chained key)
    e.add(5, [9, 9, 9, 9, 5, 6, 7, 8, 0])
    assert e.add(6, [9, 9, 9, 9, 5, 6, 7, 8, 1]) == 8
    e.check()


def test_prefix_cache_survives_free_and_evicts_least_recent():
    e = Engine(6, 4)
    a, b = list(range(10, 19)), list(range(20, 29))  # 3 blocks each, 2 full
    e.add(1, a)
    e.free(1)
    st = e.bm.stats()
    assert st.evictable_blocks == 2 and st.free_blocks == 4
    assert e.add(2, a) == 8                     # both full blocks come back from the cache
    e.free(2)
    e.add(3, b)                                 # 3 of the 4 free blocks
    e.free(3)                                   # a's blocks released first, then b's
    e.add(4, list(range(30, 39)))               # needs 3: 1 free + evicts 2 (a's, oldest)
    assert e.add(5, a[:5]) == 0                 # a's first block was evicted
    e.check()


def test_fork_then_append_copies_the_shared_partial_block():
    e = Engine(32, 4)
    e.add(1, [1, 2, 3, 4, 5, 6])
    e.fork(1, 2)
    assert e.bm.sequence(1)[1] == e.bm.sequence(2)[1]
    copies = e.append(2, [70])
    assert len(copies) == 1
    src, dst = copies[0]
    t1, t2 = e.bm.sequence(1)[1], e.bm.sequence(2)[1]
    assert t1[0] == t2[0] and t1[1] == src and t2[1] == dst and src != dst
    assert e.append(1, [80]) == []              # now the sole user: written in place
    e.check()


def test_truncate_then_append_reclaims_or_copies():
    e = Engine(32, 4)
    e.add(1, list(range(12)))                   # 3 full blocks, 2 of them cached by add
    e.truncate(1, 6)                            # rejected speculative tokens
    assert e.append(1, [99]) == []              # sole user of the cached block: in place
    e.check()
    e.add(2, list(range(12)) + [5])
    e.fork(2, 3)
    e.truncate(3, 6)
    assert len(e.append(3, [42])) == 1          # shared with sequence 2: copied
    e.check()


def test_out_of_blocks_changes_nothing():
    e = Engine(4, 4)
    e.add(1, list(range(10)))                   # 3 blocks
    before = (e.bm.stats(), e.bm.sequence(1))
    with pytest.raises(B.PAError) as ex:
        e.add(2, list(range(50, 59)))
    assert ex.value.status == B.PA_ERR_NO_BLOCKS
    with pytest.raises(B.PAError):
        e.bm.append(1, list(range(7)))          # needs 2 more blocks, 1 left
    assert (e.bm.stats(), e.bm.sequence(1)) == before
    e.check()


def test_bad_arguments():
    bm = BlockManager(8, 4)
    bm.add(1, [1, 2])
    for call in (lambda: bm.add(1, [3]), lambda: bm.add(2, []), lambda: bm.append(9, [1]),
                 lambda: bm.truncate(1, 0), lambda: bm.truncate(1, 3), lambda: bm.fork(1, 1),
                 lambda: bm.free(5), lambda: bm.descriptor([1], [3], 4),
                 lambda: bm.descriptor([1], [1], 0)):
        with pytest.raises(B.PAError) as ex:
            call()
        assert ex.value.status == B.PA_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        BlockManager(0, 16)


def test_step_descriptor_addresses_the_new_tokens():
    bm = BlockManager(64, 16)
    bm.add(10, list(range(40)))
    bm.add(11, list(range(40)) + [1, 2])
    bm.add(12, [5])
    d = bm.descriptor([10, 11, 12], [40, 1, 1], max_blocks=4, pad_block=63)
    assert d.query_start_loc.tolist() == [0, 40, 41, 42]
    assert d.seq_lens.tolist() == [40, 42, 1]
    assert d.max_query_len == 40 and d.max_seq_len == 42 and d.num_prefill_seqs == 1
    for s, sid in enumerate([10, 11, 12]):
        length, table = bm.sequence(sid)
        row = d.block_tables[s].tolist()
        assert row[:len(table)] == table and all(x == 63 for x in row[len(table):])
        q0, q1 = int(d.query_start_loc[s]), int(d.query_start_loc[s + 1])
        for i, slot in enumerate(d.slot_mapping[q0:q1].tolist()):
            p = length - (q1 - q0) + i
            assert slot == table[p // 16] * 16 + p % 16


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("caching", [True, False])
def test_random_serving_loop_keeps_every_prefix_intact(seed, caching):
    rng = random.Random(seed)
    bs = rng.choice([2, 4, 16])
    e = Engine(rng.randint(24, 80), bs, caching)
    prompts = [[rng.randrange(5) for _ in range(rng.randint(1, 5 * bs))] for _ in range(4)]
    next_id = 0
    for _ in range(300):
        live = list(e.toks)
        op = rng.random()
        try:
            if op < 0.3 or not live:
                base = rng.choice(prompts)
                tail = [rng.randrange(5) for _ in range(rng.randint(0, 2 * bs))]
                e.add(next_id, (base + tail) or [1], salt=rng.choice([0, 0, 0, 1]))
                next_id += 1
            elif op < 0.6:
                e.append(rng.choice(live), [rng.randrange(5) for _ in range(rng.randint(1, 6))])
            elif op < 0.7:
                e.fork(rng.choice(live), next_id)
                next_id += 1
            elif op < 0.8:
                sid = rng.choice(live)
                e.truncate(sid, rng.randint(1, len(e.toks[sid])))
            else:
                e.free(rng.choice(live))
        except B.PAError as ex:
            assert ex.status == B.PA_ERR_NO_BLOCKS
        e.check()
    if caching:
        assert e.reused > 0  # the loop really exercised prefix sharing
    else:
        assert e.reused == 0 and e.bm.stats().cached_blocks == 0
