"""GPU: the native block manager driving the CUDA path through several serving steps.

Sequences share a system prompt through the prefix cache (and a second tenant with another
salt does not), one is forked for parallel sampling (copy-on-write on the next append), one
drops rejected speculative tokens and verifies new drafts, and a late request hits the cache
after its donors were freed.  K/V of position p is a seeded function of the token prefix
0..p, as a model's would be, so a slot holding anything but the sequence's own prefix K/V
shows up in the output.  Every step's attention is compared with the fp64 oracle run on each
sequence's own contiguous K/V (no paging at all), and pa_copy_blocks with the oracle's
block copy, bit for bit.
"""
import hashlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_290_gb300 as pa
from paged_kv_cache_290_gb300 import binding as Bd
from paged_kv_cache_290_gb300.block_manager import BlockManager

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS, NB = 8, 2, 128, 16, 96
SCALE = 1.0 / np.sqrt(D)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_290_gb300 import build
    build.build()
    pa.load_library()
    assert torch.cuda.is_available()
    pa.get_device_error()


def _u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_copy_blocks_matches_oracle_bitwise():
    g = torch.Generator().manual_seed(31)
    kc = torch.randn(40, HKV, BS, D, generator=g).half()
    vc = torch.randn(40, HKV, BS, D, generator=g).half()
    pairs = torch.tensor([[3, 17], [17 - 16, 30], [39, 0], [5, 6]], dtype=torch.int32)
    dk, dv = kc.cuda(), vc.cuda()
    Bd.copy_blocks(dk, dv, pairs.cuda())
    assert pa.get_device_error() == (0, 0)
    rk, rv = oracle.copy_blocks(kc, vc, pairs)
    assert np.array_equal(_u16(dk), rk) and np.array_equal(_u16(dv), rv)
    # an id outside the pool: that pair is skipped and reported, the others still run
    bad = torch.tensor([[2, 40], [4, 8]], dtype=torch.int32)
    Bd.copy_blocks(dk, dv, bad.cuda())
    st, bits = pa.get_device_error()
    assert st == Bd.PA_ERR_OUT_OF_RANGE and bits & 4
    rk2, rv2 = oracle.copy_blocks(torch.from_numpy(rk.view(np.int16)),
                                  torch.from_numpy(rv.view(np.int16)), bad)
    assert np.array_equal(_u16(dk), rk2) and np.array_equal(_u16(dv), rv2)


def _kv_of_prefix(tokens, p):
    """K and V rows [Hkv, d] (fp16) of position p: a seeded function of tokens[0..p]."""
    h = hashlib.blake2b(np.asarray(tokens[:p + 1], dtype=np.int64).tobytes(), digest_size=8)
    g = torch.Generator().manual_seed(int.from_bytes(h.digest(), "little") & ((1 << 62) - 1))
    return torch.randn(2, HKV, D, generator=g).half()


class Server:
    def __init__(self):
        self.bm = BlockManager(NB, BS)
        self.kc = torch.full((NB, HKV, BS, D), float("nan"), dtype=torch.float16, device="cuda")
        self.vc = torch.full_like(self.kc, float("nan"))
        self.toks = {}
        self.g = torch.Generator().manual_seed(2024)

    def step(self, new):
        """Run one step; ``new`` maps seq id -> number of rows that are new this step (their K/V
        are written, and they are the query rows).  Returns the max abs error."""
        ids = list(new)
        qlens = [new[s] for s in ids]
        desc = self.bm.descriptor(ids, qlens, max_blocks=16, pad_block=NB - 1)
        kv = [_kv_of_prefix(self.toks[s], p) for s in ids
              for p in range(len(self.toks[s]) - new[s], len(self.toks[s]))]
        k_new = torch.stack([x[0] for x in kv]).cuda()
        v_new = torch.stack([x[1] for x in kv]).cuda()
        pa.reshape_and_cache(k_new, v_new, self.kc, self.vc, desc.slot_mapping.cuda())
        t = int(desc.query_start_loc[-1])
        q = torch.randn(t, HQ, D, generator=self.g).half()
        out = torch.full((t, HQ, D), float("nan"), dtype=torch.float16, device="cuda")
        pa.attention(q.cuda(), self.kc, self.vc, desc.block_tables.cuda(), desc.seq_lens.cuda(),
                     desc.query_start_loc.cuda(), SCALE, out, desc.max_query_len,
                     desc.max_seq_len, num_prefill_seqs=desc.num_prefill_seqs)
        st, bits = pa.get_device_error()
        assert st == 0, (st, bits, pa.last_error())
        # the oracle on each sequence's own contiguous K/V
        ks, vs, starts = [], [], []
        for s in ids:
            starts.append(sum(len(x) for x in ks))
            rows = [_kv_of_prefix(self.toks[s], p) for p in range(len(self.toks[s]))]
            ks.append(torch.stack([r[0] for r in rows]))
            vs.append(torch.stack([r[1] for r in rows]))
        ref = oracle.attention_contiguous(q, torch.cat(ks), torch.cat(vs),
                                          torch.tensor(starts, dtype=torch.int64), desc.seq_lens,
                                          desc.query_start_loc, SCALE)
        o = out.cpu().double().numpy()
        assert np.isfinite(o).all()
        err = np.abs(o - ref)
        assert err.max() <= 2e-3 and np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref)
        return err.max()

    def add(self, sid, tokens, salt=0):
        cached = self.bm.add(sid, tokens, salt)
        self.toks[sid] = list(tokens)
        return cached

    def append(self, sid, tokens):
        pairs = self.bm.append(sid, tokens)
        if pairs:
            Bd.copy_blocks(self.kc, self.vc, torch.tensor(pairs, dtype=torch.int32).cuda())
        self.toks[sid] += list(tokens)
        return pairs


def test_block_manager_drives_a_serving_loop():
    rng = np.random.default_rng(5)
    srv = Server()
    system = rng.integers(0, 1000, 70).tolist()   # 4 full blocks + 6 tokens
    # step 1: the first request computes everything; the others reuse the system prompt
    c = [srv.add(1, system + rng.integers(0, 1000, 30).tolist()),
         srv.add(2, system + rng.integers(0, 1000, 5).tolist()),
         srv.add(3, system + rng.integers(0, 1000, 50).tolist(), salt=99),  # other tenant
         srv.add(4, system[:64] + rng.integers(0, 1000, 3).tolist())]
    assert c == [0, 64, 0, 64]  # 4 full blocks of the system prompt; the tenant shares none
    srv.step({1: 100, 2: 75 - 64, 3: 120, 4: 67 - 64})
    # step 2: parallel sampling of request 2, then one decode token for everyone
    srv.bm.fork(2, 5)
    srv.toks[5] = list(srv.toks[2])
    cow = [srv.append(s, [int(rng.integers(0, 1000))]) for s in (1, 2, 3, 4, 5)]
    assert cow[1] and not cow[0] and not cow[2]      # request 2's shared partial block copied
    srv.step({s: 1 for s in (1, 2, 3, 4, 5)})
    # step 3: request 1 rejects two of three drafts (truncate), then verifies four new drafts
    srv.bm.truncate(1, len(srv.toks[1]) - 2)
    srv.toks[1] = srv.toks[1][:-2]
    srv.append(1, rng.integers(0, 1000, 4).tolist())
    srv.append(5, rng.integers(0, 1000, 3).tolist())
    srv.step({1: 4, 5: 3, 3: 1})
    # step 4: donors freed; a late request still finds the system prompt in the cache
    for s in (2, 4, 5):
        srv.bm.free(s)
        del srv.toks[s]
    assert srv.add(6, system + [7, 7, 7]) == 64
    srv.step({6: 73 - 64, 1: 1})


@pytest.mark.parametrize("make", ["mixed", "decode", "shared"])
def test_step_replays_in_a_cuda_graph(make):
    """A serving step (scatter-write, then attention) captured once in a CUDA graph and
    replayed: the mixed step forks the prefill launch, the shared-prefix step its pass, onto the
    library's side stream and joins it back with events, which a capture records as a fork and a
    join.  The replay must give the oracle's result, like an eager call."""
    from _cases import small_decode, small_mixed, small_shared
    b = (small_mixed(seed=9250) if make == "mixed" else
         small_shared(seed=9252) if make == "shared" else small_decode(seed=9251))
    sp = b.meta.get("shared_prefix_len", 0) if make == "shared" else 0
    dev = "cuda"
    kc, vc = b.k_cache_pre.to(dev), b.v_cache_pre.to(dev)
    k_new, v_new, slots = b.k_new.to(dev), b.v_new.to(dev), b.slot_mapping.to(dev)
    q = b.q.to(dev)
    bt, sl, qsl = b.block_tables.to(dev), b.seq_lens.to(dev), b.query_start_loc.to(dev)
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(max(1, pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim,
                                              b.max_seq_len)), dtype=torch.uint8, device=dev)

    def step():
        pa.reshape_and_cache(k_new, v_new, kc, vc, slots)
        pa.attention(q, kc, vc, bt, sl, qsl, b.scale, out, b.max_query_len, b.max_seq_len,
                     workspace=ws, num_prefill_seqs=b.num_prefill_seqs, shared_prefix_tokens=sp)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the default stream (creates the side stream)
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.fill_(float("nan"))
    kc.copy_(b.k_cache_pre.to(dev))
    vc.copy_(b.v_cache_pre.to(dev))
    graph.replay()
    torch.cuda.synchronize()
    st, bits = pa.get_device_error()
    assert st == 0, (st, bits, pa.last_error())
    rk, rv = oracle.reshape_and_cache(b.k_new, b.v_new, b.k_cache_pre, b.v_cache_pre,
                                      b.slot_mapping)
    assert np.array_equal(_u16(kc), rk) and np.array_equal(_u16(vc), rv)
    ref = oracle.attention_batch(b)
    o = out.cpu().double().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - ref)
    assert err.max() <= 2e-3 and np.linalg.norm(err) <= 1e-3 * np.linalg.norm(ref)
