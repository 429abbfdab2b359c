"""CPU tests of bench.py's bookkeeping: algorithmic bytes, launch counts and the multi-rank
(max-over-ranks) reduction, the latter with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench
from paged_kv_cache_290_gb300 import workloads as W
from _cases import small_mixed, small_prefix, small_spec


def test_70b_step_bytes_match_the_hand_count():
    """32 x 8192 keys x 8 kv heads x 128 x 2 B x (K+V) + Q/out + table entries + descriptor."""
    b = W.llama70b_decode(keep_contiguous=False, keep_pre=False)
    n = bench.algorithmic_bytes(b)
    kv = 32 * 8192 * 8 * 128 * 2 * 2
    qo = 2 * 32 * 64 * 128 * 2
    table = 32 * 512 * 4
    desc = 32 * 4 + 33 * 4
    assert n["kv_logical"] == n["kv_unique"] == kv == 2 ** 30
    assert n["attention_logical"] == kv + qo + table + desc == 1_074_856_196
    assert n["decode_rows"] == 32
    assert n["flops"] == 4 * 64 * 128 * 32 * 8192
    assert bench.launches_per_step(b) == 3  # scatter-write, decode partitions, merge


def test_fp8_cache_halves_the_kv_bytes():
    b16 = W.llama70b_decode(8, keep_contiguous=False, keep_pre=False)
    b8 = W.to_fp8(b16)
    n16, n8 = bench.algorithmic_bytes(b16), bench.algorithmic_bytes(b8)
    assert n8["kv_logical"] * 2 == n16["kv_logical"] == 8 * 8192 * 8 * 128 * 2 * 2
    assert n16["attention_logical"] - n8["attention_logical"] == n8["kv_logical"]
    t = int(b8.k_new.shape[0])
    assert n8["reshape_and_cache"] == t * 8 * 128 * 2 * 3 + t * 8


def test_aliased_prefix_counts_unique_blocks_once():
    b = small_prefix()
    n = bench.algorithmic_bytes(b)
    row = b.num_kv_heads * b.head_dim * 4
    shared = b.meta["shared_prefix_len"]
    assert n["kv_logical"] == sum(s.seq_len for s in b.seqs) * row
    assert n["kv_unique"] == (shared + sum(s.seq_len - shared for s in b.seqs)) * row


def test_shared_prefix_pass_splits_the_kernel_bytes():
    """With the pass, the decode kernel moves the keys past the prefix and the pass moves the
    prefix once plus every query row; together they are the step's unique K/V."""
    b = W.prefix_shared_decode(keep_contiguous=False, keep_pre=False)
    sp = bench.shared_prefix_tokens(b)
    assert sp == 2048
    n0, n = bench.algorithmic_bytes(b), bench.algorithmic_bytes(b, sp)
    row = b.num_kv_heads * b.head_dim * 4
    q = b.num_tokens * b.num_q_heads * b.head_dim * 2
    assert n["shared_prefix_kernel_bytes"] == sp * row + q
    assert n0["decode_kernel_bytes"] - n["decode_kernel_bytes"] == sp * row
    assert n["shared_prefix_kernel_flops"] == 4 * b.num_q_heads * b.head_dim * sp * b.num_tokens
    assert bench.launches_per_step(b, sp) == bench.launches_per_step(b) + 1 == 4
    # prefill rows or no whole shared partition: no pass (an FP8 cache is fine)
    assert bench.shared_prefix_tokens(W.to_fp8(b)) == 2048
    assert bench.shared_prefix_tokens(small_prefix()) == 0
    assert bench.shared_prefix_tokens(small_mixed()) == 0


def test_mixed_step_counts_prefill_launch():
    b = small_mixed()
    assert bench.launches_per_step(b) == 4
    # the full mixed step: 4 chunks x 8 pairs of 32-token Q tiles x 8 kv heads = 256 items of
    # the two-tile kernel; its 128 decode rows weigh about as much as the 2048 prefill rows
    # (estimate 128 / 2048 / 4 x 70 = 1.1), so the items go as launches of two thirds of the
    # SMs (101 + 101 + 54)
    m = W.mixed_step(16, keep_contiguous=False, keep_pre=False)
    assert bench.prefill_slice_ctas(m) == 101
    assert bench.prefill_launches(m, decode=True) == 3
    assert bench.launches_per_step(m) == 6
    assert bench.launches_per_step(m, num_sms=256) == 5
    # over an FP8 pool the decode rows weigh half as much (0.55): one full grid
    f8 = W.to_fp8(m)
    assert bench.prefill_slice_ctas(f8) == 0
    assert bench.prefill_launches(f8, decode=True) == 1
    # eight decode rows beside the chunks: one full grid
    m8 = W.mixed_step(16, num_decode=8, keep_contiguous=False, keep_pre=False)
    assert bench.prefill_launches(m8, decode=True) == 1
    # alone (no decode rows) it is one full grid
    assert bench.prefill_launches(W.mixed_step(16, num_decode=0, keep_contiguous=False,
                                               keep_pre=False), decode=False) == 1
    n = bench.algorithmic_bytes(b)
    assert n["decode_rows"] == sum(1 for s in b.seqs if s.query_len == 1)


def test_kernel_bytes_split_by_sequence_kind():
    """The decode kernel serves one-row sequences, the prefill kernel the rest: on a decode-only
    batch the decode kernel's bytes are the whole attention's; on a mixed batch the two add up
    to it (plus the descriptor, which both kernels read)."""
    b = W.llama70b_decode(keep_contiguous=False, keep_pre=False)
    n = bench.algorithmic_bytes(b)
    assert n["decode_kernel_bytes"] == n["attention_unique"]
    assert n["prefill_kernel_bytes"] == 0 and n["prefill_kernel_flops"] == 0
    m = small_mixed()
    n = bench.algorithmic_bytes(m)
    desc = m.num_seqs * 4 + (m.num_seqs + 1) * 4
    assert n["decode_kernel_bytes"] + n["prefill_kernel_bytes"] == n["attention_unique"] + desc
    # flops of the chunks: 4 Hq d per visible (query, key) pair, by brute force
    pairs = sum(sum(s.seq_len - s.query_len + i + 1 for i in range(s.query_len))
                for s in m.seqs if s.query_len > 1)
    assert n["prefill_kernel_flops"] == 4 * m.num_q_heads * m.head_dim * pairs


def test_roofline_bound_follows_arithmetic_intensity():
    peaks = {"hbm_gbs": 6000.0, "hbm_src": "h", "tflops": 2000.0, "tflops_src": "t"}
    n = {"decode_kernel_bytes": 10 ** 9, "prefill_kernel_bytes": 10 ** 8,
         "prefill_kernel_flops": 2 * 10 ** 11}
    r = bench.kernel_rooflines(n, {"decode": 0.2, "prefill": 0.25}, peaks)
    assert r["decode"]["bound"] == "hbm" and r["decode"]["unit"] == "GB/s"
    assert abs(r["decode"]["achieved"] - 5000.0) < 1e-6
    assert r["prefill"]["bound"] == "tensor" and r["prefill"]["unit"] == "TFLOP/s"
    assert abs(r["prefill"]["frac"] - 0.4) < 1e-9  # 800 TFLOP/s of 2000
    # beside the measured peaks: the nominal 8 TB/s and 2.25 PFLOP/s
    assert abs(r["decode"]["frac_of_nominal"] - 5000.0 / 8000.0) < 1e-12
    assert abs(r["prefill"]["frac_of_nominal"] - 800.0 / 2250.0) < 1e-12
    # a few rows per sequence (speculative verify) stays on the HBM roof
    n["prefill_kernel_flops"] = 10 ** 9
    r = bench.kernel_rooflines(n, {"prefill": 0.02}, peaks)
    assert r["prefill"]["bound"] == "hbm"


def test_spec_verify_shapes_and_launches():
    b = W.spec_verify(keep_contiguous=False, keep_pre=False)
    q = [s.query_len for s in b.seqs]
    assert len(q) == 64 and min(q) >= 2 and max(q) <= 6 and b.num_prefill_seqs == 64
    assert all(512 + s.query_len <= s.seq_len <= 4096 + s.query_len for s in b.seqs)
    # q_len x G <= 6 x 4 = 24 columns: over fp16 the key-parity prefill kernel serves them
    # (scatter, verify tiles; no decode launch); over FP8 the decode kernel does (scatter,
    # partitions, merge) and moves all the attention bytes
    assert not bench.verify_path(b) and bench.all_prefill(b)
    assert bench.launches_per_step(b) == 2
    assert bench.algorithmic_bytes(b)["decode_rows"] == 0
    f8 = W.to_fp8(b)
    assert bench.verify_path(f8) and not bench.all_prefill(f8)
    assert bench.launches_per_step(f8) == 3
    n = bench.algorithmic_bytes(f8)
    assert n["decode_rows"] == 0 and n["prefill_kernel_bytes"] == 0
    assert n["decode_kernel_bytes"] == n["attention_unique"]
    sp = small_spec()
    assert {s.query_len for s in sp.seqs if s.query_len > 1} == {2, 3, 4, 5, 6}


def test_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    """ncu DRAM traffic from profiles/traffic.json is attached to a kernel's roofline only while
    that kernel's source file hashes to the one the counters were taken on."""
    import hashlib
    import json
    csrc = tmp_path / "paged_kv_cache_290_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "pa_prefill.cu").write_text("kernel v1")
    h = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "w:prefill": {"dram_bytes_per_launch": 123, "source": "pa_prefill.cu",
                      "source_sha256_16": h}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("w", "prefill") == 123
    assert bench.load_traffic("w", "decode") is None   # no entry for that kernel
    (csrc / "pa_prefill.cu").write_text("kernel v2")  # source changed since the capture
    assert bench.load_traffic("w", "prefill") is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(1.5 + rank, world)
        bench.barrier(world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(2))
    assert results == [(0, 2.5), (1, 2.5)]


def test_single_rank_reduction_is_identity():
    assert bench.reduce_max(3.25, 1) == 3.25


def test_cpu_baseline_reports_a_single_core_time_for_a_small_sample():
    """The oracle's host timing on the tiny workload: the whole batch fits the sample, and its
    single-core time is reported beside the all-core one."""
    b = W.WORKLOADS["tiny_decode"](keep_contiguous=False, keep_pre=False)
    r = bench.cpu_baseline(b, bench.algorithmic_bytes(b), budget_s=3.0)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1
    assert f"of {b.num_seqs} of {b.num_seqs} sequences" in r["sample"]
    one = r["single_core"]
    assert one["cores"] == 1 and one["value"] > 0


def test_reference_arm_echoes_our_config_and_fills_the_cores():
    import argparse
    args = argparse.Namespace(workload="tiny_decode", steps=2, warmup=1, no_shared_prefix=False)
    res = bench.run_reference(args, world=1, rank=0)
    b = W.tiny_decode(keep_contiguous=False, keep_pre=False)
    assert res["config"] == bench.workload_config("tiny_decode", b, 0, 1)
    assert res["impl"] == "reference" and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0
    assert "sequences of the workload per step" in res["cpu_baseline"]["sample"]
    assert bench.run_reference(args, world=2, rank=1) is None  # other ranks do no work


def test_clock_sampler_counts_samples_in_the_soak_window():
    c = bench.ClockSampler("GPU-x")
    c.proc = None
    line = "GPU-x, {}, 2070, {}, 0x0, Not Active, Not Active, Not Active, {}"
    c.lines = [(0.0, line.format(1000, 150, "Not Active")),
               (1.0, line.format(1980, 900, "Active")),
               (1.2, line.format(2000, 950, "Active")),
               (3.0, line.format(900, 160, "Not Active"))]
    c.mark_load(0.5, 1.5)

    class _P:  # stands in for the finished nvidia-smi process
        def terminate(self): pass
        def wait(self, timeout=None): pass
    c.proc, c.thread = _P(), type("T", (), {"join": lambda self, timeout=None: None})()
    r = c.stop()
    assert r["samples"] == 4 and r["samples_under_load"] == 2
    assert r["sm_mhz"] == 1990.0 and r["sm_mhz_under_load_median"] == 1990.0
    assert r["reasons"] == ["sw_power_cap"]


def test_dominant_kernel_is_the_longest_at_its_roof():
    """The step's roofline names the kernel whose own work takes longest at its roof, not the one
    with the longest (possibly overlapping) event interval."""
    peaks = {"hbm_gbs": 6786.9, "tflops": 1876.8, "hbm_src": "m", "tflops_src": "m"}
    nbytes = {"decode_kernel_bytes": 2_153_076_204, "prefill_kernel": "prefill_pair_kernel",
              "prefill_kernel_bytes": 120_973_572, "prefill_kernel_flops": 170_448_125_952}
    # the prefill's interval (beside the decode kernel) is the longer one
    k = bench.kernel_rooflines(nbytes, {"decode": 0.4073, "prefill": 0.4183}, peaks)
    assert k["decode"]["bound"] == "hbm" and k["prefill"]["bound"] == "tensor"
    assert bench.dominant_kernel(k) == "decode"
    # alone, the prefill kernel is the step's only kernel
    k = bench.kernel_rooflines(nbytes, {"prefill": 0.2101}, peaks)
    assert bench.dominant_kernel(k) == "prefill"
    # a small decode beside heavy prefill work: the prefill bounds the step
    nbytes_small = dict(nbytes, decode_kernel_bytes=50_000_000)
    k = bench.kernel_rooflines(nbytes_small, {"decode": 0.16, "prefill": 0.22}, peaks)
    assert bench.dominant_kernel(k) == "prefill"
