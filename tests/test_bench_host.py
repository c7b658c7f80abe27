"""Host-side pieces of bench.py: argument defaults, the peak-file reader, the
committed-traffic lookup, and the multi-rank plumbing (max over ranks and the
barrier) on world_size 2 with the gloo backend on CPU."""
import hashlib
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_default_arguments_are_one_gpu_and_the_8b_decode_step_with_its_sublines():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.workload == 4 and a.impl == "ours" and a.warmup >= 3 and a.steps > 0
    assert a.sublines and a.min_seconds >= 1.0
    assert not bench.parse_args(["--workload", "2"]).sublines and not bench.parse_args(["--kv", "int8"]).sublines
    assert not bench.parse_args(["--no-sublines"]).sublines
    assert a.early_pages and not bench.parse_args(["--no-early-pages"]).early_pages
    assert not bench.parse_args(["--window", "256"]).early_pages and bench.parse_args(["--kv", "int8"]).early_pages


def test_peaks_come_from_the_measured_file_or_the_fallback():
    hbm, bf16, kind = bench.measured_peaks()
    assert hbm > 1000 and bf16 > 100 and kind in ("measured", "fallback")


def test_committed_traffic_is_ignored_when_the_kernel_changed(tmp_path, monkeypatch):
    assert bench.committed_traffic("decode.cu", "no_such_summary.md") is None
    # a summary names the sha256 of its sources (one file, or several hashed in order)
    csrc = tmp_path / "paged_kv_gqa_cache_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_bytes(b"kernel a\n")
    (csrc / "b.cuh").write_bytes(b"header b\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = lambda *names: hashlib.sha256(b"".join((csrc / n).read_bytes() for n in names)).hexdigest()[:16]
    (tmp_path / "profiles" / "one.md").write_text(f"source_sha256_16: {sha('a.cu')}\ntraffic_bytes_per_launch: 123\n")
    (tmp_path / "profiles" / "two.md").write_text(
        f"source_sha256_16: {sha('a.cu', 'b.cuh')}\ntraffic_bytes_per_launch: 456\n")
    assert bench.committed_traffic("a.cu", "one.md") == 123
    assert bench.committed_traffic(("a.cu", "b.cuh"), "two.md") == 456
    assert bench.committed_traffic(("b.cuh", "a.cu"), "two.md") is None   # the order is part of the hash
    assert bench.committed_traffic("a.cu", "two.md") is None              # the header is part of the source
    (csrc / "b.cuh").write_bytes(b"header b, changed\n")
    assert bench.committed_traffic(("a.cu", "b.cuh"), "two.md") is None   # taken on another source
    assert bench.committed_traffic("a.cu", "one.md") == 123


def test_committed_summaries_match_the_current_sources():
    # every summary the default bench reads was taken on the kernels as they are
    for srcs, name in ((("decode.cu", "decode_kernel.cuh"), "decode_workload4.md"),
                       (("decode.cu", "decode_kernel.cuh"), "decode_workload2.md"),
                       (("decode.cu", "decode_kernel.cuh"), "decode_q8_workload4.md"),
                       (("decode.cu", "decode_kernel.cuh"), "decode_f8_workload4.md"),
                       (("prefill.cu", "prefill_kernel.cuh"), "prefill_workload3.md"),
                       (("prefill8.cu", "prefill_kernel.cuh"), "prefill8_int8_workload3.md")):
        assert bench.committed_traffic(srcs, name) is not None, name


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    got = bench.reduce_max(float(10 * rank + 1))
    q.put((rank, got))
    bench.barrier()
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


def test_reduce_max_without_a_process_group_is_the_identity():
    assert not dist.is_initialized()
    assert bench.reduce_max(3.5) == 3.5


def test_timed_repeats_reach_the_minimum_time_and_count():
    reps = bench.timed_repeats(lambda: 100.0, 1.0)          # 100 ms per repeat: 10 repeats for 1 s
    assert len(reps) == 10
    assert len(bench.timed_repeats(lambda: 900.0, 1.0)) == 5  # at least 5 repeats
    t = bench.timing_summary([1.0, 2.0, 3.0], 10)
    assert t["repeats"] == 3 and t["timed_region_s"] == 0.006 and t["ms_per_step_max"] == 0.3


def test_clock_summary_parses_samples():
    c = bench.ClockSampler("0")
    c.rows = [["0", "2070", "2070", "900.5", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
              ["0", "1965", "2070", "1350.0", "0x4", "Not Active", "Not Active", "Not Active", "Not Active"],
              ["0", "2070", "2070", "1000.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w_max": 1350.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
