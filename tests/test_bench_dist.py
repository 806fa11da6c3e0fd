"""The benchmark's multi-rank host logic on CPU with gloo, world size 2: replicas report the
maximum time over ranks, throughput aggregates over ranks, and the reference arm runs on rank 0
only while the other rank exits without work."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.5 + rank, world)
        args = bench.parse_args(["--impl", "reference", "--workload", "tiny_f32", "--steps", "1", "--warmup", "1"])
        line = bench.run_reference(args, rank, world)
        q.put((rank, t, None if line is None else (line["impl"], line["n_gpus"], line["value"] > 0)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_reference_on_rank0_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict((r, (t, line)) for r, t, line in (q.get(timeout=240) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 2.5
    assert out[0][1] == ("reference", 2, True)
    assert out[1][1] is None


def test_replica_throughput_is_whole_job():
    import bench
    assert bench.replica_throughput(1e12, 4, 1000.0) == pytest.approx(4.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def test_peak_choice_follows_the_clock_record():
    """A short region at full clock divides by the burst figure; the sustained one applies only
    when the power cap was seen during a region of at least a second."""
    import bench
    peaks = {"bf16_tflops": 1915.3, "bf16_tflops_sustained": 1713.1}
    free = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    capped = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert bench.choose_peak(peaks, free, 0.014)[:2] == (1915.3, "burst")
    assert bench.choose_peak(peaks, free, 5.0)[:2] == (1915.3, "burst")
    assert bench.choose_peak(peaks, capped, 0.2)[:2] == (1915.3, "burst")
    assert bench.choose_peak(peaks, capped, 3.0)[:2] == (1713.1, "sustained")
    assert bench.choose_peak(peaks, None, 3.0)[:2] == (1915.3, "burst")


def test_fp32_alu_peak_derivation():
    import bench
    # 152 SMs x 128 lanes x 2 FLOP x 2.07 GHz
    assert bench.fp32_alu_peak(152, 2070.0) == pytest.approx(80.55, rel=1e-3)


def test_committed_traffic_only_for_the_measured_code(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu figure only while the device code carries
    the stamp it was measured on; any other stamp, a missing entry or a missing file gives null."""
    import json
    import bench
    stamp = bench.source_stamp()
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"bwd_tc_kernel": {"gqa_bf16": {"dram_bytes_per_launch": 123456, "source_stamp": stamp}},
             "fwd_tc_kernel": {"gqa_bf16": {"dram_bytes_per_launch": 7, "source_stamp": "0" * 64}}}
    (prof / "ncu_traffic.json").write_text(json.dumps(entry))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("bwd_tc_kernel", "gqa_bf16") == 123456
    assert bench.committed_traffic("fwd_tc_kernel", "gqa_bf16") is None  # measured on other code
    assert bench.committed_traffic("fwd_tc_kernel", "decode_bf16") is None  # no entry
    (prof / "ncu_traffic.json").unlink()
    assert bench.committed_traffic("bwd_tc_kernel", "gqa_bf16") is None  # no file


def test_code_stamp_ignores_comments_but_not_code():
    """The stamp follows the device code only: a comment edit keeps it, a code edit changes it."""
    from exact_attention_50_gb300 import build
    base = build.code_stamp()

    def read_with(edit):
        def read(path):
            text = open(path).read()
            return edit(text) if path.endswith("fwd_tc.cuh") else text
        return read

    assert build.code_stamp(read_with(lambda t: t + "\n// a comment only\n")) == base
    assert build.code_stamp(read_with(lambda t: t.replace("kRescaleLog2 = 8.0f", "kRescaleLog2 = 7.0f"))) != base
