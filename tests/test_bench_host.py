"""Host-side logic of bench.py: byte/op accounting, the replica aggregation over
ranks (world size 2 on the gloo backend, CPU only) and the clock parser."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_byte_accounting():
    # W: 136 bytes per 256 weights; Q8_1: 1 byte + 4/32 bytes per value; y: 4 bytes
    assert bench.matmul_bytes(1, 4096, 4096) == 4096 * 16 * 136 + 4096 + 128 * 4 + 4 * 4096
    assert bench.quantize_bytes(2, 256) == 2 * 256 * 4 + 2 * 256 + 2 * 8 * 4
    ms = (1, 2, 4, 8, 12, 16, 32, 64, 96)
    assert bench.step_ops(ms, 4096, 4096) == 2 * sum(ms) * 4096 * 4096
    assert abs(bench.matmul_bytes(1, 4096, 4096) / (4096 * 4096) - 0.53125) < 0.01


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # every rank reports its own elapsed time; the job time is the slowest
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"max": got}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        with open(tmp_path / f"r{r}.json") as f:
            assert json.load(f)["max"] == 15.0


def test_clock_parser(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "c.csv")
    with open(cs.path, "w") as f:
        f.write("0, 1900, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1950, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1800, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n")

    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    cs.proc = _P()
    out = cs.stop()
    assert out["sm_mhz"] == 1900 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3


def test_traffic_record_is_ignored_when_kernels_change(tmp_path, monkeypatch):
    p = tmp_path / "t.txt"
    p.write_text("kernel_source_sha256_16: deadbeefdeadbeef\n"
                 "dram_bytes_per_tc_launch_mean: 123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.recorded_traffic() is None
    p.write_text(f"kernel_source_sha256_16: {bench.kernel_source_hash()}\n"
                 "dram_bytes_per_tc_launch_mean: 123\n")
    assert bench.recorded_traffic() == 123.0
