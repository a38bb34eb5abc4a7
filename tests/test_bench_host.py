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


def test_calibration_thresholds():
    """Per shape the DP4A range ends at the first M at which another path is
    faster, the MMA range at the first M above it at which tcgen05 is faster
    (later wins do not reopen a range); each shape's thresholds apply to its
    weight-size class, the smallest shape's are the defaults."""
    from iq4_xs_quantized_gb300 import calibrate

    def row(dp, mma, tc):
        r = {"mma_us": mma, "tc_us": tc}
        if dp is not None:
            r["dp4a_us"] = dp
        return r
    ms = (1, 2, 3, 4, 8, 16, 32)
    a = {1: row(3.5, 7.5, 7.4), 2: row(4.4, 7.5, 7.4), 3: row(8.0, 7.6, 7.4), 4: row(9.0, 7.0, 7.4),
         8: row(None, 7.3, 7.4), 16: row(None, 10.0, 7.4), 32: row(None, 7.0, 8.0)}
    assert calibrate.shape_thresholds(a, ms) == (2, 2)     # MMA loses at M = 3: no MMA range
    b = dict(a)
    b[3] = row(8.0, 7.2, 7.4)
    assert calibrate.shape_thresholds(b, ms) == (2, 8)     # MMA through M = 8, tcgen05 from 16
    c = {m: row(None if m > 16 else 1.0, 2.0, 3.0) for m in ms}
    assert calibrate.shape_thresholds(c, ms) == (16, 32)   # dp4a untimed above 16
    as_json = {str(m): r for m, r in b.items()}            # JSON keys are strings
    assert calibrate.shape_thresholds(as_json, ms) == (2, 8)
    dp4a_cls, mma_cls, dflt = calibrate.class_crossovers({"64x64": a, "128x128": b, "256x256": c}, ms)
    assert dflt == (2, 2)
    assert dp4a_cls == [[int(round((64 * 64 * 128 * 128) ** 0.5)), 2], [int(round((128 * 128 * 256 * 256) ** 0.5)), 16]]
    assert [m for _, m in mma_cls] == [8, 32]


def test_tensor_work_and_roofline_gate():
    # padded tiles: M = 8 runs a 16-row tile (twice the method's work); M = 129
    # two 128-row tiles; N = 130 two 128-row weight tiles
    assert bench.tc_executed_flops(16, 4096, 4096) == 2 * 16 * 4096 * 4096
    assert bench.tc_executed_flops(8, 4096, 4096) == 2 * 16 * 4096 * 4096
    assert bench.tc_executed_flops(129, 256, 512) == 2 * 256 * 256 * 512
    assert bench.tc_executed_flops(1, 130, 512) == 2 * 256 * 16 * 512
    g = bench.roofline_gate([("fast", 9.25e6, 0.5e-6), ("ok", 9.25e6, 2.0e-6)], 6800.0)
    assert not g["ok"] and [v["call"] for v in g["violations"]] == ["fast"]
    assert bench.roofline_gate([("ok", 9.25e6, 2.0e-6)], 6800.0)["ok"]


def test_stored_launch_table_is_well_formed():
    """The calibration's warp-MMA launches: six integers each, a tile height
    of 8-32 rows, rows per CTA a multiple of 32 up to 256 (128 from 24
    activation rows on), a K split the K range holds, one or two CTAs per SM;
    at most one entry per (N, K, tile height)."""
    from iq4_xs_quantized_gb300 import calibrate
    table = calibrate.load_table()
    if not table or "mma_launch" not in table:
        pytest.skip("no calibrated table")
    seen = set()
    for e in table["mma_launch"]:
        assert len(e) == 6 and all(isinstance(v, int) for v in e), e
        N, K, mt, R, S, occ = e
        assert N >= 1 and K % 512 == 0 and mt in (8, 16, 24, 32), e
        assert R % 32 == 0 and 32 <= R <= (256 if mt <= 16 else 128), e
        assert 1 <= S <= min(8, K // 512) and occ in (1, 2), e
        assert (N, K, mt) not in seen, e
        seen.add((N, K, mt))

