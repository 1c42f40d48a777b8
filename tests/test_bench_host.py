"""Host-side logic of bench.py: byte counts against the pages' traffic
arithmetic, and the multi-rank timing reduction over gloo (world size 2)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from selective_state_space_138_b300 import inputs as I
from tests.oracle_pins import GOLDEN


def test_traffic_theorem_numbers_and_byte_count():
    """'Why the scan must be fused': S = B T d_in N 4, I = B T d_in 2, unfused
    6S + 3I, fused 3I (read x and delta, write y), ratio 1 + 4N."""
    g = GOLDEN["traffic"]
    bt, T, d, N = g["batch"], g["T"], g["d_in"], g["N"]
    S = bt * T * d * N * 4
    Ib = bt * T * d * 2
    assert round(S / 1e9, 2) == g["S_GB"]
    assert round(Ib / 1e9, 3) == g["I_GB"]
    assert round((6 * S + 3 * Ib) / 1e9, 1) == g["unfused_GB"]
    assert (6 * S + 3 * Ib) // (3 * Ib) == g["ratio_at_N16"] == 1 + 4 * N
    # the bench's count = the theorem's fused 3I + the z read + B, C + parameters + final state
    spec = I.ScanSpec(batch=bt, d_inner=d, L=T, N=N)
    extra = Ib + bt * T * 2 * N * 2 + d * N * 4 + 2 * d * 4 + bt * d * N * 4
    assert bench.scan_alg_bytes(spec) == 3 * Ib + extra


def test_io_counts_of_the_paper_benchmark():
    g = GOLDEN["io_counts"]
    assert g["B"] * g["L"] * g["D"] * g["N"] == g["plain"]
    assert g["B"] * g["L"] * g["D"] + g["D"] * g["N"] == g["fused"]


def test_headline_bytes_per_element_step():
    spec = I.MAMBA130M
    b = bench.scan_alg_bytes(spec)
    assert b == 203_272_192
    assert abs(b / spec.elem_steps - 0.5048) < 1e-4
    d = bench.decode_alg_bytes(I.DECODE)
    assert abs(d / I.DECODE.elem_steps_per_step - 8.517) < 1e-3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        per_rank_ms = [12.5, 17.25][rank]
        out[rank] = bench.reduce_max(per_rank_ms, world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo_world_size_2():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 17.25


def test_shards_differ_by_seed_only():
    a, b = bench.shard_spec(I.MAMBA130M, 0), bench.shard_spec(I.MAMBA130M, 1)
    assert (a.batch, a.d_inner, a.L, a.N) == (b.batch, b.d_inner, b.L, b.N)
    assert a.seed != b.seed


def test_profiled_traffic_reads_the_committed_summary(tmp_path, monkeypatch):
    """The bench takes a kernel's DRAM traffic from its committed ncu summary
    only while the recorded source hash matches the kernel's source."""
    import bench
    key = "conv1d_silu_k4_test"
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(key)
    (prof / (key + ".md")).write_text("# x\n\n- `traffic_bytes_per_launch: 12345`\n- `source_sha256: %s`\n" % h)
    assert bench.profiled_traffic(key) == 12345.0
    (prof / (key + ".md")).write_text("- `traffic_bytes_per_launch: 12345`\n- `source_sha256: %s`\n" % ("0" * 64))
    assert bench.profiled_traffic(key) is None


def test_measured_peaks_carry_every_denominator_the_bench_reports():
    """The roofline objects divide by the HBM copy bandwidth and by the bf16
    tensor peak (SSD); both must come back whether the peaks file is read or
    the fallback is taken."""
    pk = bench.measured_peaks()
    for key in ("hbm_gbs", "bf16_tflops", "sm_max_mhz", "sms", "source"):
        assert key in pk, key
    assert pk["hbm_gbs"] > 1000 and pk["bf16_tflops"] > 100


def test_scan_floors_of_the_headline_layer():
    """HBM floor of the Mamba-130M layer at 6498.7 GB/s is the 31.3 us of the
    scope table; one exponential per element-step at 32 per clock per SM is
    the binding floor."""
    pk = {"hbm_gbs": 6498.7, "sms": 148, "sm_max_mhz": 2032.0, "source": "measured"}
    sp = bench.HEADLINE
    E = sp.batch * sp.d_inner * sp.L * sp.N
    fl = bench.scan_floors_us(bench.scan_alg_bytes(sp), E, pk)
    assert abs(fl["hbm"] - 31.3) < 0.1
    assert abs(fl["exp"] - E / (148 * 32 * 2032e6) * 1e6) < 1e-6 * fl["exp"] + 0.01
    assert fl["exp"] > fl["hbm"] > fl["fp32_issue"]
