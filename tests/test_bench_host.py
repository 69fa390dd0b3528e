"""Host logic of bench.py, no GPU: algorithmic bytes, clock parsing, the
max-over-ranks aggregation, and the N>1 gather over a 2-rank gloo group."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from attention_block_gb300 import synth


def test_algorithmic_bytes_llama2_layer():
    # W_qkv 4096x12288 + W_o 4096x4096 + ln 4096 (fp16) + KV read 2x1024x32x128
    # + KV write 2x32x128 (fp16) + hidden + out (fp16) + one int32 position.
    w = synth.WORKLOADS[synth.LLAMA2_1K]
    expect = (4096 * 12288 + 4096 * 4096 + 4096 + 2 * 1024 * 32 * 128 + 2 * 32 * 128
              + 2 * 4096) * 2 + 4
    assert bench.algorithmic_bytes(w, [1024]) == expect == 151_035_908


def test_algorithmic_bytes_counts_each_rows_own_positions():
    w = synth.WORKLOADS[synth.SMALL_HEAD_B64]
    a = bench.algorithmic_bytes(w, [1024] * 64)
    b = bench.algorithmic_bytes(w, [1024] * 63 + [2048])
    assert b - a == 2 * 1024 * 32 * 64 * 2


def test_ffn_algorithmic_bytes():
    # W_gate, W_up, W_down [I, H] + the second norm's weight [H] + the rows
    # read and written [B, H], all 16-bit; the batched pair's internal a and
    # n round trips are not algorithmic bytes.
    w = synth.FFN_WORKLOADS[synth.LLAMA3_FFN_B16]
    expect = (3 * 14336 * 4096 + 4096 + 2 * 16 * 4096) * 2
    assert bench.ffn_bytes(w) == expect == 352_591_872
    w64 = synth.FFN_WORKLOADS[synth.B64_FFN]
    assert bench.ffn_bytes(w64) == (3 * 5632 * 2048 + 2048 + 2 * 64 * 2048) * 2 == 69_734_400


def test_parse_clocks():
    lines = [
        "0, 1965 MHz, 2070 MHz, 900.12 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900 MHz, 2070 MHz, 1000.0 W, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 345 MHz, 2070 MHz, 120.0 W, 0x1, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    c = bench.parse_clocks(lines)
    assert c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == pytest.approx(1932.5)
    assert c["reasons"] == ["sw_power_cap"]


def test_aggregate_uses_slowest_rank():
    agg = bench.aggregate([[100e9, 1.0, 10], [100e9, 2.0, 10]])
    assert agg["seconds"] == 2.0 and agg["gbs"] == pytest.approx(100.0)


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rows = bench.allgather_rows([float(rank + 1) * 1e9, 1.0 + rank, 5.0], world, "cpu")
    q.put((rank, rows, bench.aggregate(rows)))
    dist.destroy_process_group()


def test_two_rank_gather_and_aggregate_over_gloo():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rows, agg in res:
        assert rows == [[1e9, 1.0, 5.0], [2e9, 2.0, 5.0]]
        assert agg["seconds"] == 2.0 and agg["gbs"] == pytest.approx(1.5)


def test_reference_arm_prints_the_contract_line_on_the_host():
    """`bench.py --impl reference` (the float64 oracle on the host cores) needs
    no GPU: one short run on the tiny workload prints one JSON line with the
    contract's keys and a positive value."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_h256_mha4x64_b1_p128_f32", "--steps", "2",
                        "--warmup", "3", "--ref-budget", "0.2"],
                       capture_output=True, text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_h256_mha4x64_b1_p128_f32"


def test_kernel_hash_covers_every_included_source():
    """The traffic record is keyed by a hash of the fused kernels' sources;
    it must cover every header they include (e.g. the tcgen05 helpers)."""
    names = {os.path.basename(p) for p in bench.fused_kernel_sources()}
    assert {"cf_api.cu", "cf_kernel.cuh", "cf_kernel_rows.cuh", "cf_tc05.cuh", "cf_ptx.cuh",
            "cf_attention.cuh", "cf_attention_tc.cuh", "cf_cluster.cuh", "cf_params.h"} <= names


def test_default_workload_is_the_largest_single_gpu_one():
    from attention_block_gb300 import synth
    w = synth.WORKLOADS[bench.DEFAULT_WORKLOAD]
    sizes = {n: bench.algorithmic_bytes(x, [int(x.positions.split(":")[1])] * x.batch) * x.layers
             for n, x in synth.WORKLOADS.items() if x.positions.startswith("fixed")}
    assert w.layers == 32 and bench.DEFAULT_WORKLOAD == max(sizes, key=sizes.get)
