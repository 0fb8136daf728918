"""bench.py's bookkeeping on the CPU: the algorithmic byte counts behind the reported rooflines, the
rule that ncu traffic is reported only for the sources it was captured on, and the clock-sample
summary (throttle reasons inside the timed region)."""
import datetime
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_encode_bytes_of_the_bench_batch():
    # 64 sequences x 8 kv heads = 512 blocks per kind: bf16 in; codes, 512 B of parameters and a
    # 4-byte tile factor out per tile
    inp, out = bench.enc_bytes(512)
    assert inp == 2 * 512 * 128 * 128 * 2 == 33_554_432
    assert out == 512 * (4096 + 516) + 512 * (4096 + 516) == 4_722_688
    inp4, out4 = bench.enc_bytes(512, k_bits=4)
    assert inp4 == inp and out4 == 512 * (8192 + 516) + 512 * (4096 + 516) == 6_819_840


def test_decode_bytes_of_the_bench_call():
    # B 16 x 8 kv heads x 256 tiles, each a K and a V tile of 4096 B codes + 516 B; bf16 queries and
    # fp32 outputs of 16 x 32 heads
    cache, q, out = bench.dec_bytes()
    assert cache == 16 * 8 * 256 * 2 * (4096 + 516) == 302_252_032
    assert q == 16 * 32 * 128 * 2 and out == 16 * 32 * 128 * 4
    assert cache + q + out == 302_645_248  # the decode bytes_per_step of the bench line
    # 72 B per kv-head token at K2/V2 (32 B of codes + 4 B of parameters per cache), plus the factors
    assert cache == 16 * 8 * 32768 * 72 + 16 * 8 * 256 * 8


def test_ragged_decode_bytes():
    # the bench cache through the ragged formula: the same bytes as the fixed-length count
    assert bench.ragged_dec_bytes([32768] * 16, 32, 8, 2, 2) == bench.dec_bytes()
    # one sequence of 2 full tiles + 5 tail tokens, 4-bit K / 2-bit V, 40q/10kv heads, by hand:
    # per kv head 2 x ((8192 + 512 + 4) + (4096 + 512 + 4)) B of tiles + 5 x 128 x 2 B x 2 of tails
    cache, q, out = bench.ragged_dec_bytes([2 * 128 + 5], 40, 10, 4, 2)
    assert cache == 10 * (2 * (8708 + 4612) + 5 * 512) == 292_000
    assert q == 40 * 128 * 2 and out == 40 * 128 * 4
    # an empty sequence reads nothing of the cache
    assert bench.ragged_dec_bytes([0], 8, 2, 2, 2)[0] == 0


def test_ncu_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        committed = json.load(f)
    entry = committed["kvarn_decode_attention"]
    # the committed capture was taken on these sources: the bench reports it
    if entry["source_hash"] == bench.source_hash("kvarn_decode_attention"):
        assert bench.ncu_traffic("kvarn_decode_attention") == entry["bytes_per_launch"]
    # each kernel's hash covers its own sources only: the decode's does not change with the encoder
    assert "encode.cu" not in bench.KERNEL_SOURCES["kvarn_decode_attention"]
    assert "decode_attn.cu" not in bench.KERNEL_SOURCES["kvarn_encode_kv_blocks"]
    # a capture of other sources is not reported
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "0" * 16)
    assert bench.ncu_traffic("kvarn_decode_attention") is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_clock_summary_keeps_samples_of_the_timed_region(tmp_path):
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    lines = []
    for i, (mhz, thermal) in enumerate([(1500, "Not Active"), (2070, "Not Active"), (2070, "Not Active"),
                                        (1980, "Active"), (900, "Active")]):
        ts = (t0 + datetime.timedelta(milliseconds=100 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{ts}, {mhz}, 2070, 800.0, 0x0, Not Active, Not Active, {thermal}, Not Active")
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    c = bench.ClockSampler(0)
    c.path, c.proc = str(path), object()  # a finished sampler's file, no nvidia-smi here
    base = t0.timestamp()
    # samples 1..2 (with the 0.1 s widening: 0..3): sample 3 reports sw_thermal_slowdown
    s = c.summary(base + 0.1, base + 0.2)
    assert s["samples"] == 4 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_thermal_slowdown"]
    assert s["sm_mhz"] == 2025.0  # median of 1500, 2070, 2070, 1980
    # a region between samples takes the nearest one
    s = c.summary(base + 10.0, base + 10.0)
    assert s["samples"] == 1 and s["sm_mhz"] == 900.0
    # no sampler: no clocks, said so
    c.proc = None
    assert bench.ClockSampler.summary(c, 0, 1)["reasons"] == ["nvidia-smi unavailable"]


def test_oracle_pool_core_count():
    avail = len(os.sched_getaffinity(0))
    assert bench.pool_cores() == avail and bench.pool_cores(0) == avail
    assert bench.pool_cores(1) == 1
    assert bench.pool_cores(10 ** 6) == avail
    assert bench.pool_cores(-3) == 1
