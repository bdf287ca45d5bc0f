"""The benchmark's roofline accounting, without a GPU.

The numerator of the roofline fraction is the algorithmic work of one decode call: every cached row
read once per sequence (576 bf16 = 1152 B), the absorbed queries read and the latent outputs written
once, 4 B of block table per 64-token block, and 2 * H * (576 + 512) FLOPs per visible (token, query).
Recorded DRAM traffic is reported only while the decode sources are the ones it was measured on."""
import importlib.util
import json
import os

import mla_inputs as I

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_accounting", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_metric_point_algorithmic_work():
    b = _bench()
    p = I.make_problem(I.WORKLOADS["dsv2_b64_ctx8192"], with_weights=False)
    alg = b.decode_algorithmic(p)
    # 64 sequences x 8192 cached tokens x 1152 B
    assert alg["latent_bytes"] == 64 * 8192 * 1152 == 603_979_776
    # + q (64 x 128 x 1152 B) + o_lat (64 x 128 x 1024 B) + block table (64 x 128 blocks x 4 B)
    assert alg["bytes"] == 603_979_776 + 64 * 128 * 1152 + 64 * 128 * 1024 + 64 * 128 * 4 == 621_838_336
    assert alg["flops"] == 2 * 128 * (576 + 512) * 64 * 8192 == 146_028_888_064
    assert alg["cached_tokens"] == 64 * 8192


def test_causal_queries_count_only_visible_tokens():
    b = _bench()
    w = I.Workload("two_queries", I.DSV2, "bf16", 2, 1, 1, 2, 2, 7, "direct")
    p = I.make_problem(w, with_weights=False, lens=[10, 0])
    alg = b.decode_algorithmic(p)
    kv = p.kv_len.tolist()
    assert kv == [12, 2]
    vis = sum(max(0, k - (2 - 1 - j)) for k in kv for j in range(2))   # 11 + 12 + 1 + 2
    assert vis == 26
    assert alg["flops"] == 2 * 128 * (576 + 512) * vis
    assert alg["latent_bytes"] == (12 + 2) * 1152


def test_recorded_traffic_is_dropped_when_the_sources_change(tmp_path, monkeypatch):
    b = _bench()
    rec = {"workload": "dsv2_b64_ctx8192", "source_sha": b.decode_source_hash(), "dram_bytes_per_launch": 123}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(b, "TRAFFIC_FILE", str(path))
    assert b.recorded_traffic("dsv2_b64_ctx8192") == 123
    assert b.recorded_traffic("dsv2_b16_ctx4096") is None
    rec["source_sha"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert b.recorded_traffic("dsv2_b64_ctx8192") is None
