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


def test_reduced_precision_cache_counts_its_own_row_bytes():
    b = _bench()
    p = I.make_problem(I.WORKLOADS["dsv2_b64_ctx8192_fp8"], with_weights=False)
    alg = b.decode_algorithmic(p)
    # 512 E4M3 codes + 64 bf16 keys (128 B) + one fp32 scale = 644 B per cached token
    assert alg["latent_bytes"] == 64 * 8192 * 644 == 337_641_472
    # queries, outputs and the work per visible token are those of the bf16 cache
    assert alg["bytes"] == 337_641_472 + 64 * 128 * 1152 + 64 * 128 * 1024 + 64 * 128 * 4
    assert alg["flops"] == 146_028_888_064


def test_prefill_work_of_a_4096_token_prompt():
    b = _bench()
    alg = b.prefill_algorithmic(I.PREFILL_CASES["prefill_dsv2_L4096_T4096"])
    # query j of a whole-prompt prefill sees j + 1 tokens: 4096 * 4097 / 2 (query, key) pairs
    assert alg["pairs"] == 8_390_656
    # keys and values rebuilt for every token and head (2 * 512 * (128 + 128) FLOP), then per pair and
    # head 2 * (128 + 64) for the score and 2 * 128 for P V
    rebuild = 2 * 4096 * 512 * 128 * 256
    attend = 2 * 8_390_656 * 128 * 320
    assert rebuild == 137_438_953_472 and attend == 687_362_539_520
    assert alg["flops"] == rebuild + attend
    # bytes: the 4096 cache rows, W_UK and W_UV, the queries and the outputs, all bf16
    assert alg["bytes"] == 2 * (4096 * 576 + 128 * 256 * 512 + 4096 * 128 * 192 + 4096 * 128 * 128)
    # per-head positional keys widen each gathered row to 512 + 128 * 64 elements
    rh = b.prefill_algorithmic(I.PREFILL_CASES["prefill_dsv2_L4096_T4096_rh"])
    assert rh["bytes"] - alg["bytes"] == 2 * 4096 * 127 * 64


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
