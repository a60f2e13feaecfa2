"""Host logic of ``bench.py`` that needs no GPU: the algorithmic byte count of a call,
the kernel launches a step claims, and the lookup of recorded DRAM traffic (which must
refuse a figure once the kernel's sources have changed)."""
import importlib.util
import json
import os
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_attended_count_follows_the_window_and_the_queries(bench):
    # sliding window of 1024: the last min(1024, L) positions
    assert bench.attended_count(2048, 1024) == 1024
    assert bench.attended_count(1024, 1024) == 1024
    assert bench.attended_count(500, 1024) == 500
    assert bench.attended_count(0, 1024) == 0
    # T queries at L - T .. L - 1: the union of their windows spans W + T - 1 positions
    assert bench.attended_count(2048, 1024, T=8) == 1031
    assert bench.attended_count(5, 1024, T=8) == 5
    # full history
    assert bench.attended_count(8192, 0) == 8192
    assert bench.attended_count(8192, 0, T=4) == 8192


def test_kv_bytes_is_two_tensors_of_kvh_rows(bench):
    sliding = {"KVH": 16, "D": 256, "window": 1024}
    glob = {"KVH": 4, "D": 512, "window": 0}
    lens = np.array([2048, 10, 0])
    assert bench.kv_bytes(lens, sliding) == (1024 + 10) * 16 * 256 * 2 * 2
    assert bench.kv_bytes(lens, glob) == (2048 + 10) * 4 * 512 * 2 * 2
    # 16,384 B per attended position sliding, 8,192 B global
    assert bench.kv_bytes(np.array([1]), sliding) == 16384
    assert bench.kv_bytes(np.array([1]), glob) == 8192


def fake_call(bench, layer, **kw):
    from decode_attention_gb300 import inputs
    geo = inputs.geometry(layer)
    case = {"v": types.SimpleNamespace(shape=(8, 131072, geo["KVH"], geo["D"]))}
    return bench.Call(layer, geo, case, False, np.array([100] * 8), device="cpu", **kw)


def test_launches_per_call(bench):
    class FakeLib:
        GQA_KERNEL_TCGEN05 = 2

        def __init__(self, choice):
            self.choice = choice

        def gqa_decode_keqv_kernel(self, *args):
            return self.choice

    lib = FakeLib(2)
    # slidingDecodeGQA merges split segments in its one kernel
    assert bench.launches_per_call(lib, fake_call(bench, "sliding")) == 1
    # decodeGQA: main and combine kernels
    assert bench.launches_per_call(lib, fake_call(bench, "global")) == 2
    # multi-query: the tcgen05 kernel and the combine
    assert bench.launches_per_call(lib, fake_call(bench, "sliding", queries=8)) == 2
    # K=V on the tcgen05 kernel: the scores-operand kernel first
    assert bench.launches_per_call(lib, fake_call(bench, "global", keqv=True)) == 3
    # K=V on the mma.sync kernel (a small cache)
    assert bench.launches_per_call(FakeLib(1), fake_call(bench, "global", keqv=True)) == 2
    # the producer ahead of a decode call
    assert bench.launches_per_call(lib, fake_call(bench, "sliding", ring=1024, raw={})) == 1


def test_recorded_traffic_is_refused_once_the_kernel_changes(bench, tmp_path, monkeypatch):
    rec = {"wl": {"global": {"kernel": "gqa_decode_kernel", "dram_bytes_per_launch": 123,
                             "kernel_source_hash": bench.kernel_source_hash("gqa_decode_kernel")}},
           "old": {"global": {"kernel": "gqa_decode_kernel", "dram_bytes_per_launch": 456,
                              "kernel_source_hash": "0000000000000000"}}}
    (tmp_path / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.recorded_traffic("wl", "global", "gqa_decode_kernel") == 123
    assert bench.recorded_traffic("old", "global", "gqa_decode_kernel") is None
    # the figure belongs to one kernel
    assert bench.recorded_traffic("wl", "global", "gqa_mq_kernel") is None
    assert bench.recorded_traffic("wl", "sliding", "gqa_decode_kernel") is None
    assert bench.recorded_traffic("missing", "global", "gqa_decode_kernel") is None


def test_committed_traffic_entries_name_existing_summaries(bench):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for workload, layers in rec.items():
        if workload.startswith("_"):
            continue
        for layer, e in layers.items():
            assert e["kernel"] in bench.KERNEL_SOURCES, (workload, layer)
            assert os.path.exists(os.path.join(ROOT, "profiles", e["capture"])), (workload, layer)
            assert e["dram_bytes_per_launch"] > 0


def test_both_arms_print_the_same_config(bench):
    from decode_attention_gb300 import inputs
    wl = inputs.WORKLOADS[bench.DEFAULT_WORKLOAD]
    cfg = bench.workload_config(wl)
    assert cfg["workload"] == "paged_mixed_b256"
    assert cfg["l2"] == bench.L2_POLICY
    json.dumps(cfg)   # plain JSON
