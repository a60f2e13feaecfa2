"""The geometry constants used by the input generators match the values the
Model Spec prints (fixture ``tests/golden/geometry.json``, each entry cited)."""
import json
import os

from decode_attention_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "geometry.json")


def load():
    with open(GOLDEN) as f:
        return json.load(f)


def test_sliding_geometry():
    g = load()["slidingDecodeGQA"]
    assert inputs.SLIDING == dict(H=g["heads"], KVH=g["kv_heads"], D=g["head_dim"], window=g["window"])


def test_global_geometry():
    g = load()["decodeGQA"]
    assert g["window"] is None
    assert inputs.GLOBAL == dict(H=g["heads"], KVH=g["kv_heads"], D=g["head_dim"], window=0)


def test_page_size_and_domain():
    g = load()
    assert inputs.PAGE_SIZE == g["page_size"]
    lo, hi = g["shape_domain"]["B"]
    for w in inputs.WORKLOADS.values():
        assert lo <= w.B <= hi
        lens = w.seq_lens()
        assert lens.min() >= 1 and lens.max() <= g["shape_domain"]["S"][1]
