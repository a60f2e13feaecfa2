"""Full-size parity: the benchmark workloads at their stated sizes, built and
launched exactly as bench.py builds and launches them, with sampled sequences
checked against the fp64 oracle (the oracle computes each sampled sequence from
its attended K/V rows copied to the host)."""
import numpy as np
import pytest
import torch

import bench
from decode_attention_gb300 import inputs
from tests.helpers import assert_parity

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import decode_attention_gb300 as gqa  # noqa: E402

WORKLOADS = ["sliding_b1_s2048", "global_b8_s8192", "sliding_b64_s32768",
             "global_b16_s131072", "paged_mixed_b256", "retrofit_block_b64",
             "global_keqv_b16_s131072", "global_keqv_b8_s8192", "global_mq4_b16_s131072",
             "sliding_mq8_b64_s32768",
             "global_mq4_b8_s8192"]


def sampled(lens, k=3, seed=0):
    """First, last and a few random sequences with a non-empty range."""
    idx = [i for i, L in enumerate(lens) if L > 0]
    rng = np.random.default_rng(seed)
    pick = {idx[0], idx[-1]} | set(rng.choice(idx, size=min(k, len(idx)), replace=False).tolist())
    return sorted(pick)


def sampled_paged(lens, seed=0, at_least=16):
    """At least 16 sequences of a paged batch: the four longest (the global call gives
    them dynamic chunks), four whose sliding window starts inside a page (L > 1024,
    L % 16 != 0), the two shortest, two more with L % 16 != 0 below the window, the
    first and last, and random ones up to the count."""
    lens = np.asarray(lens)
    idx = np.arange(len(lens))
    order = np.argsort(-lens, kind="stable")
    pick = set(order[:4].tolist()) | set(order[-2:].tolist()) | {0, len(lens) - 1}
    mid_page = idx[(lens > 1024) & (lens % 16 != 0)]
    short_ragged = idx[(lens <= 1024) & (lens % 16 != 0)]
    rng = np.random.default_rng(seed)
    for group, n in ((mid_page, 4), (short_ragged, 2)):
        pick |= set(rng.choice(group, size=min(n, len(group)), replace=False).tolist())
    rest = [i for i in idx.tolist() if i not in pick]
    need = max(0, at_least - len(pick))
    pick |= set(rng.choice(rest, size=min(need, len(rest)), replace=False).tolist())
    return sorted(int(i) for i in pick if lens[i] > 0)


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_sampled_parity(name):
    wl = inputs.WORKLOADS[name]
    calls, lens = bench.build_calls(wl, wl.seed)
    for c in calls:
        c.out = torch.empty_like(c.out, dtype=torch.float32)
        c.launch(gqa)
        out32 = c.out.clone()
        c.out = torch.empty_like(out32, dtype=torch.bfloat16)
        c.launch(gqa)
        out16 = c.out.clone()
        torch.cuda.synchronize()
        assert gqa.gqa_device_status() == 0
        assert torch.equal(out16, out32.to(torch.bfloat16))
        picks = sampled_paged(lens, seed=wl.seed) if wl.paged else sampled(lens, seed=wl.seed)
        if wl.paged:
            assert len(picks) >= 16
        for b in picks:
            slices = bench.host_slices(c, b)
            ref = bench.oracle_for(c, slices)
            assert_parity(out32[b], ref, f"{name}/{c.name} b={b} L={slices[3]}")
        # sequences with nothing to attend are exact zeros
        for b, L in enumerate(lens):
            if L == 0:
                assert torch.all(out32[b] == 0)
    del calls
    torch.cuda.empty_cache()
