"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties the oracle to a closed form, an invariant of the definition, an
independent brute-force formulation, or a library routine (torch SDPA in
float64).  Chosen so that a plausible slip in the oracle -- a wrong window
bound, a wrong head mapping, a 1/sqrt(D) scale, a missing max subtraction,
swapped k/v, a k row paired with the wrong v row, a wrong page index -- fails at
least one of them.

Definition pinned (gemma-4-31B Model Spec, "Compute-graph nodes", the two
``attn.core`` rows; masks and append-before-attend from the "Gemma 4 31B-it
Text Architecture" page, "Compact form").
"""
import math

import numpy as np
import pytest
import torch

pytestmark = []

RNG = np.random.default_rng(12345)


def to_bits(x) -> np.ndarray:
    """Round float values to bf16 (RNE) and return the bit patterns."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_vals(bits: np.ndarray) -> np.ndarray:
    """Exact real values (float64) of bf16 bit patterns."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def exact_bits(x) -> np.ndarray:
    """Bits of values that must be exactly representable in bf16."""
    b = to_bits(x)
    assert np.array_equal(to_vals(b), np.asarray(x, dtype=np.float64)), "value not bf16-exact"
    return b


def random_case(B, S, H, KVH, D, seed=0):
    rng = np.random.default_rng(seed)
    q = to_bits(rng.standard_normal((B, H, D)))
    k = to_bits(rng.standard_normal((B, S, KVH, D)))
    v = to_bits(rng.standard_normal((B, S, KVH, D)))
    return q, k, v


def window_range(L, W):
    return (max(0, L - W) if W > 0 else 0), L


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("window", [0, 8])
def test_constant_values_give_that_value(oracle_lib, window):
    """If v[b, s, kvh] is the same vector c for every s, o[b, h] = c[h // g]."""
    B, S, H, KVH, D = 3, 37, 8, 2, 16
    q, k, _ = random_case(B, S, H, KVH, D, seed=1)
    c = to_bits(RNG.standard_normal((B, KVH, D)))
    v = np.broadcast_to(c[:, None, :, :], (B, S, KVH, D)).copy()
    lens = [37, 5, 1]
    out = oracle_lib.gqa_decode_f64(q, k, v, lens, window)
    g = H // KVH
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(out[b, h], to_vals(c[b, h // g]), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("window", [0, 1, 1024])
def test_length_one_returns_first_value(oracle_lib, window):
    """One attended key has weight exactly 1: o[b, h] = v[b, 0, h // g]."""
    B, S, H, KVH, D = 2, 4, 32, 4, 32
    q, k, v = random_case(B, S, H, KVH, D, seed=2)
    out = oracle_lib.gqa_decode_f64(q, k, v, [1, 1], window)
    g = H // KVH
    for b in range(B):
        for h in range(H):
            assert np.array_equal(out[b, h], to_vals(v[b, 0, h // g]))


@pytest.mark.parametrize("L,W", [(1, 0), (5, 0), (10, 4), (37, 16), (16, 16), (17, 16), (3, 16)])
def test_zero_query_gives_window_mean(oracle_lib, L, W):
    """q = 0 makes every score 0, so o is the plain mean of v over the attended range."""
    B, S, H, KVH, D = 1, 40, 4, 2, 8
    _, k, v = random_case(B, S, H, KVH, D, seed=3)
    q = np.zeros((B, H, D), dtype=np.uint16)
    out = oracle_lib.gqa_decode_f64(q, k, v, [L], W)
    lo, hi = window_range(L, W)
    vv = to_vals(v)
    for h in range(H):
        expect = vv[0, lo:hi, h // (H // KVH)].mean(axis=0)
        np.testing.assert_allclose(out[0, h], expect, rtol=1e-13, atol=1e-15)


def test_two_keys_logistic_closed_form_scale_one(oracle_lib):
    """Two keys: o = v0 + (v1 - v0) * sigmoid(s1 - s0) with s_j = <q, k_j> (scale 1).

    Scores are built from one-hot vectors so they are known without a dot
    product: q = a e_0, k_j = x_j e_0, so s_j = a x_j exactly.
    """
    D, H, KVH = 8, 2, 1
    a, x0, x1 = 1.5, 0.25, 2.0
    q = np.zeros((1, H, D)); q[0, :, 0] = a
    k = np.zeros((1, 2, KVH, D)); k[0, 0, 0, 0] = x0; k[0, 1, 0, 0] = x1
    v = RNG.standard_normal((1, 2, KVH, D))
    qb, kb, vb = exact_bits(q), exact_bits(k), to_bits(v)
    out = oracle_lib.gqa_decode_f64(qb, kb, vb, [2], 0)
    vv = to_vals(vb)
    sig = 1.0 / (1.0 + math.exp(-(a * x1 - a * x0)))
    expect = vv[0, 0, 0] + (vv[0, 1, 0] - vv[0, 0, 0]) * sig
    for h in range(H):
        np.testing.assert_allclose(out[0, h], expect, rtol=1e-14, atol=1e-15)
    # a 1/sqrt(D) scale would give a visibly different weight
    sig_scaled = 1.0 / (1.0 + math.exp(-(a * x1 - a * x0) / math.sqrt(D)))
    assert abs(sig - sig_scaled) > 0.1


def test_huge_logits_do_not_overflow(oracle_lib):
    """Scores of +-1024: without subtracting the max, exp overflows to inf/NaN.

    Head 0 (q = +1024 e_0) must return v at the one key equal to e_0; head 1
    (q = -1024 e_0) gives that key weight exp(-1024) = 0 in double, so o is the
    mean of the other values.
    """
    D, H, KVH, L, j = 8, 2, 1, 9, 4
    q = np.zeros((1, H, D)); q[0, 0, 0] = 1024.0; q[0, 1, 0] = -1024.0
    k = np.zeros((1, L, KVH, D)); k[0, j, 0, 0] = 1.0
    vb = to_bits(RNG.standard_normal((1, L, KVH, D)))
    out = oracle_lib.gqa_decode_f64(exact_bits(q), exact_bits(k), vb, [L], 0)
    vv = to_vals(vb)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out[0, 0], vv[0, j, 0])
    others = np.delete(vv[0, :, 0], j, axis=0).mean(axis=0)
    np.testing.assert_allclose(out[0, 1], others, rtol=1e-13, atol=1e-15)


def test_empty_range_is_zero(oracle_lib):
    """L_b = 0: the empty sum, o = 0 (never NaN)."""
    q, k, v = random_case(3, 8, 8, 4, 16, seed=4)
    out = oracle_lib.gqa_decode_f64(q, k, v, [0, 3, 0], 0)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[1])) and np.any(out[1] != 0)


def test_empty_batch(oracle_lib):
    q = np.zeros((0, 8, 16), np.uint16)
    k = np.zeros((0, 4, 4, 16), np.uint16)
    out = oracle_lib.gqa_decode_f64(q, k, k, np.zeros(0, np.int32), 0)
    assert out.shape == (0, 8, 16)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,KVH", [(32, 16), (32, 4)])
def test_gqa_head_mapping(oracle_lib, H, KVH):
    """Changing KV head kvh changes exactly the query heads h with h // g == kvh."""
    B, S, D = 2, 12, 16
    g = H // KVH
    q, k, v = random_case(B, S, H, KVH, D, seed=5)
    base = oracle_lib.gqa_decode_f64(q, k, v, [12, 7], 0)
    for kvh in [0, KVH // 2, KVH - 1]:
        k2, v2 = k.copy(), v.copy()
        k2[0, :, kvh] = to_bits(RNG.standard_normal((S, D)))
        v2[0, :, kvh] = to_bits(RNG.standard_normal((S, D)))
        out = oracle_lib.gqa_decode_f64(q, k2, v2, [12, 7], 0)
        changed = {h for h in range(H) if not np.array_equal(out[0, h], base[0, h])}
        assert changed == {h for h in range(H) if h // g == kvh}
        assert np.array_equal(out[1], base[1])


def test_window_at_least_length_equals_full(oracle_lib):
    """Any window >= L reads every position, so it equals the full-history result."""
    B, S, H, KVH, D = 3, 50, 8, 2, 16
    q, k, v = random_case(B, S, H, KVH, D, seed=6)
    lens = [50, 20, 1]
    full = oracle_lib.gqa_decode_f64(q, k, v, lens, 0)
    for W in [50, 64, 1024]:
        assert np.array_equal(oracle_lib.gqa_decode_f64(q, k, v, lens, W), full)
    assert not np.array_equal(oracle_lib.gqa_decode_f64(q, k, v, lens, 49)[0], full[0])


@pytest.mark.parametrize("L,W", [(50, 16), (17, 16), (16, 16), (1030, 1024), (1025, 1024)])
def test_window_equals_full_on_the_last_positions(oracle_lib, L, W):
    """Sliding over [L-W, L) equals full attention over a cache holding only those rows."""
    S, H, KVH, D = L, 4, 2, 8
    q, k, v = random_case(1, S, H, KVH, D, seed=7)
    sliding = oracle_lib.gqa_decode_f64(q, k, v, [L], W)
    lo = max(0, L - W)
    sliced = oracle_lib.gqa_decode_f64(q, k[:, lo:].copy(), v[:, lo:].copy(), [L - lo], 0)
    assert np.array_equal(sliding, sliced)
    # the same rows addressed through pos_base
    based = oracle_lib.gqa_decode_f64(q, k[:, lo:].copy(), v[:, lo:].copy(), [L], W, pos_base=lo)
    assert np.array_equal(sliding, based)


def test_output_is_a_convex_combination(oracle_lib):
    """Each coordinate of o lies between the min and max of v over the attended rows."""
    B, S, H, KVH, D = 4, 30, 8, 4, 16
    q, k, v = random_case(B, S, H, KVH, D, seed=8)
    lens, W = [30, 12, 5, 29], 10
    out = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    vv = to_vals(v)
    for b, L in enumerate(lens):
        lo, hi = window_range(L, W)
        for h in range(H):
            rows = vv[b, lo:hi, h // (H // KVH)]
            assert np.all(out[b, h] >= rows.min(axis=0) - 1e-12)
            assert np.all(out[b, h] <= rows.max(axis=0) + 1e-12)


def test_permuting_positions_consistently_changes_nothing(oracle_lib):
    """Softmax attention is a function of the set of (k, v) pairs: reordering them
    (the same permutation for k and v) leaves o unchanged up to rounding, and
    pairing keys with other rows' values does not."""
    S, H, KVH, D = 24, 8, 2, 16
    q, k, v = random_case(1, S, H, KVH, D, seed=9)
    base = oracle_lib.gqa_decode_f64(q, k, v, [S], 0)
    perm = np.random.default_rng(1).permutation(S)
    out = oracle_lib.gqa_decode_f64(q, k[:, perm].copy(), v[:, perm].copy(), [S], 0)
    np.testing.assert_allclose(out, base, rtol=1e-12, atol=1e-14)
    mismatched = oracle_lib.gqa_decode_f64(q, k, v[:, perm].copy(), [S], 0)
    assert np.max(np.abs(mismatched - base)) > 1e-3


def test_keys_and_values_play_different_roles(oracle_lib):
    """Swapping the k and v tensors changes the result (they are not interchangeable)."""
    q, k, v = random_case(1, 20, 4, 2, 8, seed=10)
    a = oracle_lib.gqa_decode_f64(q, k, v, [20], 0)
    b = oracle_lib.gqa_decode_f64(q, v, k, [20], 0)
    assert np.max(np.abs(a - b)) > 1e-3


# ---------------------------------------------------------------------------
# independent formulations
# ---------------------------------------------------------------------------

def brute_force(q, k, v, lens, W):
    """Explicit [H, S] score matrix with a boolean mask built from the query position
    t = L - 1 (causal s <= t, and t - W < s for a window), softmax over the
    masked row with scipy, then a matrix product with repeat-expanded V."""
    from scipy.special import softmax
    qv, kv, vv = to_vals(q), to_vals(k), to_vals(v)
    B, H, D = qv.shape
    _, S, KVH, _ = kv.shape
    g = H // KVH
    out = np.zeros((B, H, D))
    for b in range(B):
        t = lens[b] - 1
        s = np.arange(S)
        mask = s <= t
        if W > 0:
            mask &= s > t - W
        k_rep = np.repeat(kv[b], g, axis=1)  # [S, H, D]: head h reads kv head h // g
        v_rep = np.repeat(vv[b], g, axis=1)
        scores = np.einsum("hd,shd->hs", qv[b], k_rep)
        scores[:, ~mask] = -np.inf
        p = softmax(scores, axis=-1)
        out[b] = np.einsum("hs,shd->hd", p, v_rep)
    return out


@pytest.mark.parametrize("H,KVH,D,W", [(32, 16, 8, 0), (32, 16, 16, 5), (32, 4, 8, 0),
                                       (32, 4, 16, 7), (32, 16, 256, 1024), (32, 4, 512, 0)])
def test_brute_force_explicit_mask(oracle_lib, H, KVH, D, W):
    B, S = 3, 40
    q, k, v = random_case(B, S, H, KVH, D, seed=11 + D + W)
    lens = [40, 13, 1]
    out = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    ref = brute_force(q, k, v, lens, W)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def test_brute_force_window_edges(oracle_lib):
    """Lengths around the 1024 window: 1023, 1024, 1025, 1040 (tiny D)."""
    B, S, H, KVH, D, W = 4, 1040, 4, 2, 8, 1024
    q, k, v = random_case(B, S, H, KVH, D, seed=12)
    # make the positions just outside the window stand out so an off-by-one shows
    k[:, :, :, :] = to_bits(to_vals(k) * 0.5)
    lens = [1023, 1024, 1025, 1040]
    out = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    ref = brute_force(q, k, v, lens, W)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    # and a window shifted by one position is detectably different
    for b, L in enumerate(lens[2:], start=2):
        off_by_one = oracle_lib.gqa_decode_f64(q, k, v, lens, W + 1)
        assert np.max(np.abs(off_by_one[b] - out[b])) > 1e-6


@pytest.mark.parametrize("H,KVH,W", [(32, 16, 1024), (32, 4, 0), (32, 16, 6)])
def test_torch_sdpa_float64(oracle_lib, H, KVH, W):
    """torch.nn.functional.scaled_dot_product_attention in float64 on CPU, scale=1,
    with a boolean mask and K/V expanded to the query heads."""
    B, S, D = 3, 33, 32
    q, k, v = random_case(B, S, H, KVH, D, seed=13)
    lens = [33, 20, 2]
    out = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    g = H // KVH
    qt = torch.from_numpy(to_vals(q))[:, :, None, :]                      # [B, H, 1, D]
    kt = torch.from_numpy(to_vals(k)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(to_vals(v)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    pos = torch.arange(S)
    mask = torch.zeros(B, 1, 1, S, dtype=torch.bool)
    for b, L in enumerate(lens):
        lo, hi = window_range(L, W)
        mask[b, 0, 0] = (pos >= lo) & (pos < hi)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0)
    np.testing.assert_allclose(out, ref[:, :, 0, :].numpy(), rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------------------
# paged indexing
# ---------------------------------------------------------------------------

def scatter_to_pages(k, v, lens, page_size=16, spare=3, seed=0):
    """Copy each sequence's rows into randomly numbered pages; return pools + table."""
    B, S, KVH, D = k.shape
    need = [(L + page_size - 1) // page_size for L in lens]
    P = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(P)
    max_pages = max(1, (S + page_size - 1) // page_size)
    bt = np.full((B, max_pages), -1, np.int32)
    kp = np.full((P, page_size, KVH, D), 0x7FC0, np.uint16)   # bf16 NaN everywhere unused
    vp = np.full((P, page_size, KVH, D), 0x7FC0, np.uint16)
    off = 0
    for b, L in enumerate(lens):
        for j in range(need[b]):
            page = perm[off]
            off += 1
            bt[b, j] = page
            n = min(page_size, L - j * page_size)
            kp[page, :n] = k[b, j * page_size:j * page_size + n]
            vp[page, :n] = v[b, j * page_size:j * page_size + n]
    return kp, vp, bt


@pytest.mark.parametrize("H,KVH,D,W", [(32, 16, 16, 0), (32, 16, 16, 20), (32, 4, 32, 0)])
def test_paged_equals_contiguous(oracle_lib, H, KVH, D, W):
    """A permuted page table holding the same rows gives the identical result, and
    NaN in every slot no attended position maps to changes nothing."""
    B, S = 4, 70
    q, k, v = random_case(B, S, H, KVH, D, seed=14)
    lens = [70, 33, 16, 1]
    kp, vp, bt = scatter_to_pages(k, v, lens)
    paged = oracle_lib.gqa_decode_paged_f64(q, kp, vp, bt, lens, W)
    contig = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    assert np.array_equal(paged, contig)


def test_paged_bad_page_id_gives_nan_for_that_sequence(oracle_lib):
    B, S, H, KVH, D = 3, 40, 8, 2, 16
    q, k, v = random_case(B, S, H, KVH, D, seed=15)
    lens = [40, 40, 40]
    kp, vp, bt = scatter_to_pages(k, v, lens)
    bt[1, 1] = kp.shape[0] + 5
    out = oracle_lib.gqa_decode_paged_f64(q, kp, vp, bt, lens, 0)
    assert np.all(np.isnan(out[1]))
    assert np.all(np.isfinite(out[0])) and np.all(np.isfinite(out[2]))
    # a bad id on a page the window never reaches is never looked at
    bt2 = bt.copy(); bt2[1, 1] = bt[0, 1]
    bt2[2, 0] = -7
    out2 = oracle_lib.gqa_decode_paged_f64(q, kp, vp, bt2, lens, 16)
    assert np.all(np.isfinite(out2))


# ---------------------------------------------------------------------------
# window-capped ring-buffer cache ("Retrofit Plan: Gemma 4 31B IT -> Progressive
# Multi-Scale SWA with Block Attention Residuals", §3.3 and §7.3): position s at
# row s mod C
# ---------------------------------------------------------------------------

def ring_copy(t, lens, C, keep):
    """Ring of C rows per sequence holding positions [L - keep, L) of the
    contiguous tensor t at rows s mod C; every other row is bf16 NaN."""
    B, S, KVH, D = t.shape
    r = np.full((B, C, KVH, D), 0x7FC0, np.uint16)
    for b, L in enumerate(lens):
        for s in range(max(0, L - keep), L):
            r[b, s % C] = t[b, s]
    return r


@pytest.mark.parametrize("C,W", [(16, 16), (24, 16), (16, 5), (7, 7)])
def test_ring_equals_contiguous_on_a_wrapped_copy(oracle_lib, C, W):
    """A ring holding the same rows at s mod C gives the identical result, with NaN in
    every row outside the window: lengths below, at and across multiples of C."""
    lens = [1, W - 1 if W > 1 else 1, W, C, C + 1, 2 * C + 3, 3 * C, 5 * C - 1]
    S = max(lens)
    H, KVH, D = 8, 2, 16
    q, k, v = random_case(len(lens), S, H, KVH, D, seed=17 + C + W)
    rk, rv = ring_copy(k, lens, C, W), ring_copy(v, lens, C, W)
    ring = oracle_lib.gqa_decode_ring_f64(q, rk, rv, lens, W)
    contig = oracle_lib.gqa_decode_f64(q, k, v, lens, W)
    assert np.array_equal(ring, contig)


@pytest.mark.parametrize("H,KVH", [(32, 16), (32, 4)])
def test_ring_torch_sdpa_float64(oracle_lib, H, KVH):
    """SDPA in float64 on the rows a ring holds for the window, gathered by
    position (row s mod C), against random ring contents."""
    B, C, D, W = 3, 12, 16, 9
    q, rk, rv = random_case(B, C, H, KVH, D, seed=18)
    lens = [5, 12, 31]
    out = oracle_lib.gqa_decode_ring_f64(q, rk, rv, lens, W)
    g = H // KVH
    for b, L in enumerate(lens):
        lo, hi = window_range(L, W)
        rows = [s % C for s in range(lo, hi)]
        qt = torch.from_numpy(to_vals(q[b]))[:, None, :]                             # [H, 1, D]
        kt = torch.from_numpy(to_vals(rk[b, rows])).permute(1, 0, 2).repeat_interleave(g, dim=0)
        vt = torch.from_numpy(to_vals(rv[b, rows])).permute(1, 0, 2).repeat_interleave(g, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1.0)
        np.testing.assert_allclose(out[b], ref[:, 0, :].numpy(), rtol=1e-11, atol=1e-13)


def test_ring_rejects_windows_it_cannot_hold(oracle_lib):
    q, k, v = random_case(1, 8, 4, 2, 8, seed=19)
    for W in (0, 9):
        with pytest.raises(ValueError):
            oracle_lib.gqa_decode_ring_f64(q, k, v, [20], W)


# ---------------------------------------------------------------------------
# single K=V global cache: the key of cached value row v at position s is
# rope(w_k * v, s) (Model Spec "What to watch for" and `attn.rope` row; decoder
# listing of the "Gemma 4 31B-it Text Architecture" page)
# ---------------------------------------------------------------------------

def complex_rope_keys(v_vals, w_vals, positions, n_rot, theta):
    """Keys through a different route: each rotated pair (i, i + D/2) as the complex
    number x_i + j x_{i+D/2}, multiplied by exp(j * s * theta^(-2i/D))."""
    x = v_vals * w_vals                                   # [S, ..., D]
    D = x.shape[-1]
    half = D // 2
    z = x[..., :n_rot] + 1j * x[..., half:half + n_rot]
    freq = theta ** (-2.0 * np.arange(n_rot) / D)
    pos = np.asarray(positions, dtype=np.float64).reshape(-1, 1, 1)   # the [S, KVH, pair] axes
    z = z * np.exp(1j * pos * freq)
    k = x.copy()
    k[..., :n_rot] = z.real
    k[..., half:half + n_rot] = z.imag
    return k


@pytest.mark.parametrize("H,KVH,D,n_rot,theta,W", [(8, 2, 16, 3, 100.0, 0), (8, 2, 16, 8, 10.0, 5),
                                                   (32, 4, 64, 8, 1.0e6, 0)])
def test_keqv_complex_rope_and_sdpa(oracle_lib, H, KVH, D, n_rot, theta, W):
    B, S = 3, 37
    q, _, v = random_case(B, S, H, KVH, D, seed=20 + D + n_rot)
    w = to_bits(1.0 + 0.25 * np.random.default_rng(21).standard_normal(D))
    lens = [37, 20, 1]
    out = oracle_lib.gqa_decode_keqv_f64(q, v, w, lens, W, n_rot=n_rot, theta=theta)
    g = H // KVH
    k64 = complex_rope_keys(to_vals(v), to_vals(w), np.arange(S), n_rot, theta)   # [B, S, KVH, D]
    qt = torch.from_numpy(to_vals(q))[:, :, None, :]
    kt = torch.from_numpy(k64).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(to_vals(v)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    pos = torch.arange(S)
    mask = torch.zeros(B, 1, 1, S, dtype=torch.bool)
    for b, L in enumerate(lens):
        lo, hi = window_range(L, W)
        mask[b, 0, 0] = (pos >= lo) & (pos < hi)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0)
    np.testing.assert_allclose(out, ref[:, :, 0, :].numpy(), rtol=1e-10, atol=1e-12)


def test_keqv_global_geometry_long_positions(oracle_lib):
    """D = 512, 64 rotated pairs, theta = 1e6, keys at positions just below 131075
    (a 40-position window): the complex route again, on the rows of one sequence."""
    H, KVH, D, S = 32, 4, 512, 131080
    L, n = 131075, 40
    rng = np.random.default_rng(22)
    q = to_bits(rng.standard_normal((1, H, D)))
    v = np.zeros((1, S, KVH, D), np.uint16)
    v[0, L - n:L] = to_bits(rng.standard_normal((n, KVH, D)) * 0.3)
    w = to_bits(1.0 + 0.25 * rng.standard_normal(D))
    out = oracle_lib.gqa_decode_keqv_f64(q, v, w, [L], n)
    k_tail = complex_rope_keys(to_vals(v[0, L - n:L]), to_vals(w), np.arange(L - n, L), 64, 1.0e6)
    g = H // KVH
    qt = torch.from_numpy(to_vals(q[0]))[:, None, :]                                   # [H, 1, D]
    kt = torch.from_numpy(k_tail).permute(1, 0, 2).repeat_interleave(g, dim=0)          # [H, n, D]
    vt = torch.from_numpy(to_vals(v[0, L - n:L])).permute(1, 0, 2).repeat_interleave(g, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1.0)
    np.testing.assert_allclose(out[0], ref[:, 0, :].numpy(), rtol=1e-9, atol=1e-12)


def test_keqv_unrotated_dims_equal_plain_keys(oracle_lib):
    """Values that live on unrotated coordinates only, with power-of-two weights
    (so w * v is exact in bf16): identical to the plain oracle with k = w * v."""
    B, S, H, KVH, D, n_rot = 2, 30, 8, 2, 16, 3
    q, _, v = random_case(B, S, H, KVH, D, seed=23)
    rot = list(range(n_rot)) + list(range(D // 2, D // 2 + n_rot))
    v[..., rot] = 0
    w_vals = np.array([2.0 ** ((i % 5) - 2) for i in range(D)])
    w = exact_bits(w_vals)
    k = exact_bits(to_vals(v) * w_vals)
    lens = [30, 11]
    keqv = oracle_lib.gqa_decode_keqv_f64(q, v, w, lens, 0, n_rot=n_rot, theta=1e4)
    plain = oracle_lib.gqa_decode_f64(q, k, v, lens, 0)
    assert np.array_equal(keqv, plain)


# ---------------------------------------------------------------------------
# decode-step producer: q = rope(q_norm(q_raw)), k = rope(k_norm(k_raw)),
# v = v_norm(v_raw) at position L - 1 (Model Spec rows attn.qk_norm, attn.v_norm,
# attn.rope; decoder listing of the architecture page)
# ---------------------------------------------------------------------------

PRODUCER_GEOMS = [(32, 16, 256, 128, 1.0e4), (32, 4, 512, 64, 1.0e6), (4, 2, 16, 3, 50.0)]


def producer_case(B, H, KVH, D, seed):
    rng = np.random.default_rng(seed)
    scale = rng.uniform(0.2, 5.0, size=(B, H, 1))       # raw projections: arbitrary scales
    q = to_bits(rng.standard_normal((B, H, D)) * scale)
    k = to_bits(rng.standard_normal((B, KVH, D)) * scale[:, :KVH])
    v = to_bits(rng.standard_normal((B, KVH, D)) * 2.0)
    w_q = to_bits(1.0 + 0.25 * rng.standard_normal(D))
    w_k = to_bits(1.0 + 0.25 * rng.standard_normal(D))
    return q, k, v, w_q, w_k


def test_producer_constant_heads_closed_form(oracle_lib):
    """At position 0 (L = 1) nothing rotates: a head of constant c normalises to
    c / sqrt(c^2 + 1e-6), times the weight for q and k."""
    H, KVH, D = 4, 2, 8
    c = np.array([0.5, -2.0, 3.0, 1.0])
    q = exact_bits(np.broadcast_to(c[None, :, None], (1, H, D)))
    k = exact_bits(np.broadcast_to(c[None, :KVH, None], (1, KVH, D)))
    w = exact_bits(np.array([1.0, 2.0, 0.5, 1.5, 1.0, 0.25, 4.0, 1.0]))
    qo, ko, vo = oracle_lib.prepare_decode_f64(q, k, k, w, w, [1], 3, 10.0)
    f = c / np.sqrt(c * c + 1e-6)
    np.testing.assert_allclose(qo[0], f[:, None] * to_vals(w)[None, :], rtol=1e-14)
    np.testing.assert_allclose(ko[0], f[:KVH, None] * to_vals(w)[None, :], rtol=1e-14)
    np.testing.assert_allclose(vo[0], np.broadcast_to(f[:KVH, None], (KVH, D)), rtol=1e-14)


@pytest.mark.parametrize("H,KVH,D,n_rot,theta", PRODUCER_GEOMS)
def test_producer_torch_rms_norm_and_complex_rope(oracle_lib, H, KVH, D, n_rot, theta):
    """torch's rms_norm in float64, then the complex-exponential rotation."""
    B = 3
    q, k, v, w_q, w_k = producer_case(B, H, KVH, D, seed=30 + D)
    lens = [1, 77, 131075]
    qo, ko, vo = oracle_lib.prepare_decode_f64(q, k, v, w_q, w_k, lens, n_rot, theta)
    F = torch.nn.functional
    qn = F.rms_norm(torch.from_numpy(to_vals(q)), (D,), torch.from_numpy(to_vals(w_q)), 1e-6).numpy()
    kn = F.rms_norm(torch.from_numpy(to_vals(k)), (D,), torch.from_numpy(to_vals(w_k)), 1e-6).numpy()
    vn = F.rms_norm(torch.from_numpy(to_vals(v)), (D,), None, 1e-6).numpy()
    ones = np.ones(D)
    for b, L in enumerate(lens):
        # at position ~1.3e5 the fp64 angle itself carries ~1e-11 rad of rounding
        q_ref = complex_rope_keys(qn[b][None], ones, [L - 1], n_rot, theta)[0]
        k_ref = complex_rope_keys(kn[b][None], ones, [L - 1], n_rot, theta)[0]
        np.testing.assert_allclose(qo[b], q_ref, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(ko[b], k_ref, rtol=1e-9, atol=1e-9)
        np.testing.assert_allclose(vo[b], vn[b], rtol=1e-13, atol=1e-15)


def test_producer_rotation_keeps_same_position_dot_products(oracle_lib):
    """q and k of one token share the position, and the rotation is orthogonal:
    <q, k> per query head and its KV head does not depend on the position."""
    H, KVH, D = 32, 4, 512
    q, k, v, w_q, w_k = producer_case(1, H, KVH, D, seed=31)
    ref_q, ref_k, _ = oracle_lib.prepare_decode_f64(q, k, v, w_q, w_k, [1], 64, 1.0e6)
    ref = np.einsum("hd,hd->h", ref_q[0], np.repeat(ref_k[0], H // KVH, axis=0))
    for L in (2, 1000, 65537, 262144):
        q2 = np.repeat(q, 1, axis=0)
        qo, ko, _ = oracle_lib.prepare_decode_f64(q2, k, v, w_q, w_k, [L], 64, 1.0e6)
        dots = np.einsum("hd,hd->h", qo[0], np.repeat(ko[0], H // KVH, axis=0))
        np.testing.assert_allclose(dots, ref, rtol=1e-9, atol=1e-9)
        assert np.max(np.abs(qo[0] - ref_q[0])) > 1e-3   # and the vectors did move


def test_producer_values_equal_keys_form(oracle_lib):
    """Without v_raw (global layers) the value is v_norm(k_raw)."""
    q, k, v, w_q, w_k = producer_case(2, 32, 4, 512, seed=32)
    a = oracle_lib.prepare_decode_f64(q, k, None, w_q, w_k, [5, 9], 64, 1.0e6)
    b = oracle_lib.prepare_decode_f64(q, k, k, w_q, w_k, [5, 9], 64, 1.0e6)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert np.all(np.isnan(oracle_lib.prepare_decode_f64(q, k, v, w_q, w_k, [0, 3], 64, 1e6)[0][0]))


def test_oracle_rejects_ranges_outside_the_cache(oracle_lib):
    q, k, v = random_case(1, 8, 4, 2, 8, seed=16)
    with pytest.raises(ValueError):
        oracle_lib.gqa_decode_f64(q, k, v, [9], 0)
    with pytest.raises(ValueError):
        oracle_lib.gqa_decode_f64(q, k, v, [-1], 0)
    with pytest.raises(ValueError):   # window start before pos_base
        oracle_lib.gqa_decode_f64(q, k, v, [8], 0, pos_base=1)


def test_thread_count_does_not_change_results(oracle_lib):
    q, k, v = random_case(2, 64, 32, 4, 64, seed=17)
    a = oracle_lib.gqa_decode_f64(q, k, v, [64, 50], 0, nthreads=1)
    b = oracle_lib.gqa_decode_f64(q, k, v, [64, 50], 0, nthreads=4)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# multi-query decode: T new tokens per sequence ("Gemma 4 31B-it Text
# Architecture", "Inference behavior: Prefill, Cache, and Long Context" and
# "Compact form": positions = past_seen_tokens + arange(T_current), masks
# s <= t and t - 1024 < s <= t)
# ---------------------------------------------------------------------------

def mq_case(B, T, S, H, KVH, D, seed):
    rng = np.random.default_rng(seed)
    q = to_bits(rng.standard_normal((B, T, H, D)))
    k = to_bits(rng.standard_normal((B, S, KVH, D)))
    v = to_bits(rng.standard_normal((B, S, KVH, D)))
    return q, k, v


@pytest.mark.parametrize("T,W", [(1, 0), (3, 0), (4, 5), (5, 16), (8, 1)])
def test_mq_each_query_is_a_decode_step_at_its_position(oracle_lib, T, W):
    """Query t of a T-token step sees what a one-token decode step at length
    L - T + t + 1 sees (bitwise): the single-query oracle, with its own pins."""
    B, S, H, KVH, D = 4, 40, 8, 2, 16
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=40 + T)
    lens = [40, 21, T, max(1, T - 2)]
    out = oracle_lib.gqa_decode_mq_f64(q, k, v, lens, W)
    for t in range(T):
        step_lens = [max(0, L - T + t + 1) for L in lens]
        one = oracle_lib.gqa_decode_f64(np.ascontiguousarray(q[:, t]), k, v, step_lens, W)
        assert np.array_equal(out[:, t], one), f"query {t}"


@pytest.mark.parametrize("H,KVH,T,W", [(32, 16, 4, 1024), (32, 16, 6, 7), (32, 4, 4, 0),
                                       (32, 4, 3, 9)])
def test_mq_torch_sdpa_float64(oracle_lib, H, KVH, T, W):
    """SDPA in float64 with the Compact form's boolean mask built from the query
    positions (L - T) + arange(T): keys s <= t, and t - W < s for a window."""
    B, S, D = 3, 45, 16
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=50 + T + W)
    lens = [45, 30, T + 1]
    out = oracle_lib.gqa_decode_mq_f64(q, k, v, lens, W)
    g = H // KVH
    qt = torch.from_numpy(to_vals(q)).permute(0, 2, 1, 3)               # [B, H, T, D]
    kt = torch.from_numpy(to_vals(k)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(to_vals(v)).permute(0, 2, 1, 3).repeat_interleave(g, dim=1)
    s = torch.arange(S)[None, :]
    mask = torch.zeros(B, 1, T, S, dtype=torch.bool)
    for b, L in enumerate(lens):
        t = (L - T) + torch.arange(T)[:, None]        # query positions
        m = s <= t
        if W > 0:
            m &= s > t - W
        mask[b, 0] = m
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=1.0)
    np.testing.assert_allclose(out, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-11, atol=1e-13)


def test_mq_later_tokens_are_invisible_to_earlier_queries(oracle_lib):
    """Changing the key/value of new token t' changes queries t >= t' only."""
    B, T, S, H, KVH, D = 2, 5, 30, 8, 4, 16
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=60)
    lens = [30, 17]
    base = oracle_lib.gqa_decode_mq_f64(q, k, v, lens, 0)
    for tp in range(T):
        k2, v2 = k.copy(), v.copy()
        for b, L in enumerate(lens):
            k2[b, L - T + tp] = to_bits(-to_vals(k[b, L - T + tp]) * 3.0)
            v2[b, L - T + tp] = to_bits(to_vals(v[b, L - T + tp]) + 2.0)
        out = oracle_lib.gqa_decode_mq_f64(q, k2, v2, lens, 0)
        for t in range(T):
            same = np.array_equal(out[:, t], base[:, t])
            assert same == (t < tp), f"token {tp}, query {t}"


def test_mq_window_moves_with_each_query(oracle_lib):
    """With a window, query t drops position L - T + t - W that query t - 1 still
    sees: perturbing that one row changes query t - 1 and not query t."""
    B, T, S, H, KVH, D, W = 1, 4, 40, 4, 2, 8, 6
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=61)
    L = 40
    base = oracle_lib.gqa_decode_mq_f64(q, k, v, [L], W)
    for t in range(1, T):
        s = L - T + t - W   # seen by query t - 1 only
        v2 = v.copy()
        v2[0, s] = to_bits(to_vals(v[0, s]) + 5.0)
        out = oracle_lib.gqa_decode_mq_f64(q, k, v2, [L], W)
        assert not np.array_equal(out[0, t - 1], base[0, t - 1])
        assert np.array_equal(out[0, t:], base[0, t:])


def test_mq_queries_before_the_start_are_zero(oracle_lib):
    """L < T: queries at negative positions see nothing (o = 0); the first query at
    position 0 sees v[0] alone."""
    B, T, S, H, KVH, D = 1, 6, 8, 8, 2, 16
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=62)
    L = 3
    out = oracle_lib.gqa_decode_mq_f64(q, k, v, [L], 0)
    n_neg = T - L
    assert np.all(out[0, :n_neg] == 0.0)
    g = H // KVH
    for h in range(H):
        np.testing.assert_array_equal(out[0, n_neg, h], to_vals(v[0, 0, h // g]))


@pytest.mark.parametrize("H,KVH,D,T,W", [(32, 16, 16, 4, 20), (32, 4, 32, 3, 0)])
def test_mq_paged_equals_contiguous(oracle_lib, H, KVH, D, T, W):
    B, S = 3, 70
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=63)
    lens = [70, 33, 17]
    kp, vp, bt = scatter_to_pages(k, v, lens)
    paged = oracle_lib.gqa_decode_mq_paged_f64(q, kp, vp, bt, lens, W)
    contig = oracle_lib.gqa_decode_mq_f64(q, k, v, lens, W)
    assert np.array_equal(paged, contig)


def test_mq_paged_bad_page_hits_only_the_queries_that_see_it(oracle_lib):
    """A bad id on the page of the last new token (position L - 1, first slot of its
    page) turns only the last query into NaN."""
    B, T, S, H, KVH, D = 2, 3, 50, 8, 2, 16
    q, k, v = mq_case(B, T, S, H, KVH, D, seed=64)
    lens = [49, 33]   # L - 1 = 48 and 32: the first slot of a page
    kp, vp, bt = scatter_to_pages(k, v, lens)
    bt[0, 48 // 16] = kp.shape[0] + 3
    out = oracle_lib.gqa_decode_mq_paged_f64(q, kp, vp, bt, lens, 0)
    assert np.all(np.isnan(out[0, T - 1]))
    assert np.all(np.isfinite(out[0, :T - 1])) and np.all(np.isfinite(out[1]))
