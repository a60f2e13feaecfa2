"""Mutation check of the oracle pins (CPU only).

Each case compiles a copy of the oracle's C source with one plausible mistake
planted in it, then runs every pin of ``test_oracle_pins`` against that copy.
The pins must reject every mutant: at least one of them fails (an assertion or a
rejected call).  The real oracle passes them all (``test_oracle_pins``).
"""
import itertools
import os

import pytest

import oracle
import tests.test_oracle_pins as pins

MUTANTS = {
    "window_start_one_late": (
        "*lo = (window > 0 && L > window) ? L - window : 0;",
        "*lo = (window > 0 && L > window) ? L - window + 1 : 0;"),
    "window_start_one_early": (
        "*lo = (window > 0 && L > window) ? L - window : 0;",
        "*lo = (window > 0 && L > window + 1) ? L - window - 1 : 0;"),
    "window_ignored": (
        "*lo = (window > 0 && L > window) ? L - window : 0;",
        "*lo = 0;"),
    "scale_inverse_sqrt_d": (
        "        scores[j] = s;\n",
        "        scores[j] = s / sqrt((double)D);\n"),
    "head_map_modulo": (
        "contig_ctx c = {k, v, bb, h / g,",
        "contig_ctx c = {k, v, bb, h % KVH,"),
    "paged_head_map_modulo": (
        "paged_ctx c = {k_pages, v_pages, bt_row, h / g,",
        "paged_ctx c = {k_pages, v_pages, bt_row, h % KVH,"),
    "no_max_subtraction": (
        "\n        scores[j] = exp(scores[j] - m);",
        "\n        scores[j] = exp(scores[j]);"),
    "keys_and_values_swapped": (
        "const uint16_t *kr = k_row(ctx, j);",
        "const uint16_t *kr = v_row(ctx, j);"),
    "value_row_misaligned": (
        "const uint16_t *vr = v_row(ctx, j);",
        "const uint16_t *vr = v_row(ctx, (j + 1) % n);"),
    "normaliser_dropped": (
        "for (d = 0; d < D; ++d) out[d] /= l;",
        "(void)l;"),
    "first_term_of_normaliser_dropped": (
        "\n        l += scores[j];\n",
        "\n        l += (j > 0) ? scores[j] : 0.0;\n"),
    "last_key_dropped": (
        "attend(q_row, D, hi - lo, contig_k",
        "attend(q_row, D, hi - lo - (hi - lo > 1), contig_k"),
    "paged_slot_shifted": (
        "int64_t slot = s % x->page_size;",
        "int64_t slot = (s + 1) % x->page_size;"),
    "paged_page_index_off": (
        "int64_t page = x->bt_row[s / x->page_size];",
        "int64_t page = x->bt_row[(s + 1) / x->page_size];"),
    "query_transposed": (
        "q_row[d] = bf16_bits_to_double(q[(bb * H + h) * D + d]);\n                contig_ctx",
        "q_row[d] = bf16_bits_to_double(q[(d % H) * D + (bb * H + h) % D]);\n                contig_ctx"),
    "ring_row_shifted": (
        "const int64_t row = s % x->C;",
        "const int64_t row = (s + 1) % x->C;"),
    "ring_head_map_modulo": (
        "ring_ctx c = {k, v, bb, h / g,",
        "ring_ctx c = {k, v, bb, h % KVH,"),
    "ring_window_start_late": (
        "attend(q_row, D, hi - lo, ring_k",
        "attend(q_row, D, hi - lo - (hi - lo > 1), ring_k"),
    "keqv_frequency_exponent": (
        "(double)s * pow(theta, -2.0 * (double)i / (double)D)",
        "(double)s * pow(theta, -2.0 * (double)i / (double)(D / 2))"),
    "producer_frequency_exponent": (
        "(double)pos * pow(theta, -2.0 * (double)i / (double)D)",
        "(double)pos * pow(theta, -2.0 * (double)i / (double)(D / 2))"),
    "keqv_sine_sign": (
        "k[i] = x0 * c - x1 * sn;",
        "k[i] = x0 * c + x1 * sn;"),
    "keqv_pair_offset": (
        "const int half = D / 2;\n    for (d = 0; d < D; ++d) k[d] = w[d]",
        "const int half = D / 2 - 1;\n    for (d = 0; d < D; ++d) k[d] = w[d]"),
    "keqv_position_shift": (
        "w, D, n_rot, theta, s, k);",
        "w, D, n_rot, theta, s + 1, k);"),
    "keqv_weight_ignored": (
        "for (d = 0; d < D; ++d) k[d] = w[d] * bf16_bits_to_double(vr[d]);",
        "for (d = 0; d < D; ++d) k[d] = bf16_bits_to_double(vr[d]);"),
    "producer_eps_outside_root": (
        "1.0 / sqrt(ss / (double)D + PRODUCER_EPS);",
        "1.0 / (sqrt(ss / (double)D) + PRODUCER_EPS);"),
    "producer_norm_over_d_minus_1": (
        "1.0 / sqrt(ss / (double)D + PRODUCER_EPS);",
        "1.0 / sqrt(ss / (double)(D - 1) + PRODUCER_EPS);"),
    "producer_weight_ignored": (
        "        if (w) y[d] *= bf16_bits_to_double(w[d]);\n",
        "\n"),
    "producer_position_is_length": (
        "const int64_t pos = (int64_t)seq_lens[b] - 1;",
        "const int64_t pos = (int64_t)seq_lens[b];"),
    "producer_rope_pair_offset": (
        "    const int half = D / 2;\n    for (i = 0; i < n_rot; ++i) {\n        const double a = (double)pos",
        "    const int half = D / 2 - 1;\n    for (i = 0; i < n_rot; ++i) {\n        const double a = (double)pos"),
    "producer_rope_sign": (
        "        y[i] = x0 * c - x1 * s;",
        "        y[i] = x0 * c + x1 * s;"),
    "producer_value_weighted": (
        "            rms_norm_head(vr, NULL, D, yv);",
        "            rms_norm_head(vr, w_k, D, yv);"),
    "mq_position_one_late": (
        "const int64_t p = L - T + t; /* position of query t */",
        "const int64_t p = L - T + t + 1;"),
    "mq_position_one_early": (
        "const int64_t p = L - T + t; /* position of query t */",
        "const int64_t p = L - T + t - 1;"),
    "mq_every_query_at_the_last_position": (
        "const int64_t p = L - T + t; /* position of query t */",
        "const int64_t p = L - 1 + 0 * t;"),
    "mq_window_anchored_at_the_length": (
        "*lo = (window > 0 && *hi > window) ? *hi - window : 0;",
        "*lo = (window > 0 && L > window) ? L - window : 0;"),
    "mq_queries_reversed": (
        "query_range(seq_lens[bb], T, t, window, &lo, &hi);\n                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[row * D + d]);\n                const int64_t n = hi - lo;\n                contig_ctx",
        "query_range(seq_lens[bb], T, T - 1 - t, window, &lo, &hi);\n                for (d = 0; d < D; ++d) q_row[d] = bf16_bits_to_double(q[row * D + d]);\n                const int64_t n = hi - lo;\n                contig_ctx"),
    "mq_head_map_modulo": (
        "const int64_t kvh = h / g; /* the query head's KV head */",
        "const int64_t kvh = h % KVH;"),
    "mq_query_rows_head_major": (
        "const int64_t row = (bb * T + t) * H + h; /* [B, T, H] index */",
        "const int64_t row = (bb * H + h) * T + t;"),
    "mq_paged_head_map_modulo": (
        "const int64_t kvh = h / g;\n                int64_t lo, hi, s;",
        "const int64_t kvh = h % KVH;\n                int64_t lo, hi, s;"),
    "empty_range_not_zero": (
        "if (n <= 0) return; /* empty sum */",
        "if (n <= 0) { for (d = 0; d < D; ++d) out[d] = 1.0; return; }"),
}


def _expand(fn):
    """All argument combinations of a pin's pytest parametrize marks."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [{}]
    axes = []
    for m in marks:
        names = [n.strip() for n in m.args[0].split(",")]
        values = m.args[1]
        axes.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
    out = []
    for combo in itertools.product(*axes):
        d = {}
        for part in combo:
            d.update(part)
        out.append(d)
    return out


PIN_FUNCS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    so = oracle.compile_variant(src.replace(before, after), os.path.join(tmp_path, f"m_{name}.so"))
    mutant = oracle.OracleLibrary(so)
    failed = []
    for fn in PIN_FUNCS:
        for kwargs in _expand(fn):
            try:
                fn(mutant, **kwargs)
            except (AssertionError, ValueError):
                failed.append(fn.__name__)
                break
    assert failed, f"no pin rejects mutant {name}"
