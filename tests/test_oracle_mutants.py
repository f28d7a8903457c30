"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

Each case swaps one rule of the oracle for a wrong one -- an index off by one,
a flipped half, a reversed pairing, a dropped term, a different tie rule -- and
re-runs the pin that is meant to catch it. A mutant that survives would mean
the pins cannot tell the pages' method from a near miss.
"""

import numpy as np
import pytest

from conftest import read_golden
from oracle import numerics, schedules
import test_oracle_pins as pins
import test_oracle_properties as props


def _plant_ring_rule(monkeypatch, phase, rule):
    orig = schedules._ring_phase

    def patched(w, rings, r, reduce, combine, name):
        return orig(w, rings, rule if name == phase else r, reduce, combine, name)

    monkeypatch.setattr(schedules, "_ring_phase", patched)


def test_mutant_reduce_scatter_index(monkeypatch):
    _plant_ring_rule(monkeypatch, "reduce-scatter", lambda p, s: p + s)
    with pytest.raises(AssertionError):
        pins.test_ring_send_table_fig_4_2(read_golden)


def test_mutant_all_gather_index(monkeypatch):
    _plant_ring_rule(monkeypatch, "all-gather", lambda p, s: p - s)
    with pytest.raises(AssertionError):
        pins.test_ring_trace_4gpu(read_golden)


def test_mutant_intra_group_slice_rule(monkeypatch):
    # "send slice (l - s)" in phase 1 leaves local rank l owning slice l+1 and
    # breaks the hierarchical sum order
    _plant_ring_rule(monkeypatch, "intra-group reduce-scatter", lambda p, s: p - s)
    with pytest.raises(AssertionError):
        props.test_scale_and_bf16_finish_applied_once()


def test_mutant_receiver_overwrites_instead_of_adding(monkeypatch):
    orig = schedules._ring_phase

    def patched(w, rings, rule, reduce, combine, name):
        return orig(w, rings, rule, reduce, (lambda a, b: a) if reduce else combine, name)

    monkeypatch.setattr(schedules, "_ring_phase", patched)
    with pytest.raises(AssertionError):
        pins.test_ring_trace_4gpu(read_golden)


def test_mutant_rabenseifner_keeps_other_half(monkeypatch):
    src = schedules.rabenseifner_allreduce

    def flipped(x, **kw):
        # run with rank bits complemented: the kept half is the other one
        N = x.shape[0]
        out, st = src(x[::-1].copy(), **kw)
        st.owned = {N - 1 - i: v for i, v in st.owned.items()}
        return out[::-1], st

    monkeypatch.setattr(schedules, "rabenseifner_allreduce", flipped)
    with pytest.raises(AssertionError):
        pins.test_rabenseifner_fig_4_5(read_golden)


def test_mutant_tree_pairs_far_ranks_first(monkeypatch):
    def far_first(values):
        vals = list(values)
        while len(vals) > 1:
            h = len(vals) // 2
            vals = [vals[m] + vals[m + h] for m in range(h)]
        return vals[0]

    monkeypatch.setattr(numerics, "_tree", far_first)
    with pytest.raises(AssertionError):
        props.test_brute_force_every_algorithm(8, 64)


def test_mutant_ring_order_starts_one_rank_late(monkeypatch):
    orig = numerics._left_fold

    def late(x, ranks, cols=slice(None)):
        return orig(x, ranks[1:] + ranks[:1], cols)

    monkeypatch.setattr(numerics, "_left_fold", late)
    with pytest.raises(AssertionError):
        props.test_brute_force_every_algorithm(5, 31)


def test_mutant_bf16_ties_away_from_zero(monkeypatch):
    def away(x):
        bits = np.ascontiguousarray(x, np.float32).view(np.uint32)
        return ((bits + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)

    monkeypatch.setattr(numerics, "f32_to_bf16_rne", away)
    with pytest.raises(AssertionError):
        props.test_bf16_rne_hand_built(0x3F808000, 0x3F80)


def test_mutant_bf16_truncation(monkeypatch):
    def trunc(x):
        return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)

    monkeypatch.setattr(numerics, "f32_to_bf16_rne", trunc)
    with pytest.raises(AssertionError):
        props.test_bf16_rne_matches_torch_conversion()


# ---- schedule variants (recursive doubling, double binary tree, torus)

import test_oracle_variants as variants  # noqa: E402


def test_mutant_doubling_far_partner_first(monkeypatch):
    src = schedules.recursive_doubling_allreduce

    def far_first(x, **kw):
        # distance N/2 first: run on ranks with their bits reversed
        N = x.shape[0]
        k = N.bit_length() - 1
        rev = [int(format(i, f"0{k}b")[::-1], 2) if k else 0 for i in range(N)]
        out, st = src(x[rev].copy(), **kw)
        st.sends = [(s, rev[a], rev[b], lo, hi) for s, a, b, lo, hi in st.sends]
        return out[np.argsort(rev)], st

    monkeypatch.setattr(schedules, "recursive_doubling_allreduce", far_first)
    with pytest.raises(AssertionError):
        variants.test_recursive_doubling_fig_4_5(read_golden)
    with pytest.raises(AssertionError):
        variants.test_recursive_doubling_order_is_the_balanced_tree(8)


def test_mutant_tree_without_mirror(monkeypatch):
    monkeypatch.setattr(schedules, "double_binary_trees",
                        lambda N: [schedules.binary_tree(N), schedules.binary_tree(N)])
    with pytest.raises(AssertionError):
        variants.test_double_binary_tree_fig_4_6(read_golden)
    with pytest.raises(AssertionError):
        variants.test_double_binary_tree_inner_nodes_disjoint(8)


def test_mutant_tree_children_folded_high_first(monkeypatch):
    orig = schedules.double_binary_trees

    def reversed_children(N):
        return [(p, [sorted(c, reverse=True) for c in ch]) for p, ch in orig(N)]

    monkeypatch.setattr(schedules, "double_binary_trees", reversed_children)
    with pytest.raises(AssertionError):
        variants.test_double_binary_tree_order_closed_form(16, read_golden)


def test_mutant_tree_root_without_child(monkeypatch):
    orig = schedules.binary_tree

    def no_top(N):  # the in-order tree left dangling, rank 0 alone
        p, c = orig(N)
        if N > 1:
            top = c[0][0]
            c[0] = []
            p[top] = -1
        return p, c

    monkeypatch.setattr(schedules, "binary_tree", no_top)
    with pytest.raises(AssertionError):
        variants.test_double_binary_tree_fig_4_6(read_golden)


def test_mutant_torus_columns_first(monkeypatch):
    src = schedules.torus_allreduce

    def y_first(x, dims, **kw):  # run the transposed torus: Y lines first
        dims = list(dims) + [1] * (3 - len(dims))
        X, Y, Z = dims
        perm = [xx + X * (yy + Y * zz) for zz in range(Z) for xx in range(X) for yy in range(Y)]
        out, st = src(x[perm].copy(), (Y, X, Z), **kw)
        return out[np.argsort(perm)], st

    monkeypatch.setattr(schedules, "torus_allreduce", y_first)
    with pytest.raises(AssertionError):
        variants.test_torus_order_closed_form((2, 8))


def test_mutant_torus_line_ring_starts_one_late(monkeypatch):
    _plant_ring_rule(monkeypatch, "dim X reduce-scatter", lambda p, s: p - 1 - s)
    with pytest.raises(AssertionError):
        variants.test_torus_order_closed_form((4, 4))


# ---- blockwise INT8 compression and error feedback

from oracle import compress  # noqa: E402
import test_oracle_compress as comp  # noqa: E402


def _plant_quantizer(monkeypatch, scale_of, round_fn=np.rint, whole_tensor=False):
    def quantize(x, block):
        x = np.asarray(x, np.float32)
        b = x.size if whole_tensor else block
        nb = compress.n_blocks(x.size, block)
        codes = np.zeros(x.size, np.int8)
        scales = np.zeros(nb, np.float32)
        for k in range(compress.n_blocks(x.size, b)):
            xb = x[k * b:(k + 1) * b]
            s = scale_of(np.max(np.abs(xb)))
            for j in range(k * b // block, min(nb, ((k + 1) * b + block - 1) // block)):
                scales[j] = s
            if s:
                codes[k * b:(k + 1) * b] = np.clip(round_fn((xb / s).astype(np.float32)), -127, 127)
        return codes, scales

    monkeypatch.setattr(compress, "quantize_blockwise", quantize)


def test_mutant_scale_over_128(monkeypatch):
    _plant_quantizer(monkeypatch, lambda m: np.float32(np.float32(m) / np.float32(128)))
    with pytest.raises(AssertionError):
        comp.test_exact_grid_values()


def test_mutant_one_scale_per_tensor(monkeypatch):
    _plant_quantizer(monkeypatch, lambda m: np.float32(np.float32(m) / np.float32(127)), whole_tensor=True)
    with pytest.raises(AssertionError):
        comp.test_zero_tiny_and_ragged_blocks()


def test_mutant_codes_truncated(monkeypatch):
    _plant_quantizer(monkeypatch, lambda m: np.float32(np.float32(m) / np.float32(127)), round_fn=np.trunc)
    with pytest.raises(AssertionError):
        comp.test_codes_are_the_nearest_level_brute_force()


def test_mutant_feedback_sign_flipped(monkeypatch):
    def flipped(g, e, c):
        x = g + e
        v = c(x)
        return v, v - x

    monkeypatch.setattr(compress, "error_feedback_step", flipped)
    with pytest.raises(AssertionError):
        comp.test_error_feedback_worked_example(read_golden)


def test_mutant_feedback_residual_dropped(monkeypatch):
    monkeypatch.setattr(compress, "error_feedback_step", lambda g, e, c: (c(g), e * 0))
    with pytest.raises(AssertionError):
        comp.test_error_feedback_worked_example(read_golden)
