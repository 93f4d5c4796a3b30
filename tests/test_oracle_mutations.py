"""Planted mistakes in the oracle must fail its pins.

Each case rewrites one line of one oracle function (on the CPU, in a copy of the
function: the oracle's files are not touched) into a plausible slip -- a dropped
scale or normaliser, an off-by-one causal diagonal, a wrong head map, a reversed
rotation, a sign error in the gradient -- installs the copy where the oracle and
its pins look it up, and checks that at least one of the pins listed for it then
fails.  The unmutated oracle passes the same pins first, so a failure is the
mutation's doing and not a call error.

Mutations that change nothing the oracle returns are not listed: the direction in
which the ring passes its blocks does not change ring_sim's output (each device
still meets every block once, and the fold is order independent), so such a
mutant would be equivalent, not wrong.
"""

import inspect
import sys
import textwrap

import pytest

import oracle
import oracle.attention
import oracle.backward
import oracle.layouts
import oracle.merge
import oracle.ring
import oracle.tiles
import oracle.ulysses
import tests.test_oracle_pins as pins
from tests.conftest import GOLDEN


def _mutant(module, name, old, new):
    """A copy of module.name with the one occurrence of ``old`` replaced by ``new``."""
    src = textwrap.dedent(inspect.getsource(getattr(module, name)))
    assert src.count(old) == 1, f"{module.__name__}.{name}: mutation site found {src.count(old)} times"
    ns = dict(vars(module))
    exec(compile(src.replace(old, new), f"<mutant of {module.__name__}.{name}>", "exec"), ns)
    return ns[name]


def _install(monkeypatch, original, mutant):
    """Replace every reference to ``original`` in the oracle's modules and the pins module."""
    n = 0
    for modname, mod in list(sys.modules.items()):
        if mod is None or not (modname == "oracle" or modname.startswith("oracle.")
                               or modname == pins.__name__):
            continue
        for attr, val in list(vars(mod).items()):
            if val is original:
                monkeypatch.setattr(mod, attr, mutant)
                n += 1
    assert n > 0


def _first_failure(checks):
    """Index of the first check that raises, or None when all pass."""
    for i, check in enumerate(checks):
        try:
            check()
        except Exception:  # an assertion, or a crash of the mutated code
            return i
    return None


Z, S_, C = oracle.ZIGZAG, oracle.STRIPED, oracle.CONTIGUOUS

# The pins, as calls with their parameters filled in.
PIN = {
    "scipy": pins.test_full_attention_matches_scipy,
    "scipy_causal": pins.test_full_attention_causal_matches_scipy,
    "closed_forms": pins.test_full_attention_closed_forms,
    "rows_sum_to_one": pins.test_full_attention_rows_sum_to_one,
    "gqa": pins.test_gqa_head_mapping,
    "rows_equal_full": pins.test_full_attention_rows_equals_full,
    "attention_rows": pins.test_attention_rows_equals_full,
    "printed_counts": lambda: pins.test_printed_causal_pair_counts(GOLDEN),
    "small_tables": pins.test_layout_small_tables,
    "zigzag_balance": pins.test_zigzag_exact_balance,
    "toy_ring": lambda: pins.test_toy_ring_equals_attention(GOLDEN),
    "module23": lambda: pins.test_module23_example(GOLDEN),
    "ring_invariance": lambda: pins.test_ring_layout_invariance(Z),
    "pass_blocks": lambda: pins.test_pass_blocks_closed_form(3),
    "held_partials": lambda: pins.test_held_blocks_give_ring_partials(Z),
    "partials_merge": lambda: pins.test_ring_partials_merge_to_ring(Z, True),
    "merge_halves": pins.test_merge_of_halves_is_attention,
    "merge_empty": pins.test_merge_ignores_empty_parts,
    "tiles_brute_ragged": lambda: pins.test_tile_counts_bruteforce(C, 64, 4, 5),
    "tiles_brute_zigzag": lambda: pins.test_tile_counts_bruteforce(Z, 96, 4, 8),
    "tiles_closed_32k": pins.test_tile_counts_closed_forms_seq32k,
    "bwd_fd": lambda: pins.test_backward_finite_differences(True),
    "bwd_fd_noncausal": lambda: pins.test_backward_finite_differences(False),
    "bwd_special": pins.test_backward_special_cases,
    "bwd_rows_fd": lambda: pins.test_backward_rows_finite_differences(True),
    "ring_bwd": lambda: pins.test_ring_backward_equals_attention_backward(Z, True),
    "to_natural": lambda: pins.test_to_natural_inverts_the_layout(Z),
    "ulysses_exchange": lambda: pins.test_ulysses_exchange(Z),
    "ulysses_attention": pins.test_ulysses_attention_equals_full,
}

A, L, R = oracle.attention, oracle.layouts, oracle.ring

# (id, module, function, original text, planted slip, pins expected to catch it)
CASES = [
    # attention: the definition the ring reaches
    ("causal_diagonal_dropped", A, "full_attention", "pos[None, :] <= pos[r0:r1, None]",
     "pos[None, :] < pos[r0:r1, None]", ["scipy_causal", "closed_forms"]),
    ("scale_1_over_d", A, "full_attention", "sc = _scale(d, scale)",
     "sc = 1.0 / d if not scale else float(scale)", ["scipy", "closed_forms"]),
    ("gqa_modulo_map", A, "full_attention", "kh = k[b, h // group]", "kh = k[b, h % Hkv]", ["gqa"]),
    ("lse_base_2", A, "full_attention", "shift + np.log(z)", "shift + np.log2(z)", ["scipy", "closed_forms"]),
    ("softmax_not_normalised", A, "full_attention", "out[b, h, r0:r1] = probs @ vh",
     "out[b, h, r0:r1] = e @ vh", ["scipy", "rows_sum_to_one"]),
    ("rows_causal_diagonal_dropped", A, "full_attention_rows", "pos[None, :] <= qp[:, None]",
     "pos[None, :] < qp[:, None]", ["rows_equal_full"]),
    ("attention_rows_diagonal_dropped", A, "attention_rows", "kp[None, :limit] <= qp[rows, None]",
     "kp[None, :limit] < qp[rows, None]", ["attention_rows"]),
    # layouts: which positions a device owns
    ("zigzag_pairs_p_with_n_plus_p", L, "layout_positions", "second = (2 * n_shards - 1 - p) * c",
     "second = (n_shards + p) * c", ["small_tables", "zigzag_balance"]),
    ("striped_is_contiguous", L, "layout_positions", "pos[rows] = local * n_shards + p",
     "pos[rows] = p * s_n + local", ["printed_counts", "small_tables"]),
    ("pair_count_diagonal_dropped", L, "causal_pair_counts", "all_keys[None, :] <= q[:, None]",
     "all_keys[None, :] < q[:, None]", ["printed_counts"]),
    ("to_natural_gathers_instead_of_scattering", L, "to_natural", "out[..., pos, :] = x",
     "out = x[..., pos, :]", ["to_natural"]),
]

M, T, B_, U = oracle.merge, oracle.tiles, oracle.backward, oracle.ulysses

CASES += [
    # the ring: exchange, online-softmax fold, per-step partials
    ("exchange_reversed", R, "pass_blocks", "blocks[(p - 1) % n_shards]", "blocks[(p + 1) % n_shards]",
     ["pass_blocks"]),
    ("fold_output_not_rescaled", R, "_absorb", "o_new = o_old * corr[:, None] + p @ v_blk",
     "o_new = o_old + p @ v_blk", ["toy_ring", "module23", "ring_invariance"]),
    ("fold_denominator_not_rescaled", R, "_absorb", "l_new = l_old * corr + p.sum(axis=1)",
     "l_new = l_old + p.sum(axis=1)", ["toy_ring", "module23", "ring_invariance"]),
    ("partial_step_reversed", R, "ring_partials", "r = (p - t) % n_shards", "r = (p + t) % n_shards",
     ["held_partials"]),
    # merging (O_t, LSE_t) pairs
    ("merge_weights_not_normalised", M, "merge_partials", "out = (frac[..., None] * o_parts).sum(axis=0)",
     "out = (w[..., None] * o_parts).sum(axis=0)", ["merge_halves", "partials_merge"]),
    ("merge_lse_reference_dropped", M, "merge_partials", "lse = np.where(live, ref + np.log(z), -np.inf)",
     "lse = np.where(live, np.log(z), -np.inf)", ["merge_halves", "partials_merge"]),
    # causal tile classification
    ("full_tile_boundary_strict", T, "tile_counts", "all_ok = kmax[None, :] <= qmin[:, None]",
     "all_ok = kmax[None, :] < qmin[:, None]", ["tiles_brute_ragged", "tiles_closed_32k"]),
    ("skip_tile_boundary_loose", T, "tile_counts", "none_ok = kmin[None, :] > qmax[:, None]",
     "none_ok = kmin[None, :] >= qmax[:, None]", ["tiles_brute_ragged", "tiles_brute_zigzag"]),
    # gradients
    ("ds_sign_of_delta", B_, "attention_backward_rows", "ds = p * (dp - delta)", "ds = p * (dp + delta)",
     ["bwd_fd", "bwd_rows_fd"]),
    ("dq_scale_dropped", B_, "attention_backward_rows", "dq = sc * (ds @ k)", "dq = ds @ k",
     ["bwd_fd", "bwd_rows_fd"]),
    ("dp_against_keys", B_, "attention_backward_rows", "dp = do_rows @ v.T", "dp = do_rows @ k.T",
     ["bwd_fd_noncausal", "bwd_rows_fd"]),
    ("dv_from_ds", B_, "attention_backward_rows", "p[:, key_idx].T @ do_rows", "ds[:, key_idx].T @ do_rows",
     ["bwd_fd", "bwd_special"]),
    ("ring_bwd_probabilities_unnormalised", B_, "ring_backward", "p_blk = np.exp(s - lse[b, h, qp][:, None])",
     "p_blk = np.exp(s)", ["ring_bwd"]),
    ("ring_bwd_group_overwrites", B_, "ring_backward", "dk[b, g, rows[r]] += dk_acc",
     "dk[b, g, rows[r]] = dk_acc", ["ring_bwd"]),
    # Ulysses' exchange
    ("ulysses_keeps_layout_order", U, "ulysses_seq_to_head", "out[q, :, :, s] = x",
     "out[q, :, :, p * s_n + i] = x", ["ulysses_exchange", "ulysses_attention"]),
    ("ulysses_back_in_natural_order", U, "ulysses_head_to_seq", "out[:, q * hl:(q + 1) * hl, p * s_n + i] = y",
     "out[:, q * hl:(q + 1) * hl, s] = y", ["ulysses_exchange", "ulysses_attention"]),
    # masks by position, exchanges by count, brute-force tile classes
    ("mask_ignores_positions", A, "full_attention",
     "pos = np.arange(S, dtype=np.int64) if positions is None else np.asarray(positions, np.int64)",
     "pos = np.arange(S, dtype=np.int64)", ["rows_equal_full", "bwd_fd"]),
    ("held_blocks_one_exchange_too_many", R, "held_blocks", "for _ in range(step):",
     "for _ in range(step + 1):", ["pass_blocks", "held_partials"]),
    ("brute_force_diagonal_dropped", T, "tile_classes_bruteforce",
     "(kp[j0:j0 + tile][None, :] <= qp[i0:i0 + tile][:, None])",
     "(kp[j0:j0 + tile][None, :] < qp[i0:i0 + tile][:, None])", ["tiles_brute_ragged", "tiles_brute_zigzag"]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_fails_a_pin(case, monkeypatch):
    _, module, name, old, new, pin_names = case
    checks = [PIN[n] for n in pin_names]
    assert _first_failure(checks) is None, "the unmutated oracle must pass these pins"
    _install(monkeypatch, getattr(module, name), _mutant(module, name, old, new))
    assert _first_failure(checks) is not None, f"no pin of {pin_names} caught the planted mistake"
