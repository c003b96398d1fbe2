"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutant swaps one small piece of oracle/uniprefill_oracle.py for a wrong
variant; the pins of test_oracle_pins.py must then fail.
"""
import numpy as np
import pytest

import oracle
import oracle.uniprefill_oracle as O
import tests.test_oracle_pins as pins


class _Patch:
    """Swap a function in the oracle module and in the package namespace that re-exports it."""

    def __init__(self, mp):
        self.mp = mp

    def setattr(self, mod, name, fn):
        self.mp.setattr(mod, name, fn)
        if hasattr(oracle, name):
            self.mp.setattr(oracle, name, fn)


@pytest.fixture
def patch(monkeypatch):
    return _Patch(monkeypatch)


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, IndexError, ValueError, FloatingPointError):
        return True
    return False


def _golden_cases():
    return pins._golden("topp_cases.json")["cases"]


def test_wrong_gqa_mapping_is_caught(patch):
    patch.setattr(O, "kv_head_of", lambda h, group: h % 2)
    assert _fails(pins.test_gqa_equals_explicit_head_expansion)


def test_strict_causal_mask_is_caught(patch):
    patch.setattr(O, "causal_visible", lambda qp, kp: kp[None, :] < qp[:, None])
    with np.errstate(invalid="ignore"):
        assert _fails(pins.test_closed_form_at_q_zero, 50, 16)


def test_missing_causal_mask_is_caught(patch):
    patch.setattr(O, "causal_visible", lambda qp, kp: np.ones((len(qp), len(kp)), dtype=bool))
    assert _fails(pins.test_closed_form_at_q_zero, 50, 16)
    assert _fails(pins.test_reduces_to_library_causal_attention_when_window_is_whole_sequence, 33)


def test_softmax_over_the_wrong_axis_is_caught(patch):
    def bad(z):
        m = z.max(axis=1, keepdims=True)
        e = np.exp(z - m)
        return e / e.sum(axis=0, keepdims=True)
    patch.setattr(O, "softmax_rows", bad)
    with np.errstate(invalid="ignore", divide="ignore"):
        assert _fails(pins.test_block_mass_sums_to_one_over_G, 64)


def test_missing_sqrt_dk_scale_is_caught(patch):
    real = O.softmax_rows
    patch.setattr(O, "softmax_rows", lambda z: real(z * np.sqrt(16.0)))   # undo the 1/sqrt(16)
    assert _fails(pins.test_reduces_to_library_causal_attention_when_window_is_whole_sequence, 33)


def test_dividing_the_short_block_by_its_length_is_caught(patch):
    def bad(s, cu_seqlens, G):
        cu = [int(c) for c in cu_seqlens]
        cb = O.cu_blocks_of(cu, G)
        out = np.zeros(int(cb[-1]))
        for r in range(len(cu) - 1):
            for g in range(int(cb[r + 1] - cb[r])):
                lo = cu[r] + g * G
                hi = min(cu[r + 1], lo + G)
                out[cb[r] + g] = s[lo:hi].sum() / (hi - lo)
        return out
    patch.setattr(O, "block_scores_from_tokens", bad)
    assert _fails(pins.test_block_mass_sums_to_one_over_G, 64)


def test_ascending_tie_break_is_caught(patch):
    patch.setattr(O, "rank_order", lambda b: np.lexsort((np.arange(len(b)), -np.asarray(b))))
    case = [c for c in _golden_cases() if c["name"].startswith("ties")][0]
    assert _fails(pins.test_topp_golden, case)
    assert _fails(pins.test_packed_key_order_matches_rank_order)


def test_strict_threshold_is_caught(patch):
    def bad(bbar, p):
        order = O.rank_order(bbar)
        cum = np.cumsum(np.asarray(bbar, dtype=np.float64)[order])
        return order, int(np.argmax(cum > p * cum[-1])) + 1
    patch.setattr(O, "topp_kstar", bad)
    case = [c for c in _golden_cases() if c["name"].startswith("ties")][0]
    assert _fails(pins.test_topp_golden, case)


def test_forgetting_the_window_is_caught(patch):
    real = O.select_request

    def bad(bbar, N, G, n, A, p):
        return real(bbar, N, G, 0, A, p)
    patch.setattr(O, "select_request", bad)
    case = [c for c in _golden_cases() if c["name"].startswith("sinks")][0]
    assert _fails(pins.test_topp_golden, case)


def test_window_mean_over_n_instead_of_n_eff_is_caught(patch):
    real = O.token_scores

    def bad(Q, K, cu_seqlens, n):
        s = real(Q, K, cu_seqlens, n)
        cu = [int(c) for c in cu_seqlens]
        for r in range(len(cu) - 1):
            N = cu[r + 1] - cu[r]
            s[cu[r]:cu[r + 1]] *= min(n, N) / n
        return s
    patch.setattr(O, "token_scores", bad)
    assert _fails(pins.test_closed_form_at_q_zero, 10, 16)


@pytest.mark.parametrize("bad_layer_rule", ["inclusive", "first"])
def test_wrong_drop_history_rule_is_caught(patch, bad_layer_rule):
    def bad(kept_len, drop_layer, layer, orig_len, kv_len):
        if bad_layer_rule == "inclusive":
            prev = [l for l in range(len(drop_layer)) if drop_layer[l] and l <= layer]
        else:
            prev = [l for l in range(len(drop_layer)) if drop_layer[l] and l < layer][:1]
        out = np.zeros(len(orig_len), dtype=np.int64)
        for r in range(len(orig_len)):
            base = int(kept_len[max(prev)][r]) if prev else int(orig_len[r])
            out[r] = base + int(kv_len[r]) - int(orig_len[r])
        return out
    patch.setattr(O, "seqused", bad)
    assert _fails(pins.test_eq17_golden)
