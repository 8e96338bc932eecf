"""Shows that the oracle's pins are sharp: each plausible slip, planted in a copy of one
oracle function on the CPU, makes at least one pin in test_oracle_pins.py fail."""
import numpy as np
import pytest

import oracle.kda_oracle as ko
import test_oracle_pins as pins


def _token(decay_axis="rows", sign=-1.0, read_before=False, pred_transposed=False,
           order_override=None, skip_decay=False):
    def kda_token(S, q_hat, k_hat, v, gamma, beta, order="decay_first"):
        order = order_override or order
        e = np.exp(gamma)
        if skip_decay:
            e = np.ones_like(e)
        decay = e[..., :, None] if decay_axis == "rows" else e[..., None, :]
        b = np.asarray(beta)[..., None]
        base = decay * S if order == "decay_first" else S
        if pred_transposed:
            pred = np.einsum("...ij,...j->...i", base, k_hat)
        else:
            pred = np.einsum("...ij,...i->...j", base, k_hat)
        u = b * (v + sign * pred)
        S_new = decay * S + k_hat[..., :, None] * u[..., None, :]
        src = S if read_before else S_new
        o = np.einsum("...ij,...i->...j", src, q_hat)
        return o, S_new
    return kda_token


def _gate(no_exp=False, bias_sign=1.0):
    def activate_gate(g, a_log, dt_bias, lower_bound):
        g = np.asarray(g, dtype=np.float64)
        a = np.asarray(a_log, dtype=np.float64)[:, None]
        a = a if no_exp else np.exp(a)
        bias = np.asarray(dt_bias, dtype=np.float64).T
        return float(lower_bound) * ko.sigmoid(a * (g + bias_sign * bias))
    return activate_gate


MUTANTS = {
    "no_decay": ("kda_token", _token(skip_decay=True)),
    "delta_sign_flipped": ("kda_token", _token(sign=+1.0)),
    "output_read_before_update": ("kda_token", _token(read_before=True)),
    "memory_transposed_in_prediction": ("kda_token", _token(pred_transposed=True)),
    "decay_on_value_axis": ("kda_token", _token(decay_axis="cols")),
    "literal_order_as_default": ("kda_token", _token(order_override="literal")),
    "gate_without_exp_on_a_log": ("activate_gate", _gate(no_exp=True)),
    "gate_bias_subtracted": ("activate_gate", _gate(bias_sign=-1.0)),
    "no_l2_normalisation": ("l2_normalize", lambda x, eps=ko.L2_EPS: np.asarray(x, float)),
    "beta_used_as_probability": ("sigmoid", None),
}

PIN_CALLS = [
    (pins.test_gate_midpoint_and_three_quarters, {}),
    (pins.test_one_token_closed_form, {}),
    (pins.test_pure_decay_when_beta_is_zero, {}),
    (pins.test_orthonormal_keys_are_retrieved_exactly, {}),
    (pins.test_delta_rule_overwrites_instead_of_adding, {}),
    (pins.test_decay_and_delta_order, {"order": "decay_first"}),
    (pins.test_scalar_memory_matches_geometric_series, {}),
    (pins.test_decode_step_equals_last_scan_step, {}),
    (pins.test_normalisation_and_linearity_invariances, {}),
]


def _beta_as_probability(monkeypatch):
    """beta taken as given (no sigmoid) while the gate keeps its sigmoid: feed the
    oracle logit(clip(x)) so that its sigmoid hands back x itself."""
    real_forward = ko.kda_forward

    def kda_forward(q, k, v, g, beta_logits, *a, **kw):
        x = np.clip(np.asarray(beta_logits, dtype=np.float64), 1e-12, 1 - 1e-12)
        return real_forward(q, k, v, g, np.log(x / (1 - x)), *a, **kw)
    monkeypatch.setattr(ko, "kda_forward", kda_forward)
    monkeypatch.setattr(pins, "kda_forward", kda_forward)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, monkeypatch):
    target, fn = MUTANTS[name]
    if name == "beta_used_as_probability":
        _beta_as_probability(monkeypatch)
    else:
        monkeypatch.setattr(ko, target, fn)
        if hasattr(pins, target):
            monkeypatch.setattr(pins, target, fn)
    caught = []
    for f, kw in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                f(**kw)
        except Exception as e:  # AssertionError, or a shape error from a transposed operand
            caught.append((f.__name__, type(e).__name__))
    assert caught, f"no pin caught the mutant {name}"


def test_control_unmutated_oracle_passes_every_listed_pin():
    for f, kw in PIN_CALLS:
        f(**kw)
