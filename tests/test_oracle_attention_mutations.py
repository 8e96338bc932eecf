"""Shows that the pins of ``kda_attention`` are sharp: each plausible slip in its glue
(decay sign or use, beta handling, where the norm and the scale go), planted in a copy of
the function on the CPU, makes at least one pin in test_oracle_attention_pins.py fail."""
import numpy as np
import pytest

import oracle.kda_oracle as ko
import test_oracle_attention_pins as pins


def _attention(decay_sign=1.0, use_decay=True, sigmoid_beta=False, always_norm=False,
               scale_on_key=False, order_override=None):
    def kda_attention(query, key, value, beta, decay=None, initial_state=None,
                      softmax_scale=None, use_qk_l2norm=True, order="decay_first"):
        order = order_override or order
        q = np.asarray(query, dtype=np.float64)
        k = np.asarray(key, dtype=np.float64)
        v = np.asarray(value, dtype=np.float64)
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        scale = dk ** -0.5 if softmax_scale is None else float(softmax_scale)
        if use_qk_l2norm or always_norm:
            q, k = ko.l2_normalize(q), ko.l2_normalize(k)
        if scale_on_key:
            k = scale * k
        else:
            q = scale * q
        d = np.zeros((B, T, H)) if (decay is None or not use_decay) else \
            decay_sign * np.asarray(decay, dtype=np.float64)
        gamma = np.broadcast_to(d[..., None], (B, T, H, dk))
        b = np.asarray(beta, dtype=np.float64)
        if sigmoid_beta:
            b = ko.sigmoid(b)
        S = (np.zeros((B, H, dk, dv)) if initial_state is None
             else np.array(initial_state, dtype=np.float64, copy=True))
        out = np.zeros((B, T, H, dv))
        for t in range(T):
            o, S = ko.kda_token(S, q[:, t], k[:, t], v[:, t], gamma[:, t], b[:, t], order)
            out[:, t] = o
        return out, S
    return kda_attention


MUTANTS = {
    "decay_sign_flipped": _attention(decay_sign=-1.0),
    "decay_ignored": _attention(use_decay=False),
    "beta_through_sigmoid": _attention(sigmoid_beta=True),
    "norm_applied_when_disabled": _attention(always_norm=True),
    "scale_on_key": _attention(scale_on_key=True),
    "literal_order_as_default": _attention(order_override="literal"),
}

PIN_CALLS = [
    (pins.test_scalar_recurrence_by_hand_decay_first_and_literal, {}),
    (pins.test_scalar_two_tokens_by_hand, {}),
    (pins.test_one_token_closed_form, {"norm": True}),
    (pins.test_one_token_closed_form, {"norm": False}),
    (pins.test_pure_decay_closed_form, {}),
    (pins.test_orthonormal_keys_exact_retrieval, {}),
    (pins.test_norm_off_equals_norm_on_for_unit_inputs, {}),
    (pins.test_default_scale_and_agreement_with_the_gated_form, {}),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, monkeypatch):
    monkeypatch.setattr(pins, "kda_attention", MUTANTS[name])
    caught = []
    for f, kw in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                f(**kw)
        except Exception as e:
            caught.append((f.__name__, type(e).__name__))
    assert caught, f"no pin caught the mutant {name}"


def test_control_copy_passes_every_pin(monkeypatch):
    monkeypatch.setattr(pins, "kda_attention", _attention())
    for f, kw in PIN_CALLS:
        f(**kw)
