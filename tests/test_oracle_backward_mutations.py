"""Shows that the finite-difference pins of the oracle backward are sharp: plausible slips,
planted by editing one line of a copy of ``kda_backward``'s source on the CPU, make a pin in
test_oracle_backward_pins.py fail."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle.kda_oracle as ko
import test_oracle_backward_pins as pins

SRC = textwrap.dedent(inspect.getsource(ko.kda_backward))

MUTANTS = {
    "output_cotangent_not_added": ("dS = dS + qh[..., :, None] * do[..., None, :]", "dS = dS"),
    "query_grad_from_old_state": ('dq_hat[:, t] = np.einsum("bhij,bhj->bhi", S_new, do)',
                                  'dq_hat[:, t] = np.einsum("bhij,bhj->bhi", S_prev, do)'),
    "prediction_grad_sign": ("dp = -b[..., None] * du", "dp = b[..., None] * du"),
    "key_grad_missing_prediction_term": ('dk_t += np.einsum("bhij,bhj->bhi", base, dp)',
                                         "dk_t += 0.0"),
    "decay_not_applied_to_adjoint": ("dS = e[..., :, None] * dS_dec", "dS = dS_dec"),
    "gate_grad_against_decayed_state": ("dgamma[:, t] = e * np.sum(dS_dec * S_prev, axis=-1)",
                                        "dgamma[:, t] = e * np.sum(dS_dec * S_dec, axis=-1)"),
    "norm_grad_without_projection": (
        "dk_ = dk_hat / nk - k * np.sum(k * dk_hat, axis=-1, keepdims=True) / nk ** 3",
        "dk_ = dk_hat / nk"),
    "beta_grad_without_sigmoid_derivative": ('"dbeta_logits": dbeta * beta * (1.0 - beta),',
                                             '"dbeta_logits": dbeta,'),
    "a_log_grad_missing_z": ('"da_log": np.sum(dz * z, axis=(0, 1, 3)),',
                             '"da_log": np.sum(dz, axis=(0, 1, 3)),'),
}


def mutant(old, new):
    assert SRC.count(old) == 1, old
    ns = dict(vars(ko))
    exec(compile(SRC.replace(old, new), "<mutant>", "exec"), ns)
    return ns["kda_backward"]


PIN_CALLS = [
    (pins.test_directional_derivatives_match_finite_differences,
     {"order": "decay_first", "with_final": True}),
    (pins.test_directional_derivatives_match_finite_differences,
     {"order": "decay_first", "with_final": False}),
    (pins.test_value_gradient_closed_form_single_token, {}),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, monkeypatch):
    monkeypatch.setattr(pins, "kda_backward", mutant(*MUTANTS[name]))
    caught = []
    for f, kw in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                f(**kw)
        except Exception as e:
            caught.append((f.__name__, type(e).__name__))
    assert caught, f"no pin caught the mutant {name}"


def test_control_copy_passes(monkeypatch):
    monkeypatch.setattr(pins, "kda_backward", mutant("dp = -b[..., None] * du",
                                                     "dp = -b[..., None] * du"))
    for f, kw in PIN_CALLS:
        f(**kw)
