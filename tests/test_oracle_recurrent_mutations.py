"""Shows that the pins of ``recurrent_attention`` are sharp: slips planted by editing one
line of a copy of its source on the CPU make a pin in test_oracle_recurrent_pins.py fail."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle.kda_oracle as ko
import test_oracle_recurrent_pins as pins

SRC = textwrap.dedent(inspect.getsource(ko.recurrent_attention))

MUTANTS = {
    "key_gate_on_value_axis": ("h = np.exp(a[b, t])[:, :, None] * h * np.exp(bv[b, t])[:, None, :]",
                               "h = np.exp(a[b, t])[:, None, :] * h * np.exp(bv[b, t])[:, :, None]"),
    "output_before_write": ('out[b, t] = np.einsum("hij,hi->hj", h, scale * q[b, t])',
                            'out[b, t] = np.einsum("hij,hi->hj", h - kk[b, t][:, :, None] * vv[b, t][:, None, :], scale * q[b, t])'),
    "reverse_ignored": ("order = range(hi - 1, lo - 1, -1) if reverse else range(lo, hi)",
                        "order = range(lo, hi)"),
    "gqa_interleaved": ("kk = np.repeat(k, grp, axis=2)  # key / value head of every query head",
                        "kk = np.tile(k, (1, 1, grp, 1))"),
    "g_gamma_dropped": ("a = a + np.asarray(g_gamma, dtype=np.float64)[:, None, :, None]",
                        "a = a"),
    "memory_transposed_in_read": ('out[b, t] = np.einsum("hij,hi->hj", h, scale * q[b, t])',
                                  'out[b, t] = np.einsum("hij,hj->hi", h, scale * q[b, t])'),
    "default_scale_one": ("scale = D ** -0.5 if softmax_scale is None else float(softmax_scale)",
                          "scale = 1.0 if softmax_scale is None else float(softmax_scale)"),
}


def mutant(old, new):
    assert SRC.count(old) == 1, old
    ns = dict(vars(ko))
    exec(compile(SRC.replace(old, new), "<mutant>", "exec"), ns)
    return ns["recurrent_attention"]


PIN_CALLS = [pins.test_ungated_is_causal_linear_attention, pins.test_all_gates_against_brute_force,
             pins.test_default_scale_and_initial_state_decay,
             pins.test_reverse_equals_time_flipped_forward,
             pins.test_grouped_kv_heads_equal_repeated_heads,
             pins.test_packed_sequences_equal_separate_calls]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_mutant(name, monkeypatch):
    monkeypatch.setattr(pins, "recurrent_attention", mutant(*MUTANTS[name]))
    caught = []
    for f in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                f()
        except Exception as e:
            caught.append((f.__name__, type(e).__name__))
    assert caught, f"no pin caught the mutant {name}"


def test_control_copy_passes(monkeypatch):
    monkeypatch.setattr(pins, "recurrent_attention", mutant("grp = Hq // Hkv", "grp = Hq // Hkv"))
    for f in PIN_CALLS:
        f()
