"""Planted mistakes in the oracle's numpy functions must fail a pin.

``test_oracle_mutants.py`` plants mistakes in the C source; the attention and
patch-formation oracles are numpy code in ``oracle/__init__.py``.  Each mutant
here is a one-line textual change to the source of ``Oracle.attend``,
``Oracle.attend_mla``, ``Oracle.attend_prefill`` or ``form_patch`` (a dropped term, a flipped sign, a wrong head, a missing scale,
the wrong end of the spectrum), compiled into a stand-in and run through the
pins of that function; it passes the test only by failing one of them.
"""
import inspect
import textwrap
import types

import numpy as np
import pytest

import oracle as O
from tests import oracle_pins as P

ATTEND_MUTANTS = {
    "value_patch_dropped": ("vv = vv + uv @ vvm.T", "vv = vv"),
    "key_patch_dropped": ("kk = kk + uk @ vk.T", "kk = kk"),
    "delta_sign": ("self.rotate(kf[rows, g, :], c.delta,", "self.rotate(kf[rows, g, :], -c.delta,"),
    "scale_dropped": ("sc = scale * (K @ qf[s, h])", "sc = K @ qf[s, h]"),
    "wrong_kv_head": ("for h in range(g * G, (g + 1) * G):", "for h in range(g, Hq, H):"),
    "softmax_not_normalised": ("pr = w / w.sum()", "pr = w"),
    "first_chunk_table_for_all": ("th = inv_freq[ci] if", "th = inv_freq[seq_starts[s]] if"),
}

MLA_ATTEND_MUTANTS = {
    "c_patch_dropped": ("cl = cl + uc @ vc.T", "cl = cl"),
    "key_c_patch_dropped": ("keys.append(np.concatenate([cl, kr], axis=1))",
                            "keys.append(np.concatenate([sf[rows, :kv_lora], kr], axis=1))"),
    "values_unpatched": ("lat.append(cl)", "lat.append(sf[rows, :kv_lora].copy())"),
    "rope_patch_dropped": ("kr = kr + ur @ vr.T", "kr = kr"),
    "delta_sign": ("self.rotate(sf[rows, kv_lora:], c.delta,", "self.rotate(sf[rows, kv_lora:], -c.delta,"),
    "scale_dropped": ("sc = scale * (K @ qf[s, h])", "sc = K @ qf[s, h]"),
    "softmax_not_normalised": ("pr = w / w.sum()", "pr = w"),
    "first_chunk_table_for_all": ("th = inv_freq[ci] if", "th = inv_freq[seq_starts[s]] if"),
}

PREFILL_MUTANTS = {
    "value_patch_dropped": ("vv = vv + uv @ vvm.T", "vv = vv"),
    "key_patch_dropped": ("kk = kk + uk @ vk.T", "kk = kk"),
    "delta_sign": ("self.rotate(kf[rows, g, :], c.delta,", "self.rotate(kf[rows, g, :], -c.delta,"),
    "scale_dropped": ("sc = scale * (K @ qf[s, t, h])", "sc = K @ qf[s, t, h]"),
    "first_token_for_all": ("sc = scale * (K @ qf[s, t, h])", "sc = scale * (K @ qf[s, 0, h])"),
    "wrong_kv_head": ("for h in range(g * G, (g + 1) * G):", "for h in range(g, Hq, H):"),
    "softmax_not_normalised": ("pr = w / den", "pr = w"),
    "lse_without_max": ("lse[s, t, h] = mx + np.log(den)", "lse[s, t, h] = np.log(den)"),
    "lse_base_2": ("lse[s, t, h] = mx + np.log(den)", "lse[s, t, h] = mx + np.log2(den)"),
    "lse_unscaled": ("lse[s, t, h] = mx + np.log(den)", "lse[s, t, h] = (mx + np.log(den)) / scale"),
}

FORM_PATCH_MUTANTS = {
    "sigma_dropped": ("return w[:, :m] * s[:m], zt[:m, :].T.copy()", "return w[:, :m], zt[:m, :].T.copy()"),
    "smallest_directions": ("return w[:, :m] * s[:m], zt[:m, :].T.copy()",
                            "return w[:, -m:] * s[-m:], zt[-m:, :].T.copy()"),
    "v_from_left_vectors": ("return w[:, :m] * s[:m], zt[:m, :].T.copy()",
                            "return zt[:m, :].T.copy() * s[:m], w[:, :m]"),
}

ATTEND_PINS = [P.pin_attend_single_token, P.pin_attend_uniform_keys, P.pin_attend_fused_identity,
               P.pin_attend_relative_position, P.pin_attend_per_chunk_tables, P.pin_attend_rows_are_the_row_oracle]
FORM_PATCH_PINS = [P.pin_form_patch_full_rank, P.pin_eckart_young]
PREFILL_PINS = [P.pin_attend_prefill_is_per_token_decode, P.pin_attend_prefill_lse_closed_form,
                P.pin_attend_prefill_lse_merge]
MLA_ATTEND_PINS = [P.pin_attend_mla_is_gqa_attention, P.pin_attend_mla_single_token,
                   P.pin_attend_mla_relative_position, P.pin_attend_mla_per_chunk_tables,
                   P.pin_attend_rows_are_the_row_oracle]


def _mutated(fn, old, new, env):
    src = textwrap.dedent(inspect.getsource(fn))
    assert src.count(old) == 1, (fn.__name__, old)
    ns = dict(env)
    exec(compile(src.replace(old, new), f"<mutant {fn.__name__}>", "exec"), ns)
    return ns[fn.__name__]


def _fails_some(pins, orc):
    for pin in pins:
        try:
            pin(orc)
        except (AssertionError, ValueError, IndexError):
            return True
    return False


@pytest.fixture(scope="module")
def orc():
    return O.default()


def test_unmutated_functions_pass(orc):
    for pin in ATTEND_PINS + FORM_PATCH_PINS + MLA_ATTEND_PINS + PREFILL_PINS:
        pin(orc)


@pytest.mark.parametrize("name", list(ATTEND_MUTANTS))
def test_attend_mutant_is_caught(name, orc):
    old, new = ATTEND_MUTANTS[name]
    fn = _mutated(O.Oracle.attend, old, new, vars(O))
    mut = O.Oracle()
    mut.attend = types.MethodType(fn, mut)
    assert _fails_some(ATTEND_PINS, mut), f"attend mutant {name} passed every pin"


@pytest.mark.parametrize("name", list(MLA_ATTEND_MUTANTS))
def test_mla_attend_mutant_is_caught(name, orc):
    old, new = MLA_ATTEND_MUTANTS[name]
    fn = _mutated(O.Oracle.attend_mla, old, new, vars(O))
    mut = O.Oracle()
    mut.attend_mla = types.MethodType(fn, mut)
    assert _fails_some(MLA_ATTEND_PINS, mut), f"attend_mla mutant {name} passed every pin"


@pytest.mark.parametrize("name", list(PREFILL_MUTANTS))
def test_prefill_mutant_is_caught(name, orc):
    old, new = PREFILL_MUTANTS[name]
    fn = _mutated(O.Oracle.attend_prefill, old, new, vars(O))
    mut = O.Oracle()
    mut.attend_prefill = types.MethodType(fn, mut)
    assert _fails_some(PREFILL_PINS, mut), f"attend_prefill mutant {name} passed every pin"


@pytest.mark.parametrize("name", list(FORM_PATCH_MUTANTS))
def test_form_patch_mutant_is_caught(name, orc, monkeypatch):
    old, new = FORM_PATCH_MUTANTS[name]
    fn = _mutated(O.form_patch, old, new, vars(O))
    monkeypatch.setattr(O, "form_patch", fn)
    assert _fails_some(FORM_PATCH_PINS, orc), f"form_patch mutant {name} passed every pin"
