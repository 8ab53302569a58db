"""The pins must catch plausible mistakes: each case plants one error in a copy
of the oracle's C source (CPU only), builds it, and checks that some pin fails."""
import ctypes
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "decay_on_write_term": ("+ beta * vt[n] * kt[m];", "+ alpha * beta * vt[n] * kt[m];"),
    "erase_sign": ("(S[n * P->dk + m] - beta * Sk[n] * kt[m])",
                   "(S[n * P->dk + m] + beta * Sk[n] * kt[m])"),
    "transposed_readout": ("acc += S[n * P->dk + m] * qt[m];", "acc += S[m * P->dk + n] * qt[m];"),
    "key_head_map": ("const int32_t hk = h / (P->Hv / P->Hk);", "const int32_t hk = h % P->Hk;"),
    "skip_root_step": ("for (int32_t s = 0; s < len; ++s) gdn_step",
                       "for (int32_t s = (len > 1); s < len; ++s) gdn_step"),
    "decay_sign": ("const double alpha = exp(P->g[t * P->Hv + h]);",
                   "const double alpha = exp(-P->g[t * P->Hv + h]);"),
    "drop_beta_in_erase": ("- beta * Sk[n] * kt[m]", "- Sk[n] * kt[m]"),
    # the selected-output entry point: value head and node swapped, and the
    # request's row offset dropped from its read-out row
    "selected_swap_head_node": ("int32_t b = (int32_t)J->sel[3 * u], h = (int32_t)J->sel[3 * u + 1];\n"
                                "            int32_t i = (int32_t)J->sel[3 * u + 2];",
                                "int32_t b = (int32_t)J->sel[3 * u], h = (int32_t)J->sel[3 * u + 2];\n"
                                "            int32_t i = (int32_t)J->sel[3 * u + 1];"),
    "selected_drop_request_offset": ("readout(P, S, (int64_t)P->offsets[b] + i, h, J->out + u * P->dv);",
                                     "readout(P, S, (int64_t)i, h, J->out + u * P->dv);"),
}

PIN_CASES = [
    lambda: [pins.test_hand_worked_values(c) for c in pins._parse_golden(pins.GOLDEN)],
    lambda: pins.test_delta_rule_write_property(0),
    lambda: pins.test_beta_zero_closed_form(0),
    lambda: pins.test_brute_force_all_forests(4),
    lambda: pins.test_head_sharing_equals_duplicated_key_heads(),
    lambda: pins.test_chain_matches_matrix_form(),
    # every request has Hv nodes here, so a swapped (h, i) stays inside the arrays
    lambda: pins.test_verify_selected_matches_verify("square"),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, name
    mutated = tmp_path / "gdn_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           str(mutated), "-o", str(so), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(str(so))))
    caught = 0
    for case in PIN_CASES:
        try:
            case()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught mutant {name}"
