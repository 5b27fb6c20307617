"""Each plausible mistake in the oracle must fail at least one pin.

A mistake is planted in a copy of the oracle source (on the CPU, in a temporary
directory), the copy is compiled, and every pin of oracle_pins.py runs against
it. The test passes when some pin raises. This checks the pins' power, not the
oracle: the stock build passes every pin in test_oracle_pins.py.
"""
import os
import shutil

import pytest

import oracle as O
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(O.__file__), "art_oracle.c")

MUTANTS = {
    "mag_normalised_by_current_norm": [("fabs(nn - nprev) / nprev", "fabs(nn - nprev) / nn")],
    "magnitude_sign_dropped": [("fabs(nn - nprev) / nprev", "(nn - nprev) / nprev")],
    "cosine_uses_wrong_norm": [("1.0 - dot / (nn * nprev)", "1.0 - dot / (nn * nn)")],
    "non_strict_comparison": [("dmag < J->eps_mag && ddir < J->eps_dir",
                               "dmag <= J->eps_mag && ddir <= J->eps_dir")],
    "only_magnitude_tested": [("dmag < J->eps_mag && ddir < J->eps_dir", "dmag < J->eps_mag")],
    "only_direction_tested": [("dmag < J->eps_mag && ddir < J->eps_dir", "ddir < J->eps_dir")],
    "either_statistic_suffices": [("dmag < J->eps_mag && ddir < J->eps_dir",
                                   "(dmag < J->eps_mag || ddir < J->eps_dir)")],
    "patience_not_consecutive": [("counter = stable ? counter + 1 : 0",
                                  "counter = stable ? counter + 1 : counter")],
    "patience_off_by_one": [("counter >= J->patience", "counter > J->patience")],
    "block0_gate_missing": [("(seen0 || !has0)", "1")],
    "block0_gate_always": [("(seen0 || !has0)", "seen0")],
    "stop_one_block_late": [("{ bu = i; break; }", "{ bu = i + 1 > n ? n : i + 1; break; }")],
    "gqa_head_mapping": [("(size_t)g * G + h) * d + e", "(size_t)h * sh->num_kv_heads + g) * d + e")],
    "score_scale_dropped": [("s[t * G + h] = acc * inv_sqrt_d;", "s[t * G + h] = acc;")],
    "page_index_uses_block_size": [("t / Ps]", "t / Bk]")],
    "probe_index_ignored": [("row_off[t] + J->probe_idx[k])", "row_off[t] + k)")],
    "output_not_normalised": [("for (int e = 0; e < d; ++e) oh[e] /= Zh;", "")],
    "tail_not_masked": [("hi = lo + Bk < seq_len ? lo + Bk : seq_len", "hi = lo + Bk")] * 2,
    "duplicate_not_detected": [("if (seen[L[i]]) {", "if (0) {")],
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, mutant_dir):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert old in src, f"mutation site for {name} not found"
        src = src.replace(old, new, 1)
    d = mutant_dir / name
    d.mkdir()
    csrc = d / "art_oracle.c"
    csrc.write_text(src)
    lib = O.build(force=True, src=str(csrc), lib=str(d / "liboracle.so"))
    orc = O.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"mutant {name} passed every pin"
    shutil.rmtree(d, ignore_errors=True)
