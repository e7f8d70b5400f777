"""Plant plausible mistakes in a copy of the oracle and check the pins fail.

Each mutant is a one-line edit of oracle/kvi_oracle.c (a dropped term, a
flipped sign, a wrong frequency, a reversed tie-break, an off-by-one in
placement, a div/mod swap in paging, a stride slip, a bad bf16 decode, a
swapped interleaved pair, a reversed or misplaced Llama 3.1 blend, a table
rotation sign),
compiled to a temporary library on the CPU; the pin suite is then run against
it in a subprocess and must fail.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kvi_oracle.c")

MUTANTS = {
    "scores_drop_first_term": (
        "for (int64_t j = 0; j < e; ++j)\n            s += ",
        "for (int64_t j = 1; j < e; ++j)\n            s += "),
    "topk_tie_to_higher_id": (
        "return (x->id > y->id) - (x->id < y->id);",
        "return (x->id < y->id) - (x->id > y->id);"),
    "place_off_by_one": (
        "pos[j] = p;\n        p += fact_len[sel[j]];",
        "p += fact_len[sel[j]];\n        pos[j] = p;"),
    "rotate_sign_flip": (
        "y[i] = x0 * c - x1 * s;", "y[i] = x0 * c + x1 * s;"),
    "rotate_drop_term": (
        "y[i + half] = x1 * c + x0 * s;", "y[i + half] = x1 * c;"),
    "rotate_wrong_frequency": (
        "const double w = pow(theta, -2.0 * (double)i / (double)d);",
        "const double w = pow(theta, -1.0 * (double)i / (double)d);"),
    "rotate_interleaved_pairing": (
        "const double x0 = x[i], x1 = x[i + half];\n        y[i] = x0 * c - x1 * s;\n        y[i + half] = x1 * c + x0 * s;",
        "const double x0 = x[2 * i], x1 = x[2 * i + 1];\n        y[2 * i] = x0 * c - x1 * s;\n        y[2 * i + 1] = x1 * c + x0 * s;"),
    "slot_div_mod_swap": (
        "*off = (int32_t)(p % block_size);", "*off = (int32_t)(p / block_size);"),
    "token_rows_v_reads_k": (
        "const uint16_t *vrow = kv + (((int64_t)l * 2 + 1) * n_tokens + row) * hd;",
        "const uint16_t *vrow = kv + (((int64_t)l * 2 + 0) * n_tokens + row) * hd;"),
    "bf16_decode_shift": ("(uint32_t)b << 16", "(uint32_t)b << 15"),
    "interleaved_pair_swapped": (
        "*a = 2 * i;\n        *b = 2 * i + 1;", "*a = 2 * i + 1;\n        *b = 2 * i;"),
    "llama3_blend_reversed": (
        "omega[i] = (1.0 - g) * w / factor + g * w;", "omega[i] = g * w / factor + (1.0 - g) * w;"),
    "llama3_edges_swapped": (
        "if (lambda < orig / high) {", "if (lambda < orig / low) {"),
    "table_rotation_sign": (
        "y[ia] = x[ia] * c[i] - x[ib] * sn[i];", "y[ia] = x[ia] * c[i] + x[ib] * sn[i];"),
    "graph_keeps_self": ("            if (j == i) continue;\n", "            if (j == i && n < 0) continue;\n"),
    "search_forgets_visited": ("                if (seen[f]) continue;\n", "                if (seen[f] && n < 0) continue;\n"),
    "search_expands_the_worst": (
        "for (int64_t i = 0; i < nc && np < width && np < 1024; ++i) {",
        "for (int64_t i = nc - 1; i >= 0 && np < width && np < 1024; --i) {"),
    "search_never_marks_expanded": ("                c[i].expanded = 1;\n", "\n"),
    "search_seeds_not_cut_to_beam": ("    if (nc > beam) nc = beam;\n", "\n"),
    "search_beam_one_short": ("nc = m < beam ? m : beam;", "nc = m < beam - 1 ? m : beam - 1;"),
}
PIN_FILES = ["test_oracle_pins.py", "test_oracle_graph_pins.py"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-shared",
                           "-fPIC", "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, KVI_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
