"""The oracle against its pins, and planted-mutation controls (CPU only).

A mutation is planted in a copy of the oracle's C source, on the CPU; every
mutant must fail at least one pin, which shows the pins can catch a dropped
term, a transposed index, a wrong layer or an off-by-one.
"""
import os
import subprocess
import sys

import pytest

import oracle
from tests import oracle_pins

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


MUTANTS = {
    "transposed_page_layer": ("int64_t block = page * num_layers + l;",
                              "int64_t block = l * num_layers + page;"),
    "dropped_token_term": ("return block * page_size * row_bytes + token_in_page * row_bytes;",
                           "return block * page_size * row_bytes;"),
    "token_major_inside_page": ("return block * page_size * row_bytes + token_in_page * row_bytes;",
                                "return (page * page_size + token_in_page) * num_layers * row_bytes"
                                " + l * row_bytes;"),
    "last_layer_skipped": ("for (int64_t l = 0; l < num_layers; ++l) {",
                           "for (int64_t l = 0; l + 1 < num_layers; ++l) {"),
    "load_reads_layer0": ("host_row_offset(host_idx[i], layer, num_layers",
                          "host_row_offset(host_idx[i], 0, num_layers"),
    "burst_off_by_one": ("for (int64_t l = layer_begin; l < layer_end; ++l) {",
                         "for (int64_t l = layer_begin + 1; l < layer_end; ++l) {"),
    "short_row": ("memcpy(dst, src, (size_t)row_bytes);\n    }\n  }",
                  "memcpy(dst, src, (size_t)row_bytes - 1);\n    }\n  }"),
    "pf_layer_major": ("return (h * num_layers + l) * row_bytes;",
                       "return (l * num_layers + h) * row_bytes;"),
    "pf_dropped_layer_term": ("return (h * num_layers + l) * row_bytes;",
                              "return (h * num_layers) * row_bytes;"),
    "pf_load_reads_layer0": ("pf_host_row_offset(host_idx[i], layer, num_layers, row_bytes)",
                             "pf_host_row_offset(host_idx[i], 0, num_layers, row_bytes)"),
    "device_slot_of_host": ("const uint8_t* src = src_layer + device_row_offset(device_idx[i], row_bytes);",
                            "const uint8_t* src = src_layer + device_row_offset(host_idx[i] % device_slots, row_bytes);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mutation_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(os.path.join(REPO, "oracle", "hicache_oracle.c")).read()
    assert old in src, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c_path = tmp_path / "hicache_oracle.c"
    c_path.write_text(mutated)
    # the mutant includes the oracle's own header
    (tmp_path / "hicache_oracle.h").write_text(
        open(os.path.join(REPO, "oracle", "hicache_oracle.h")).read())
    so = str(tmp_path / "libmutant.so")
    oracle.build_oracle(str(c_path), so, extra_flags=("-Wno-unused-variable",
                                                      "-Wno-unused-but-set-variable"))
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import oracle\n"
            "from tests.oracle_pins import run_all_pins\n"
            "f = run_all_pins(oracle.load(%r))\n"
            "print(f)\n"
            "sys.exit(3 if f else 0)\n") % (REPO, so)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    # exit 3: pins reported failures; a crash of the mutant also counts as caught
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr}"
