"""The oracle against its pins, and planted mistakes against the pins.

Every pin in ``oracle_pins`` must hold for the committed oracle. Then each
mutation below is planted in a copy of kv_oracle.c (on the CPU, in a temp
directory), compiled, and the whole pin suite is run on it in a child
process: every mutant must be caught (a failing pin, or a crash).
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin_holds(pin, oracle_lib):
    pin(oracle_lib)


# (name, original text, planted mistake)
MUTANTS = [
    ("stride_drops_factor_2",
     "int64_t stride = (int64_t)d->page_size * blocks_of(d);\n    for (int64_t i = 0; i < n; ++i) {\n        int64_t p, o;",
     "int64_t stride = (int64_t)d->page_size * (int64_t)d->layer_num;\n    for (int64_t i = 0; i < n; ++i) {\n        int64_t p, o;"),
    ("mha_blocks_per_page_L",
     "return d->latent_only ? (int64_t)d->layer_num : 2 * (int64_t)d->layer_num;",
     "return d->latent_only ? (int64_t)d->layer_num : (int64_t)d->layer_num;"),
    ("mla_blocks_per_page_2L",
     "return d->latent_only ? (int64_t)d->layer_num : 2 * (int64_t)d->layer_num;",
     "return 2 * (int64_t)d->layer_num;"),
    ("mla_latent_in_block_2l",
     "return d->latent_only ? layer : 2 * layer;",
     "return 2 * layer;"),
    ("mla_asymmetric_rejected",
     "if (!d->latent_only && d->head_dim != d->v_head_dim) return ORA_ASYMMETRIC;",
     "if (d->head_dim != d->v_head_dim) return ORA_ASYMMETRIC;"),
    ("tail_pad_one_block_short",
     "out[4] = (int64_t)d->page_size * (blocks * R);",
     "out[4] = (int64_t)d->page_size * ((blocks - 1) * R);"),
    ("envelope_block_offset_transposed",
     "b * ((int64_t)d->page_size * R) + o * R;",
     "o * ((int64_t)d->page_size * R) + b * R;"),
    ("v_written_to_k_block",
     "memcpy(M + vb, V + i * R, (size_t)R);",
     "memcpy(M + kb, V + i * R, (size_t)R);"),
    ("k_and_v_blocks_swapped_in_gather",
     "memcpy(outK + r * R, M + kb, (size_t)R);",
     "memcpy(outK + r * R, M + vb, (size_t)R);"),
    ("gather_output_row_ignores_start",
     "int64_t r = cu[s] + (j - st);",
     "int64_t r = cu[s] + j;"),
    ("gather_offset_from_wrong_operand",
     "int64_t o = j % ps;",
     "int64_t o = k % ps;"),
    ("id_bound_allows_2_pow_31",
     "int64_t limit = ((int64_t)1 << 31) - 1;",
     "int64_t limit = ((int64_t)1 << 31);"),
    ("page_map_ignored",
     "phys = v2p[page];",
     "phys = page;"),
    ("tombstoned_page_not_clamped",
     "if (phys < 0) return 0;                    /* tombstoned page -> sink */",
     "if (phys < 0) phys = -phys;"),
    ("move_copies_half_the_blocks",
     "for (int64_t b = 0; b < blocks; ++b)\n            memcpy(snap",
     "for (int64_t b = 0; b < blocks / 2; ++b)\n            memcpy(snap"),
    ("move_decodes_offset_with_page_size",
     "*o = id % stride;",
     "*o = id % d->page_size;"),
    ("last_view_end_drops_block_reach",
     "out[6] = d->anchor + (blocks - 1) * d->page_size * R + n_rows * R;",
     "out[6] = d->anchor + n_rows * R;"),
    ("layer_stride_one_block",
     "int64_t page_bytes = (int64_t)d->page_size * blocks * R;",
     "int64_t page_bytes = (int64_t)d->page_size * (blocks - 1) * R;"),
    ("mla_move_rows_names_2L_blocks",
     "int64_t blocks = blocks_of(d);\n    int err = 0;\n    for (int64_t i = 0; i < m; ++i) {",
     "int64_t blocks = 2 * (int64_t)d->layer_num;\n    int err = 0;\n    for (int64_t i = 0; i < m; ++i) {"),
    ("block_table_entry_not_scaled",
     "out[(int64_t)s * max_pages + k] = (int32_t)(phys < 0 ? 0 : phys * blocks);",
     "out[(int64_t)s * max_pages + k] = (int32_t)(phys < 0 ? 0 : phys);"),
    ("block_table_prefix_floor",
     "int64_t np = len > 0 ? (len + ps - 1) / ps : 0;",
     "int64_t np = len > 0 ? len / ps : 0;"),
    ("kf_gather_entry_read_as_physical_page",
     "int e = decode_id(d, p * ps + o, &p, &o);",
     "int e = decode_id(d, p * ps * blocks_of(d) + o, &p, &o);"),
    ("kf_gather_drops_offset",
     "int e = decode_id(d, p * ps + o, &p, &o);",
     "int e = decode_id(d, p * ps, &p, &o);"),
    ("swa_map_skipped",
     "            else mapped = tmap[t];",
     "            else mapped = t;"),
    ("asymmetric_not_rejected",
     "if (!d->latent_only && d->head_dim != d->v_head_dim) return ORA_ASYMMETRIC;",
     ""),
]


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, orig, mut, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kv_oracle.c")).read()
    assert src.count(orig) == 1, f"mutation site for {name} not unique/present"
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(src.replace(orig, mut))
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", str(c), "-o", str(so)])
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), str(so)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived every pin:\n{r.stdout}\n{r.stderr}"
