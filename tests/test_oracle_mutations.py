"""Planted mistakes: each is a plausible slip in the oracle's arithmetic (a sign, an index, an
off-by-one, a swapped operand, a dropped rule).  A mutated copy of oracle.c is compiled into a
temporary library and the pins are run against it in a fresh process; every mutation must make
at least one pin fail, which shows the pins tie the oracle to the pages rather than to itself."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "bf16_round_up_on_ties": ("return (uint16_t)((lo & 1u) ? lo + 1 : lo);", "return (uint16_t)(lo + 1);"),
    "int8_ties_away": ("else n = (fmod(f, 2.0) == 0.0) ? f : f + 1.0;", "else n = f + 1.0;"),
    "int8_symmetric_clamp": ("if (a <= -128.0) return -128;", "if (a <= -127.0) return -127;"),
    "e4m3_overflow_to_nan": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 448.0) return (uint8_t)(sign | 0x7F);"),
    "rope_sign": ("    y[j] = fmaf(a, c, -bs);", "    y[j] = fmaf(a, c, bs);"),
    "rope_pairs_swapped": ("    float a = x[j], b = x[j + half];", "    float b = x[j], a = x[j + half];"),
    "gqa_map": ("      int hk = h / group;", "      int hk = h % num_kv_heads;"),
    "causal_drops_diagonal": ("(int64_t)past[r] + i + 1;", "(int64_t)past[r] + i;"),
    "scores_read_v": ("dot += qv[d] * pool_value(pool, kv_kind, kv_scale, pool_index(blk, 0,",
                      "dot += qv[d] * pool_value(pool, kv_kind, kv_scale, pool_index(blk, 1,"),
    "page_slot_off_by_one": ("int logical_block = (int)(pos / B), slot = (int)(pos % B);\n      int blk = logical_block < max_blocks_per_seq\n                    ? block_table[(size_t)r * max_blocks_per_seq + logical_block] : -1;\n      if (blk < 0 || blk >= num_blocks) {\n        status",
                             "int logical_block = (int)(pos / B), slot = (int)((pos + 1) % B);\n      int blk = logical_block < max_blocks_per_seq\n                    ? block_table[(size_t)r * max_blocks_per_seq + logical_block] : -1;\n      if (blk < 0 || blk >= num_blocks) {\n        status"),
    "draft_mask_word": ("mrow[j / 32] >> (j % 32)", "mrow[0] >> (j % 32)"),
    "draft_self_dropped": ("if (j != i && !((mrow", "if (!((mrow"),
    "draft_offsets_ignored": ("int64_t rpos = (int64_t)past[r] + off;", "int64_t rpos = (int64_t)past[r] + i;"),
    "draft_mask_row": ("gen_mask + (row - ctx_rows) * mask_words", "gen_mask + (row) * mask_words"),
    "draft_offset_range": ("if (off < 0 || off >= new_len[r])", "if (off < 0)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_every_planted_mistake_fails_a_pin(name, tmp_path):
    src = open(SRC).read()
    before, after = MUTATIONS[name]
    assert src.count(before) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(before, after))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", str(lib), str(mutated), "-lm"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught {name}:\n{r.stdout[-2000:]}"
