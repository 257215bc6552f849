"""The oracle's pins have teeth: plant plausible mistakes in copies of
pa_oracle.c (compiled here, on the CPU) and check that a pin fails for each.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

MUTANTS = {
    # causal window one key short (query i sees keys 0..L-n+i-1)
    "causal_off_by_one": (["const int visible = L - n + i + 1;"],
                          ["const int visible = L - n + i;"]),
    # GQA: query head h read from KV head h % Hkv instead of h / group
    "gqa_modulo": (["const int g = h / group;"],
                   ["const int g = h % J->num_kv_heads;"]),
    # token j read from the wrong offset inside its block
    "offset_shift": (["int64_t base = (((int64_t)b * J->num_kv_heads + g) * bs"
                      " + j % bs) * D;"],
                     ["int64_t base = (((int64_t)b * J->num_kv_heads + g) * bs"
                      " + (j + 1) % bs) * D;"]),
    # softmax without the max shift (overflows on large scores)
    "no_max_shift": (["      s[j] = exp(s[j] - smax);\n      denom += s[j];\n"
                      "    }\n    double* o"],
                     ["      s[j] = exp(s[j]);\n      denom += s[j];\n"
                      "    }\n    double* o"]),
    # K scale applied to V
    "scale_swap": (["o[d] += s[j] * (J->v_scale *"],
                   ["o[d] += s[j] * (J->k_scale *"]),
    # sliding window one key wide too many (keys p - W .. p)
    "window_off_by_one": (["  int first = position - window + 1;"],
                          ["  int first = position - window;"]),
    # NVFP4 codes written high nibble first
    "nvfp4_nibble_order": (["      codes[d / 2] |= (uint8_t)(c << (4 * (d & 1)));"],
                           ["      codes[d / 2] |= (uint8_t)(c << (4 - 4 * (d & 1)));"]),
    # INT4 scale max |x| / 8 instead of / 7
    "int4_scale": (["div_f32(amax, 7.0f)"], ["div_f32(amax, 8.0f)"]),
    # ties to odd
    "ties_to_odd": (["(c & 1) == 0 && (best & 1) == 1"],
                    ["(c & 1) == 1 && (best & 1) == 0"]),
    # cache written as [block][offset][head] instead of [block][head][offset]
    "layout_swap": (["((b * num_kv_heads + h) * (int64_t)block_size + o) *"
                     " head_dim + d;"],
                    ["((b * block_size + o) * (int64_t)num_kv_heads + h) *"
                     " head_dim + d;"]),
    # copy_blocks forgets V
    "copy_k_only": (["      ((char*)v_cache)[dst * block_bytes + i] =\n"
                     "          ((char*)v_cache)[src * block_bytes + i];\n"],
                    [""]),
}

# which pin must catch which planted mistake
CATCHERS = {
    "causal_off_by_one": lambda: pins.test_paged_equals_contiguous_sdpa(8, 2),
    "gqa_modulo": lambda: pins.test_paged_equals_contiguous_sdpa(8, 2),
    "offset_shift": lambda: pins.test_paged_equals_contiguous_sdpa(4, 4),
    "no_max_shift": pins.test_closed_forms,
    "scale_swap": pins.test_paged_bf16_and_fp8_match_sdpa_on_decoded_values,
    "ties_to_odd": pins.test_e4m3_encode_roundtrip_and_ties,
    "window_off_by_one": pins.test_window_of_one_key_is_the_own_value,
    "nvfp4_nibble_order": pins.test_nvfp4_write_properties,
    "int4_scale": pins.test_int4_write_properties,
    "layout_swap": pins.test_fig2_reshape_writes_only_the_new_slots,
    "copy_k_only": pins.test_copy_blocks_copies_whole_blocks_only,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(SRC).read()
    olds, news = MUTANTS[name]
    for old, new in zip(olds, news):
        assert old in src, f"mutation site not found: {old!r}"
        src = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC",
                    "-shared", "-D_POSIX_C_SOURCE=200809L", "-o", str(so),
                    str(c), "-lm", "-lpthread"], check=True)
    prev = oracle.swap_library(str(so))
    try:
        with pytest.raises((AssertionError, oracle.OracleError)):
            CATCHERS[name]()
    finally:
        oracle.restore_library(prev)
