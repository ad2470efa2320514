"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins catch every one of them (CPU only).

Each mutant replaces one snippet of ``oracle/pa_oracle.c`` (which must occur
exactly once), is compiled with gcc into a temporary library, and must fail
at least one of the checks in ``pins.py``.
"""
import os

import pytest

import oracle
import pins

MUTANTS = {
    "gqa_head_modulo": ("int h = kv_head * group + g; /* so that h / group == kv_head */",
                        "int h = g * num_kv_heads + kv_head;"),
    "scale_dropped": ("z[j] = scale * dot;", "z[j] = dot;"),
    "one_token_short": ("attend(out + row * head_dim, NULL, NULL, &wsum, q, Kc, Vc, ctx, head_dim, scale, z);",
                        "attend(out + row * head_dim, NULL, NULL, &wsum, q, Kc, Vc, ctx > 1 ? ctx - 1 : ctx, head_dim, scale, z);"),
    "table_index_modulo": ("int64_t block = table_row[j / block_size];",
                           "int64_t block = table_row[j % block_size];"),
    "pool_head_offset_swapped": ("return ((block * num_kv_heads + kv_head) * block_size + offset_in_block) * (int64_t)head_dim;",
                                 "return ((block * block_size + offset_in_block) * num_kv_heads + kv_head) * (int64_t)head_dim;"),
    "f16_exponent_bias": ("magnitude = ldexp((double)(1024 + fraction), exponent - 25);",
                          "magnitude = ldexp((double)(1024 + fraction), exponent - 24);"),
    "f16_subnormal_scale": ("magnitude = ldexp((double)fraction, -24);",
                            "magnitude = ldexp((double)fraction, -25);"),
    "bf16_shift": ("uint32_t word = (uint32_t)b << 16;", "uint32_t word = (uint32_t)b << 15;"),
    "weights_not_normalised": ("double a = z[j] / L;", "double a = z[j];"),
    "value_read_from_key_pool": ("Vc[(int64_t)j * head_dim + i] = orc_elem_to_double(v_pool, base + i, dtype);",
                                 "Vc[(int64_t)j * head_dim + i] = orc_elem_to_double(k_pool, base + i, dtype);"),
    "slot_block_offset_swapped": ("int64_t block = slot / block_size;\n        int offset = (int)(slot % block_size);",
                                  "int64_t block = slot % block_size;\n        int offset = (int)(slot / block_size);"),
    "copy_value_direction": ("memmove((char *)v_pools[layer] + dst * block_bytes,\n                    (const char *)v_pools[layer] + src * block_bytes, (size_t)block_bytes);",
                             "memmove((char *)v_pools[layer] + src * block_bytes,\n                    (const char *)v_pools[layer] + dst * block_bytes, (size_t)block_bytes);"),
    "merge_drops_rescale": ("L += l_p[p] * exp(m_p[p] - M);", "L += l_p[p];"),
    "swap_value_from_key_pool": ("(const char *)src_v[layer] + src * block_bytes, (size_t)block_bytes);",
                                 "(const char *)src_k[layer] + src * block_bytes, (size_t)block_bytes);"),
    "prefill_position_off_by_one": ("int position = ctx - n + i;", "int position = ctx - n + i - 1;"),
    "prefill_query_row": ("int64_t row = (int64_t)(first + i) * num_heads + h;",
                          "int64_t row = (int64_t)(first + n - 1 - i) * num_heads + h;"),
    "prefill_not_causal": ("Kc, Vc, position + 1, head_dim,", "Kc, Vc, ctx, head_dim,"),
    "prefill_prefix_ignored": ("int position = ctx - n + i;", "int position = i;"),
    "prefill_head_order": ("int h = kv_head * group + g;\n                    int64_t row = (int64_t)(first + i)",
                           "int h = g * num_kv_heads + kv_head;\n                    int64_t row = (int64_t)(first + i)"),
    "max_not_subtracted_in_weights": ("z[j] = exp(z[j] - M); /* z now holds the unnormalised weights w_j */",
                                      "z[j] = exp(z[j] - M) * (j == 0 ? 2.0 : 1.0);"),
}


def _run_checks(orc, golden):
    failures = []
    for check in pins.ORACLE_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError) as e:
            failures.append(f"{check.__name__}: {e}")
    for check in pins.GOLDEN_CHECKS:
        try:
            check(orc, golden)
        except (AssertionError, ValueError) as e:
            failures.append(f"{check.__name__}: {e}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, golden, tmp_path):
    original, mutated = MUTANTS[name]
    with open(oracle.SOURCE, encoding="utf-8") as f:
        text = f.read()
    assert text.count(original) == 1, f"snippet for {name} must occur exactly once"
    src = os.path.join(tmp_path, "mutant.c")
    with open(src, "w", encoding="utf-8") as f:
        f.write(text.replace(original, mutated))
    lib = oracle.compile_oracle(src, os.path.join(tmp_path, "libmutant.so"),
                                include_dir=os.path.dirname(oracle.SOURCE))
    failures = _run_checks(oracle.Oracle(lib), golden)
    assert failures, f"mutant {name} passed every pin"


@pytest.mark.parametrize("name", ["copy_value_direction", "slot_block_offset_swapped"])
def test_shared_prefix_pin_catches(name, tmp_path):
    """The shared-prefix = private-copies pin on its own catches a copy in the
    wrong direction and a slot split the wrong way round: the oracle's step
    then disagrees with the numpy-built private pools.  (A wrong table index
    reads the same wrong logical block through shared and private tables
    alike; the SDPA and relabelling pins catch that one.)"""
    original, mutated = MUTANTS[name]
    with open(oracle.SOURCE, encoding="utf-8") as f:
        text = f.read()
    src = os.path.join(tmp_path, "mutant.c")
    with open(src, "w", encoding="utf-8") as f:
        f.write(text.replace(original, mutated))
    lib = oracle.compile_oracle(src, os.path.join(tmp_path, "libmutant.so"),
                                include_dir=os.path.dirname(oracle.SOURCE))
    with pytest.raises((AssertionError, ValueError)):
        pins.check_shared_prefix_equals_private_copies(oracle.Oracle(lib))
