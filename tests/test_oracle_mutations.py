"""The pins must catch plausible mistakes in the oracle.  Each case plants one
mistake in a copy of oracle.c (off-by-one index, dropped scale, wrong head
mapping, K for V, dropped key, broken merge, ...), builds it on the CPU, runs the
pin suite against that build, and requires at least one pin to fail."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")

MUTATIONS = {
    "slot_offset_off_by_one": ("long long offset = pos % block_size;",
                               "long long offset = (pos + 1) % block_size;"),
    "slot_wrong_block": ("int32_t phys = block_tables[(int64_t)s * max_blocks + logical_block];",
                         "int32_t phys = block_tables[(int64_t)s * max_blocks + (logical_block ? logical_block - 1 : 0)];"),
    "ceil_is_floor": ("if (n * block_size < num_tokens) n += 1; /* round up */", ""),
    "write_value_into_k": ("memcpy((char *)k_cache + dst_elem * eb,\n               (const char *)key",
                           "memcpy((char *)k_cache + dst_elem * eb,\n               (const char *)value"),
    "scale_dropped": ("x[j - j_begin] = pr->scale * dot;", "x[j - j_begin] = dot;"),
    "gqa_mapping_modulo": ("int g = h / group; /* kv-head serving q-head h */",
                           "int g = h % pr->num_kv_heads;"),
    "values_from_k_pool": ("o[d] += w * load_elem(pr->v_cache, v_off + d, pr->dtype);\n    }\n    free(x);\n    return OR_OK;\n}\n\nstatic int check_problem",
                           "o[d] += w * load_elem(pr->k_cache, v_off + d, pr->dtype);\n    }\n    free(x);\n    return OR_OK;\n}\n\nstatic int check_problem"),
    "own_key_dropped": ("int64_t n = pos + 1;                      /* keys 0..pos are visible */",
                        "int64_t n = pos > 0 ? pos : 1;"),
    "no_exponential": ("for (int64_t j = 0; j < n; ++j) { x[j] = exp(x[j] - mx); z += x[j]; }",
                       "for (int64_t j = 0; j < n; ++j) { x[j] = 1.0 + x[j] - mx; z += x[j]; }"),
    "merge_without_rescale": ("for (int i = 0; i < nparts; ++i) total += l[i] * exp(m[i] - big);",
                              "for (int i = 0; i < nparts; ++i) total += l[i];"),
    "q_dims_reversed": ("dot += load_elem(pr->q, q_off + d, pr->dtype) *",
                        "dot += load_elem(pr->q, q_off + (pr->head_dim - 1 - d), pr->dtype) *"),
    "bf16_low_half": ("uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;",
                      "uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 15;"),
    "encode_keeps_causal_mask": ("if (pr->non_causal) n = ctx;              /* encode: the whole sequence */", ""),
    "copy_blocks_k_only": ("memcpy((char *)dst_v + (int64_t)dst * block_bytes,\n               (const char *)src_v",
                           "memcpy((char *)dst_v + (int64_t)dst * block_bytes,\n               (const char *)src_k"),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(os.path.join(ORACLE_DIR, "oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {name}"
    (tmp_path / "oracle.c").write_text(src.replace(old, new))
    shutil.copy(os.path.join(ORACLE_DIR, "oracle.h"), tmp_path / "oracle.h")
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", str(tmp_path / "oracle.c"), "-o", str(lib),
                    "-lm"], check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"no pin caught the planted mistake '{name}'"
