"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the pins
catch every one of them: a pin suite that a dropped term, a wrong sign or index or a
transposed operand passes would prove nothing."""
import os
import subprocess

import pytest

import oracle
import oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "ref_attn.c")).read()

MUTATIONS = {
    "causal_excludes_self": ("int hi = causal == 1 ? p : L - 1;", "int hi = causal == 1 ? p - 1 : L - 1;"),
    "noncausal_drops_last": ("int hi = causal == 1 ? p : L - 1;", "int hi = causal == 1 ? p : L - 2;"),
    "context_only_query_inside_row": ("int c = causal == 2 ? L : L - n;", "int c = L - n;"),
    "dense_key_row_shift": ("const uint16_t *kj = k + ((size_t)(cu_k[r] + j) * num_kv_heads",
                            "const uint16_t *kj = k + ((size_t)(cu_k[r] + j + (j > 0)) * num_kv_heads"),
    "dense_no_causal": ("            int hi = causal ? p : L - 1;\n            int lo = 0;\n            if (window_left >= 0) lo = p - window_left > 0 ? p - window_left : 0;\n            for (int h = 0; h < num_qo_heads; ++h) {\n                int hk = h / group;\n                const uint16_t *qv = q + ((size_t)t * num_qo_heads + h) * head_dim;\n                float *o = out + ((size_t)t * num_qo_heads + h) * head_dim;\n                float m = -INFINITY;",
                        "            int hi = L - 1;\n            int lo = 0;\n            if (window_left >= 0) lo = p - window_left > 0 ? p - window_left : 0;\n            for (int h = 0; h < num_qo_heads; ++h) {\n                int hk = h / group;\n                const uint16_t *qv = q + ((size_t)t * num_qo_heads + h) * head_dim;\n                float *o = out + ((size_t)t * num_qo_heads + h) * head_dim;\n                float m = -INFINITY;"),
    "empty_context_not_zero": ("for (int d = 0; d < head_dim; ++d) o[d] = 0.0f;\n                    if (lse)",
                               "for (int d = 0; d < head_dim; ++d) o[d] = 1.0f;\n                    if (lse)"),
    "window_one_short": ("lo = p - window_left > 0 ? p - window_left : 0;",
                          "lo = p - window_left + 1 > 0 ? p - window_left + 1 : 0;"),
    "window_ignored": ("if (window_left >= 0) lo", "if (window_left >= 1000000) lo"),
    "gqa_modulo_mapping": ("int hk = h / group;", "int hk = h % num_kv_heads;"),
    "k_v_swapped": ("size_t ko = cache_offset(page, 0, slot, hk,", "size_t ko = cache_offset(page, 1, slot, hk,"),
    "no_sm_scale": ("s[j] = sm_scale * dot;", "s[j] = dot;"),
    "unnormalised": ("float w = s[j] / l;", "float w = s[j];"),
    "lse_log2": ("m + logf(l)", "m + log2f(l)"),
    "lse_without_max": ("m + logf(l)", "logf(l)"),
    "slot_shift": ("int slot = p % page_size;\n            for (int hk",
                   "int slot = (p + 1) % page_size;\n            for (int hk"),
    "page_index_off_by_one": ("int64_t page = kv_indices[kv_indptr[r] + p / page_size];\n            if (page < 0 || page >= max_pages) { free",
                              "int64_t page = kv_indices[kv_indptr[r] + (p + 1) / page_size];\n            if (page < 0 || page >= max_pages) { free"),
    "row_length_ignores_last_page": ("return (npages - 1) * page_size + last_page_len[r];",
                                     "return npages * page_size;"),
    "append_one_late": ("int p = c + i;\n            int64_t page", "int p = c + i + 1;\n            int64_t page"),
    "append_v_into_k": ("memcpy(kv_layer + vo,", "memcpy(kv_layer + ko,"),
    "query_token_of_row_start": ("int t = qo_indptr[r] + i;\n            int p = c + i;\n            int hi",
                                 "int t = qo_indptr[r];\n            int p = c + i;\n            int hi"),
}


def _build(tmp_path, name, src):
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", str(c), "-o", str(so),
                    "-lm"], check=True)
    return oracle.load(str(so))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    assert SRC.count(old) >= 1, f"mutation anchor for {name} not found"
    lib = _build(tmp_path, name, SRC.replace(old, new))  # every occurrence (paged and dense paths)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib=lib)
        except (AssertionError, ValueError, IndexError) as e:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


# ---- the index oracle (oracle/plan_ref.py): mistakes planted in a copy of its source ----

import importlib.util  # noqa: E402

import plan_pins  # noqa: E402
from oracle import plan_ref  # noqa: E402

PLAN_SRC = open(plan_ref.__file__).read()

PLAN_MUTATIONS = {
    # context_only_views keeps the LAST pages of a row instead of the first
    "context_only_keeps_last_pages": ("new_i.extend(int(x) for x in kvi[kvp[r]: kvp[r] + keep])",
                                      "new_i.extend(int(x) for x in kvi[kvp[r + 1] - keep: kvp[r + 1]])"),
    # ... keeps one page too many when the context ends on a page boundary
    "context_only_extra_page": ("keep = -(-ctx // page_size)", "keep = ctx // page_size + 1 if ctx else 0"),
    # ... leaves the last page's fill as it was
    "context_only_fill_unchanged": ("new_l.append(last_page_len_of(ctx, page_size) if ctx > 0 else 0)",
                                    "new_l.append(int(last_page_len[r]) if ctx > 0 else 0)"),
    "append_slot_one_late": ("p = c + i\n            pages[qo[r] + i]", "p = c + i + 1\n            pages[qo[r] + i]"),
    "append_row_start_position": ("c = int(L[r]) - n\n", "c = 0\n"),
    "perm_prompt_rows_reversed": ("for r in prompt:\n        perm.extend", "for r in prompt[::-1]:\n        perm.extend"),
    "sink_row_keeps_pages": ("dec_kvi.append(int(sink_page))", "dec_kvi.extend(int(x) for x in kvi[kvp[r]: kvp[r + 1]])"),
}


@pytest.mark.parametrize("name", sorted(PLAN_MUTATIONS))
def test_plan_mutant_is_caught(name, tmp_path):
    old, new = PLAN_MUTATIONS[name]
    assert PLAN_SRC.count(old) == 1, f"mutation anchor for {name} not found"
    path = tmp_path / f"plan_ref_{name}.py"
    path.write_text(PLAN_SRC.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"plan_ref_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in plan_pins.ALL_PLAN_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError) as e:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"
