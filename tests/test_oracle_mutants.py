"""The pins catch plausible mistakes.

Each case plants one mistake in a temporary copy of the oracle source (never
in the committed oracle; every occurrence of the anchor text is changed),
builds it on the CPU, and runs the pin suites against that library. The
suites must fail for every mutant.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

# (name, text in oracle.cpp, replacement)
MUTANTS = [
    ("unstable_sort",
     "std::stable_sort(gather_idx.begin(), gather_idx.end(),",
     "std::sort(gather_idx.begin(), gather_idx.end(),"),
    ("masked_keys_first",
     "? (int64_t)layer_id * El + id : E;",
     "? (int64_t)layer_id * El + id : -1;"),
    ("layer_offset_dropped",
     "? (int64_t)layer_id * El + id : E;",
     "? id : E;"),
    ("offset_off_by_one",
     "expert_offsets[i] = (int32_t)(i - group_start);",
     "expert_offsets[i] = (int32_t)(i - group_start + 1);"),
    ("gather_wrong_row",
     "token_data + (size_t)(g * row_stride),",
     "token_data + (size_t)(i * row_stride),"),
    ("scale_wrong_offset",
     ": token_data + (size_t)(g * row_stride + H);",
     ": token_data + (size_t)(g * row_stride + H - 4);"),
    ("token_id_not_looked_up",
     "token_out[i] = token_in ? token_in[g] : (int32_t)g;",
     "token_out[i] = token_in ? token_in[i] : (int32_t)g;"),
    ("tail_ids_not_minus_one",
     "token_out[i] = -1;",
     "token_out[i] = 0;"),
    ("masked_select_not_transposed",
     "if (routingMap[t * Eu + e] != 0) {\n                    if (pos < n) copy_elem(permuteProbs, pos, probs, t * Eu + e, probsDtype);",
     "if (routingMap[e * T + t] != 0) {\n                    if (pos < n) copy_elem(permuteProbs, pos, probs, e * T + t, probsDtype);"),
    ("padded_prob_index_mod",
     "copy_elem(permuteProbs, i, probs, v * Eu + i / capacity, probsDtype);",
     "copy_elem(permuteProbs, i, probs, v * Eu + i % capacity, probsDtype);"),
    ("weight_dropped",
     "if (has_probs) term = x * p;\n                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;\n            }\n        }\n    } else {",
     "term = x;\n                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;\n            }\n        }\n    } else {"),
    ("token_index_mod",
     "const int64_t t = i / topK;",
     "const int64_t t = i % T;"),
    ("zero_prob_not_skipped",
     "p = weight[i];\n                if (p == 0.0f) continue;",
     "p = weight[i];"),
    ("invalid_not_skipped",
     "if (v < 0 || v >= permutedRows) continue;",
     "if (v < 0) continue;"),
    ("padded_invalid_first",
     "sort_key[i] = (v >= 0 && v < T) ? v : T;  // invalid last",
     "sort_key[i] = (v >= 0 && v < T) ? v : -1;"),
    ("not_padded_invalid_last",
     "sort_key[i] = (v >= 0 && v < permutedRows) ? v : -1;  // invalid first",
     "sort_key[i] = (v >= 0 && v < permutedRows) ? v : permutedRows;"),
    ("permute_token_id_mod",
     "permuteTokenId[i] = padded ? sortedIndices[order[i]] : (int32_t)(order[i] / topK);",
     "permuteTokenId[i] = padded ? sortedIndices[order[i]] : (int32_t)(order[i] % topK);"),
    ("bf16_truncates",
     "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;",
     ""),
    ("half_ties_away",
     "if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u))) r += 1;",
     "if (rest >= 0x1000u) r += 1;"),
    ("accumulate_descending",
     "for (int64_t i = 0; i < n; ++i) {\n            const int64_t v = sortedIndices[i];\n            if (v < 0 || v >= permutedRows) continue;",
     "for (int64_t i = n - 1; i >= 0; --i) {\n            const int64_t v = sortedIndices[i];\n            if (v < 0 || v >= permutedRows) continue;"),
    ("context_session_micro_swapped",
     "sess[g] = (int32_t)(b / micro);",
     "sess[g] = (int32_t)(b % micro);"),
    ("context_flag_ignored",
     "const bool ready = needSchedule == 0 || flag == 1;",
     "const bool ready = true;"),
    ("context_block_layer_ignored",
     "key[g] = layer * El + id;",
     "key[g] = id;"),
    ("permute_copies_wrong_row",
     "if (r < n) std::memcpy(dst + (size_t)r * row_bytes, src + (size_t)t * row_bytes, row_bytes);",
     "if (r < n) std::memcpy(dst + (size_t)r * row_bytes, src + (size_t)(r % T) * row_bytes, row_bytes);"),
    ("permute_slot_off_by_one",
     "if (j < topK) sortedIndices[t * topK + j] = ro < n ? (int32_t)ro : -1;",
     "if (j < topK) sortedIndices[t * topK + j] = ro < n ? (int32_t)ro + 1 : -1;"),
    ("permute_pad_not_minus_one",
     "sortedIndices[e * capacity + r] = -1;",
     "sortedIndices[e * capacity + r] = 0;"),
    ("double_weighting",
     "if (has_probs) term = x * p;\n                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;\n            }\n        }\n    } else {",
     "if (has_probs) term = (x * p) * p;\n                acc[(size_t)(t * H + h)] = acc[(size_t)(t * H + h)] + term;\n            }\n        }\n    } else {"),
    ("update_modes_swapped",
     "(balanceMode == 0 ? localRankId : b) % count",
     "(balanceMode == 0 ? b : localRankId) % count"),
    ("update_count_column_read",
     "out = table[e * F + 1 + c];",
     "out = table[e * F + c];"),
    ("update_count_not_checked",
     "if (count >= 1 && count <= F - 1) {",
     "if (count >= 1) {"),
    ("update_threshold_strict",
     "(active && !(sc < threshold[k]))",
     "(active && sc > threshold[k])"),
    ("update_threshold_first_only",
     "(active && !(sc < threshold[k]))",
     "(active && !(sc < threshold[0]))"),
    ("update_active_ignored",
     "const bool active = activeMask ? activeMask[b] != 0 : true;",
     "const bool active = true;"),
    ("full_tail_rows_ignored",
     "const int64_t gathered = full_tail ? Y : U;",
     "const int64_t gathered = U;"),
    ("full_tail_last_row_dropped",
     "const int64_t gathered = full_tail ? Y : U;",
     "const int64_t gathered = full_tail ? Y - 1 : U;"),
    ("full_tail_ids_not_looked_up",
     "} else if (full_tail) {",
     "} else if (false) {"),
    ("full_tail_offsets_not_minus_one",
     "token_out[i] = token_in ? token_in[g] : (int32_t)g;\n            expert_offsets[i] = -1;",
     "token_out[i] = token_in ? token_in[g] : (int32_t)g;\n            expert_offsets[i] = 0;"),
    ("context_full_tail_rows_ignored",
     "if (!(i < U || (full_tail && g < n_src))) continue;",
     "if (!(i < U)) continue;"),
    ("context_full_tail_ids_not_looked_up",
     "} else if (full_tail && g < n_src) {",
     "} else if (false) {"),
]


PIN_FILES = ["test_oracle_pins.py", "test_oracle_context_pins.py", "test_oracle_permute_pins.py",
             "test_oracle_update_expert_pins.py", "test_oracle_full_tail_pins.py"]


def run_mutant(name, old, new, workdir):
    """Build the oracle with one planted mistake and run every pin suite on it.
    Returns (anchor found, pins failed, pytest tail)."""
    src = open(SRC).read()
    if src.count(old) < 1:
        return False, False, ""
    mutant_src = os.path.join(workdir, f"{name}.cpp")
    with open(mutant_src, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_library(mutant_src, os.path.join(workdir, f"lib{name}.so"))
    env = dict(os.environ, USC_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"]
                       + [os.path.join(HERE, f) for f in PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return True, r.returncode != 0, r.stdout[-2000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """name -> result. In a plain run every mutant is built and checked at
    once (independent compile + pytest processes); under pytest-xdist, whose
    workers each run this fixture, every test runs its own mutant only."""
    workdir = str(tmp_path_factory.mktemp("mutants"))
    by_name = {m[0]: m for m in MUTANTS}
    if os.environ.get("PYTEST_XDIST_WORKER"):
        return lambda name: run_mutant(*by_name[name], workdir)
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {name: ex.submit(run_mutant, *m, workdir) for name, m in by_name.items()}
        done = {name: f.result() for name, f in futs.items()}
    return lambda name: done[name]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, mutant_results):
    found, caught, tail = mutant_results(name)
    assert found, f"mutant {name}: anchor text not found"
    assert caught, f"mutant {name} passed every pin:\n{tail}"
