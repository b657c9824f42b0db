"""Planted mistakes in the C oracle, on the CPU: do the pins catch them?

Each mutant is a copy of ``oracle/ep_oracle.c`` with one plausible slip: a wrong
operator, index, stride, loop order or bound, a dropped term or rounding, a
transposed operand. Each copy is compiled to its own library under a temporary
directory. The oracle's pins (``test_oracle_pins.py``) then run against it in a
child process, and at least one of them must fail on an assertion. The pins run
in a fixed order and the run stops at the first failure; every mutant keeps its
accesses in bounds on the inputs of the pins that run before the one that catches
it, so a crash would be a mistake in the mutant, not a catch. The unmutated source
must pass the same pin run, which shows that the runner itself works.

The mistakes are planted in a copy of the oracle only; the library under
``oracle/`` and the CUDA path are not touched.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")

# pins run in this order (fast first); the child stops at the first failure
PINS = [
    ("test_capacities", (4, 8, 8, 16, (16, 2, 64))),
    ("test_worked_example_dispatch", ()),
    ("test_worked_example_payload_and_combine", ()),
    ("test_fold_rounds_each_product_before_its_sum", ()),
    ("test_errors_flagged_and_pairs_dropped", ()),
    ("test_w1_is_a_stable_counting_sort_by_expert", ()),
    ("test_payload_rows_are_the_source_tokens", ()),
    ("test_combine_one_hot_weights_return_the_expert_row", ()),
    ("test_identity_experts_reproduce_a1", (1,)),
    ("test_combine_scales_exactly_with_weights", ()),
    ("test_weight_on_input_scaling_closed_forms", ()),
    ("test_agrs_worked_example_by_hand", ()),
    ("test_agrs_one_rank_is_the_single_fold", ()),
    ("test_agrs_drops_bad_pairs_like_the_router", ()),
    ("test_agrs_route_equals_two_stage_combine_of_the_all_to_all_route", (2, 24)),
    ("test_pagemode_two_stage_rounding_bounded", ()),
    ("test_combine_within_fp32_sum_bound_of_exact", (2, 32)),
    ("test_invariants_random_medium", ()),
    ("test_random_tiny_cases_agree_including_errors", ()),
    ("test_exhaustive_tiny_w2_e4_k2_t3", ()),
]

# (name, text in the source, replacement, which occurrence: an index, or None for all)
MUTANTS = [
    ("capacities: slots not clamped to e_local",
     "*slots = imin(K, e_local);", "*slots = K;", 0),
    ("route: destination by modulo",
     "int d = row[k] / e_local;", "int d = row[k] % W;", None),
    ("route: padding ids flagged as errors",
     "if (e < 0) continue;", "if (e < 0) { *err |= OR_ERR_EXPERT_ID; continue; }", 0),
    ("route: id E - 1 rejected (off by one)",
     "if (e >= E) { *err |= OR_ERR_EXPERT_ID; continue; }",
     "if (e >= E - 1) { *err |= OR_ERR_EXPERT_ID; continue; }", 0),
    ("route: repeated ids not dropped",
     "if (dup) { *err |= OR_ERR_DUPLICATE; continue; }", "if (0) { *err |= OR_ERR_DUPLICATE; continue; }", 0),
    ("route: slot numbered by token index, not compacted",
     "slot_on[d] = send_cnt[s * W + d]++;", "slot_on[d] = t; send_cnt[s * W + d]++;", 0),
    ("route: columns filled from the last one",
     "int col = used_cols[d]++;", "int col = S - 1 - used_cols[d]++;", 0),
    ("route: column stored as the local expert id",
     "send_eloc[at] = row[k] - d * e_local;", "send_eloc[at] = col;", 0),
    ("route: weight of the first pick for every column",
     "send_w[at] = weights[((size_t)s * Tm + t) * K + k];",
     "send_w[at] = weights[((size_t)s * Tm + t) * K + 0];", 0),
    ("exchange: counts not transposed",
     "recv_cnt[d * W + s] = send_cnt[s * W + d];", "recv_cnt[d * W + s] = send_cnt[d * W + s];", 0),
    ("deliver: source ranks walked in descending order",
     "for (int s = 0; s < W; ++s) {\n            for (int slot = 0; slot < recv_cnt[d * W + s]; ++slot) {",
     "for (int s = W - 1; s >= 0; --s) {\n            for (int slot = 0; slot < recv_cnt[d * W + s]; ++slot) {", 0),
    ("deliver: slots walked in descending order",
     "for (int slot = 0; slot < recv_cnt[d * W + s]; ++slot) {",
     "for (int slot = recv_cnt[d * W + s] - 1; slot >= 0; --slot) {", 0),
    ("pair rows: column taken as the top-k index",
     "int k = send_k[(((size_t)s * W + d) * Tm + slot) * S + c];", "int k = c;", 0),
    ("pack: row of the slot index instead of its token",
     "src_rows + ((size_t)s * Tm + t) * rb, rb);", "src_rows + ((size_t)s * Tm + slot) * rb, rb);", 0),
    ("deliver: rank indices transposed",
     "recv_x + (((size_t)d * W + s) * Tm + slot) * rb, rb);",
     "recv_x + (((size_t)s * W + d) * Tm + slot) * rb, rb);", 0),
    ("bf16 widening shifted by 15",
     "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;", 0),
    ("bf16 rounding truncates",
     "u += 0x7FFFu + lsb;", "u += 0u * lsb;", 0),
    ("bf16 rounding ties away from zero",
     "u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;", 0),
    ("combine: last top-k pick dropped",
     "for (int k = 0; k < K; ++k) {\n                int32_t f = pair_row[g * K + k];",
     "for (int k = 0; k < K - 1; ++k) {\n                int32_t f = pair_row[g * K + k];", 0),
    ("combine: weight index transposed",
     "float w = weights[g * K + k];\n                const uint16_t *x = rows",
     "float w = weights[(size_t)k * W * Tm + g];\n                const uint16_t *x = rows", 0),
    ("combine: weights ignored",
     "float p = w * bf16_to_f32(x[i]);\n                    acc[i] = acc[i] + p;",
     "float p = 0.0f * w + bf16_to_f32(x[i]);\n                    acc[i] = acc[i] + p;", 0),
    ("combine: rounds to bf16 after every add",
     "float p = w * bf16_to_f32(x[i]);\n                    acc[i] = acc[i] + p;",
     "float p = w * bf16_to_f32(x[i]);\n                    acc[i] = out_f32 ? acc[i] + p : bf16_to_f32(f32_to_bf16(acc[i] + p));", 0),
    ("all-gather route: expert owner by modulo",
     "if (!kept[k] || row[k] / e_local != d) continue;", "if (!kept[k] || row[k] % W != d) continue;", 0),
    ("all-gather route: per-rank output not rounded to bf16",
     "float y = bf16_to_f32(f32_to_bf16(yd[i]));", "float y = yd[i];", 0),
    ("all-gather route: bf16 reduce-scatter sums kept in fp32",
     "else acc[i] = bf16_to_f32(f32_to_bf16(acc[i] + y));", "else acc[i] = acc[i] + y;", 0),
    ("weight on input: weight not rounded to bf16 first",
     "float w = bf16_to_f32(f32_to_bf16(weights[g]));", "float w = weights[g];", 0),
    ("two-stage combine: partials not rounded to bf16",
     "float pr = bf16_to_f32(f32_to_bf16(part[i]));", "float pr = part[i];", 0),
    ("two-stage combine: destinations summed in descending order",
     "for (int d = 0; d < W; ++d) {\n                int slot = -1;",
     "for (int d = W - 1; d >= 0; --d) {\n                int slot = -1;", 0),
    ("combine: each product fused into its sum (one rounding per term)",
     "float p = w * bf16_to_f32(x[i]);\n                    acc[i] = acc[i] + p;",
     "double p = (double)w * (double)bf16_to_f32(x[i]);\n                    acc[i] = (float)((double)acc[i] + p);", 0),
    ("combine: top-k pairs folded in reverse order",
     "for (int k = 0; k < K; ++k) {\n                int32_t f = pair_row[g * K + k];",
     "for (int k = K - 1; k >= 0; --k) {\n                int32_t f = pair_row[g * K + k];", 0),
    ("two-stage combine: each product fused into the partial sum",
     "float p = bf16_to_f32(x[i]) * send_w[at];\n                        part[i] = part[i] + p;",
     "double p = (double)bf16_to_f32(x[i]) * (double)send_w[at];\n                        part[i] = (float)((double)part[i] + p);", 0),
    ("all-gather route: each product fused into the rank's sum",
     "float p = w * bf16_to_f32(a1[g * h + i]);\n                            yd[i] = yd[i] + p;",
     "double p = (double)w * (double)bf16_to_f32(a1[g * h + i]);\n                            yd[i] = (float)((double)yd[i] + p);", 0),
]

CHILD = r"""
import sys
root, libpath = sys.argv[1], sys.argv[2]
sys.path.insert(0, root)
import oracle.build
oracle.build.build = lambda *a, **k: libpath
from oracle import ref
ref._lib = None
import tests.test_oracle_pins as P
for name, args in PINS:
    try:
        getattr(P, name)(*args)
    except Exception as e:
        print("caught by", name, type(e).__name__)
        sys.exit(1)
print("all pins pass")
sys.exit(0)
""".replace("PINS", repr(PINS))


def _mutate(src, old, new, which):
    n = src.count(old)
    assert n >= 1, f"mutation site not found: {old!r}"
    if which is None:
        return src.replace(old, new)
    assert which < n
    at = -1
    for _ in range(which + 1):
        at = src.index(old, at + 1)
    return src[:at] + new + src[at + len(old):]


def _build(tmp, name, text):
    c = os.path.join(tmp, name + ".c")
    so = os.path.join(tmp, name + ".so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-w",
                    "-fPIC", "-shared", "-o", so, c], check=True)
    return so


def _run_pins(so):
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, so], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    return r.returncode, (r.stdout + r.stderr[-400:]).strip()


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("mutants"))
    src = open(SRC).read()
    jobs = [("original", src)]
    for i, (name, old, new, which) in enumerate(MUTANTS):
        jobs.append((name, _mutate(src, old, new, which)))
    libs = [(name, _build(tmp, f"m{i}", text)) for i, (name, text) in enumerate(jobs)]
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        outs = list(ex.map(lambda nl: _run_pins(nl[1]), libs))
    return {name: out for (name, _), out in zip(libs, outs)}


def test_the_unmutated_oracle_passes_the_pin_run(results):
    rc, log = results["original"]
    assert rc == 0, log


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(results, name):
    rc, log = results[name]
    assert rc == 1 and "caught by" in log, f"no pin caught the mutant: {log}"
