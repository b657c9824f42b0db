"""The benchmark's measurement arithmetic, checked on the CPU against counts
taken independently from the oracle's routing: the algorithmic bytes that the
roofline divides by, the all-gather / reduce-scatter byte count, the DRAM
traffic lookup and the variant bookkeeping."""
import argparse

import numpy as np
import pytest

import bench
from combine_ep_route_gb300 import workloads as wl
from oracle import ref


@pytest.mark.parametrize("cfg,over", [(1, {}), (2, {}), (3, {"T": 96}), (4, {"T": 40}), (5, {"T": 20})])
def test_algorithmic_bytes_from_the_oracles_routing(cfg, over):
    s = wl.spec(cfg, **over)
    x = wl.make(s, num_tokens=np.maximum(s.T - np.arange(s.W) % 5, 0).astype(np.int32))
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    # pairs = delivered rows; routed tokens = tokens holding at least one slot
    n_pairs = int(m.expert_num_tokens.sum())
    n_routed = len({(si, int(t)) for si in range(s.W) for d in range(s.W)
                    for t in m.send_tok[si, d][:m.send_cnt[si, d]]})
    bx, bp = 2 * s.h, sum(x.extra_row_bytes)
    disp, comb = bench.algorithmic_bytes(x)
    assert disp == (bx + bp) * (n_routed + n_pairs)
    assert comb == bx * n_pairs + 2 * s.h * int(x.num_tokens.sum())
    # fp32 output and a narrower dispatched row (quantised payloads)
    _, comb32 = bench.algorithmic_bytes(x, out_bytes_per_elem=4)
    assert comb32 == bx * n_pairs + 4 * s.h * int(x.num_tokens.sum())
    d8, _ = bench.algorithmic_bytes(x, x_row_bytes=s.h, extra_bytes=64)
    assert d8 == (s.h + 64) * (n_routed + n_pairs)


def test_agrs_bytes_by_brute_force():
    s = wl.spec(2, T=48)
    x = wl.make(s, num_tokens=np.array([48, 10, 0, 48, 7, 30, 48, 1], np.int32))
    parts, n_local = bench.agrs_bytes(x)
    e_local = s.E // s.W
    want_local, n_tok = 0, 0
    for r in range(s.W):
        for t in range(int(x.num_tokens[r])):
            n_tok += 1
            ranks = {int(e) // e_local for e in x.topk_ids[r, t] if e >= 0}
            want_local += len(ranks)
    assert n_local == want_local
    row, meta = 2 * s.h, 8 * s.K
    assert parts["gather"] == (row + meta) * n_tok * (1 + s.W)
    assert parts["experts"] == s.W * n_tok * meta + want_local * row + s.W * n_tok * row
    assert parts["reduce_scatter"] == s.W * n_tok * row + s.W * s.T * row


def test_traffic_lookup_follows_the_kernel_sources(tmp_path, monkeypatch):
    src = bench.kernel_source_hash("dispatch_fused")
    f = tmp_path / "traffic.txt"
    f.write_text("# comment\n"
                 f"kernel=dispatch_fused config=3 source={src} bytes_per_launch=123\n"
                 "kernel=combine config=3 source=0000000000000000 bytes_per_launch=456\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_for("dispatch_fused", 3) == 123.0
    assert bench.traffic_for("dispatch_fused", 2) is None      # another workload
    assert bench.traffic_for("combine", 3) is None             # taken on other sources
    # a kernel's hash covers its own translation unit, not another kernel's
    assert bench.kernel_source_hash("dispatch_fused") != bench.kernel_source_hash("combine")
    assert bench.kernel_source_hash("agrs_gather") == bench.kernel_source_hash("agrs_reduce")


def test_source_key_ignores_comments_and_layout_only():
    code = 'int f(int a) {\n    return a + 1;  // one more\n}\nconst char *s = "x // y";\n'
    same = '/* doc */ int f(int a)\n{ return a + 1; }\n// trailing\nconst char *s = "x // y";'
    assert bench.code_tokens(code) == bench.code_tokens(same)
    assert bench.code_tokens(code) != bench.code_tokens(code.replace("a + 1", "a + 2"))
    assert bench.code_tokens(code) != bench.code_tokens(code.replace('"x // y"', '"x /* y"'))
    assert bench.code_tokens("char c = '\\''; int b; // z") == "char c = '\\''; int b;"


def test_traffic_only_for_the_unchanged_named_workload(tmp_path, monkeypatch):
    src = bench.kernel_source_hash("dispatch_fused")
    f = tmp_path / "traffic.txt"
    f.write_text(f"kernel=dispatch_fused config=3 source={src} bytes_per_launch=123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))

    def args(**kw):
        d = dict(config=3, tokens_per_rank=None, experts=None, hidden=None, top_k=None)
        d.update(kw)
        return argparse.Namespace(**d)
    a = args()
    assert bench.traffic_config(a, bench.workload_spec(a)) == 3
    assert bench.traffic_for("dispatch_fused", bench.traffic_config(a, bench.workload_spec(a))) == 123.0
    # a smaller case of the same shape, or a variant, moves other bytes
    for over in (dict(tokens_per_rank=256), dict(experts=64), dict(hidden=2048), dict(top_k=4)):
        a = args(**over)
        assert bench.traffic_config(a, bench.workload_spec(a)) is None
    a = args()
    assert bench.traffic_config(a, bench.workload_spec(a), {"x_dtype": "fp8"}) is None
    assert bench.traffic_for("dispatch_fused", None) is None


def test_variant_bookkeeping():
    base = argparse.Namespace(x_dtype="bf16", weight_on_input=False, ragged=False, zero_pad=False)
    assert bench.variant_of(base) == {}
    v = bench.variant_of(argparse.Namespace(x_dtype="fp8", weight_on_input=True, ragged=True, zero_pad=True))
    assert v["x_dtype"] == "fp8" and v["weight_on_input"] and v["zero_pad"] and "ragged" in v


def test_cpu_baseline_all_cores_replicas():
    r = bench.cpu_baseline_all_cores(1, budget_s=0.5, bytes_per_replica=1 << 28)
    assert r is not None and r["value"] > 0 and r["cores"] >= 1
    assert r["unit"] == bench.UNIT and "replicas" in r["sample"]


def test_cpu_baseline_all_cores_reports_none_when_a_replica_fails():
    import time
    t0 = time.monotonic()
    assert bench.cpu_baseline_all_cores(99, budget_s=0.5, bytes_per_replica=1 << 28) is None   # no workload 99
    assert time.monotonic() - t0 < 120


def _run_bench(*argv, env=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    e = dict(os.environ, **(env or {}))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), *argv], capture_output=True,
                       text=True, timeout=300, env=e, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    (d,) = _run_bench("--impl", "reference", "--config", "1", "--steps", "3", "--warmup", "1")
    assert d["impl"] == "reference" and d["steps"] == 3 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny-w2-e8-k2-t16-h128"
    # the whole run fits the budget, so every step is the full workload
    assert d["config"]["tokens_per_rank"] == 16 and "full workload" in d["cpu_baseline"]["sample"]


def test_reference_arm_prints_nothing_on_other_ranks():
    assert _run_bench("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "1",
                      env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}) == []
