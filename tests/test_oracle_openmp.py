"""The -fopenmp build of the oracle (used only to time it on all host cores)
gives the same bits as the one-thread build: its pragmas split the row copies
and the combine into independent blocks, each output element computed by one
thread in the written order. Each build runs in its own child process."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import hashlib, json, sys
sys.path.insert(0, sys.argv[1])
from oracle import ref
from combine_ep_route_gb300 import workloads as wl
if sys.argv[2] == "omp":
    ref.use_openmp(True)
out = {}
for cfg, T in ((2, 64), (4, 32), (5, 16)):
    x = wl.make(wl.spec(cfg, T=T))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    rows = ref.dispatch_rows(m, x.a1)
    h = hashlib.sha256(rows.tobytes())
    h.update(ref.combine(m, x.topk_weights, rows).tobytes())
    h.update(ref.combine(m, x.topk_weights, rows, out_f32=True).tobytes())
    out[cfg] = h.hexdigest()
print(json.dumps(out))
"""


def _run(mode):
    env = dict(os.environ, OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, mode], capture_output=True, text=True,
                       timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_openmp_build_gives_identical_results():
    try:
        from oracle import build
        build.build(openmp=True)
    except subprocess.CalledProcessError:
        pytest.skip("no OpenMP in this compiler")
    assert _run("omp") == _run("one")
