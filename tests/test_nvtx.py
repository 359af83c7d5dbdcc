"""NVTX ranges of the C-ABI calls, checked on the CPU with a recording NVTX tool.

Each call that enqueues GPU work (or waits for it) opens a range named after
itself in the domain "kvevict".  A small tool (tests/nvtx_recorder.c, loaded
through NVTX_INJECTION64_PATH as a profiler would be) logs the ranges of a child
process that calls every traced entry point with a null problem: each call
returns KV_ERR_INVALID_ARG before any CUDA work, but its range has already been
opened and closed, so this runs without a GPU.
"""
import json
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

TRACED = ["kv_score_attention", "kv_score_rescore", "kv_score", "kv_pool_scores", "kv_select_topk",
          "kv_head_budgets", "kv_block_scores", "kv_compact_blocks", "kv_evict_fused", "kv_compact",
          "kv_check_status", "kv_evict_host"]
UNTRACED = ["kv_score_workspace_size", "kv_select_workspace_size", "kv_make_offsets"]

CHILD = r"""
import ctypes, json, sys
sys.path.insert(0, sys.argv[1])
import kv_cache_eviction_split_gb300 as kv
lib = kv.load()
ints = (ctypes.c_size_t, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int)
rcs = {}
for name in json.loads(sys.argv[2]):
    fn = getattr(lib, name)
    args = [0 if t in ints else None for t in fn.argtypes]
    rcs[name] = int(fn(*args))
print(json.dumps(rcs))
"""


@pytest.fixture(scope="module")
def recorder(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    import kv_cache_eviction_split_gb300 as kv
    kv.build()
    inc = os.path.join(os.path.dirname(os.path.dirname(kv._build.nvcc())), "include")
    if not os.path.exists(os.path.join(inc, "nvtx3", "nvToolsExt.h")):
        pytest.skip("no NVTX 3 headers in the CUDA toolkit")
    out = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_recorder.so")
    subprocess.run([cc, "-shared", "-fPIC", "-O1", "-I", inc, os.path.join(HERE, "nvtx_recorder.c"),
                    "-o", out], check=True, capture_output=True)
    return out


def _run(recorder, tmp_path, names):
    log = str(tmp_path / "nvtx.log")
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder, KV_NVTX_LOG=log)
    res = subprocess.run([sys.executable, "-c", CHILD, ROOT, json.dumps(names)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    rcs = json.loads(res.stdout.strip().splitlines()[-1])
    lines = open(log).read().splitlines() if os.path.exists(log) else []
    return rcs, lines


def test_every_traced_call_opens_and_closes_its_range(recorder, tmp_path):
    import kv_cache_eviction_split_gb300 as kv
    rcs, lines = _run(recorder, tmp_path, TRACED)
    assert all(rcs[n] == kv.KV_ERR_INVALID_ARG for n in TRACED), rcs
    assert lines[0] == "domain kvevict"
    expected = []
    for n in TRACED:
        expected += ["push kvevict %s" % n, "pop kvevict"]
    assert lines[1:] == expected


def test_size_queries_open_no_range(recorder, tmp_path):
    rcs, lines = _run(recorder, tmp_path, UNTRACED)
    assert all(rc != 0 for rc in rcs.values())
    assert not any(line.startswith("push") for line in lines)
