"""Debug mode (PKV_DEBUG in the environment): a compute call reports a device-side error bit itself.

The mode is read once per process, so each case runs in a child process of its own.  An out-of-pool
block id is the planted error: the decode kernel flags it (PKV_EFLAG_BLOCK_ID) and treats its keys as
absent, which in debug mode makes the call itself return PKV_ERR_BOUNDS (PkvError code -4), and
without the mode leaves the bit for check_errors.  A CUDA-graph capture is not checked (no
synchronisation inside a capture) and still works in the mode.
"""

import os
import subprocess
import sys

import pytest
import torch

import paged_kv_cache_rmsnorm_gb300 as pkv

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, torch
sys.path.insert(0, ROOT)
import paged_kv_cache_rmsnorm_gb300 as pkv
from paged_kv_cache_rmsnorm_gb300.graphs import DecodeGraph
from tests.gpu_helpers import GpuStep
from workloads import build_workload

pkv.init()
wl = build_workload("debug mode", "decode", 51, [599, 99], [1, 1], spare_blocks=1)
gs = GpuStep(wl)
gs.store()  # a clean call: returns normally in either mode
out = pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, gs.block_table, wl.max_seqlen_k, wl.scale)
bt = gs.block_table.clone()
bt[0, 1] = wl.num_blocks + 5  # an entry outside the pool
results = []
for name, call in (
        ("decode", lambda: pkv.attn_decode(gs.q, gs.kc, gs.vc, gs.context_lens, bt, wl.max_seqlen_k, wl.scale)),
        ("noalloc", lambda: pkv.attn_decode_noalloc(gs.q, gs.kc, gs.vc, gs.context_lens, bt, wl.max_seqlen_k,
                                                    wl.scale, torch.empty_like(gs.q)))):
    try:
        call()
        torch.cuda.synchronize()
        results.append(f"{name}:returned:{','.join(pkv.check_errors())}")
    except pkv.PkvError as e:
        results.append(f"{name}:raised:{e.code}:{','.join(pkv.check_errors()) or 'clear'}")
# graph capture of store + decode in the same process
g = DecodeGraph(gs.q, gs.k, gs.v, gs.positions, gs.slots, gs.wq, gs.wk, gs.kc, gs.vc, gs.context_lens, gs.block_table,
                wl.max_seqlen_k, wl.scale).capture()
g.replay()
torch.cuda.synchronize()
results.append("graph:ok:" + (",".join(pkv.check_errors()) or "clear"))
print("RESULTS " + " ".join(results))
""".replace("ROOT", repr(ROOT))


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.build()
    yield


def _run(debug: str | None) -> list[str]:
    env = dict(os.environ)
    env.pop("PKV_DEBUG", None)
    if debug is not None:
        env["PKV_DEBUG"] = debug
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULTS ")][-1]
    return line.split()[1:]


def test_debug_mode_reports_the_bad_block_at_the_call():
    res = _run("1")
    # both decode entry points return PKV_ERR_BOUNDS themselves; the bit is read and cleared with it
    assert res[0] == "decode:raised:-4:clear"
    assert res[1] == "noalloc:raised:-4:clear"
    assert res[2] == "graph:ok:clear"


@pytest.mark.parametrize("value", [None, "0"])
def test_without_debug_mode_the_bit_waits_for_check_errors(value):
    res = _run(value)
    assert res[0] == "decode:returned:block_id"
    assert res[1] == "noalloc:returned:block_id"
    assert res[2] == "graph:ok:clear"
