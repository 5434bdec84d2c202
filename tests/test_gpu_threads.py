"""Launch-state caches under concurrency: the fused layer and the dense block
called for the first time in a fresh process from two host threads at once,
each on its own stream with its own plan and workspace, both checked against
the fp64 oracle; and, when a second GPU is present, the same calls with that
device current (shared-memory attributes and occupancy are per device)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading
import numpy as np, torch
sys.path.insert(0, ROOT)
import oracle, workloads as W
import sparse_graph_attention_head_gb300 as gat
from tests.parity import assert_bf16, assert_fp32

def fused(dev, seed, res):
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(dev)
    d = W.make_fused(seed=seed, n=3000, deg=W.zipf_degrees(np.random.default_rng(seed), 3000, dmax=900))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda a: t(a.view(np.int16)).view(torch.bfloat16)
    with torch.cuda.stream(s):
        rp, ci = t(d["row_ptr"]), t(d["col_idx"])
        q, k, v = bf(d["q"]), bf(d["k"]), bf(d["v"])
        plan = gat.Plan(rp, stream=s)
        out = gat.gat_fused_layer(rp, ci, q, k, v, d["scale"], plan=plan, stream=s)
    s.synchronize()
    o, c = oracle.fused_layer(d["row_ptr"], d["col_idx"], d["q"], d["k"], d["v"], d["H"], d["Dh"],
                              d["scale"], want_cond=True)
    assert_bf16(out.float().cpu().numpy().astype(np.float64), o, c, name=f"fused dev{dev} seed{seed}")
    res.append(("fused", dev, seed))

def dense(dev, seed, res):
    torch.cuda.set_device(dev)
    s = torch.cuda.Stream(dev)
    w = W.make_dense(seed=seed, B=37)
    names = ("nodes", "pair_feats", "edge_mask", "ln_w", "ln_b", "Wq", "Wk", "Wv", "W1", "b1", "W2",
             "b2", "Wout")
    with torch.cuda.stream(s):
        tt = {k: torch.from_numpy(np.ascontiguousarray(w[k])).to(dev) for k in names}
        out = gat.gat_dense_masked_attention(tt["nodes"], tt["pair_feats"], tt["edge_mask"],
                                             tt["ln_w"], tt["ln_b"], w["ln_eps"],
                                             *[tt[k] for k in names[5:]], H=w["H"], stream=s)
    s.synchronize()
    o, c = oracle.dense_block(w, want_cond=True)
    assert_fp32(out.cpu().numpy().astype(np.float64), o, c, name=f"dense dev{dev} seed{seed}")
    res.append(("dense", dev, seed))

devs = list(range(min(2, torch.cuda.device_count())))
res, errs = [], []
def run(fn, dev, seed):
    try:
        fn(dev, seed, res)
    except Exception as e:  # reported by the parent
        errs.append(repr(e))
for dev in devs:
    ths = [threading.Thread(target=run, args=(fn, dev, seed))
           for fn, seed in ((fused, 31), (fused, 32), (dense, 33), (dense, 34))]
    for th in ths:
        th.start()
    for th in ths:
        th.join()
print("results", sorted(res), "errors", errs)
sys.exit(1 if errs or len(res) != 4 * len(devs) else 0)
'''


def test_first_calls_from_two_host_threads_and_each_device():
    import __graft_entry__
    __graft_entry__.build()
    code = f"ROOT = {ROOT!r}\n" + CHILD
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert torch.cuda.device_count() >= 1
