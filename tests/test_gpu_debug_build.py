"""The MOE_DEBUG build on the GPU: its self-test check sets MOE_DEV_ASSERT (the
release build's compiles to nothing), and the layer's kernels run under every one
of its device-side checks (TMA coordinates, staging offsets, the router exchange)
with a clean status word and the oracle's results."""

import json
import os
import subprocess
import sys

import pytest
import torch

import ragged_grouped_gemm_topk_gb300 as moe_gpu
from _parity import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs in a child process with MOE_DEBUG=1, so the package loads the debug library.
CHILD = r"""
import json, sys
sys.path.insert(0, "tests")
import numpy as np, torch
import ragged_grouped_gemm_topk_gb300 as moe_gpu
from ragged_grouped_gemm_topk_gb300 import build, workloads as W, _lib
from oracle import moe as om
from _parity import f64, logits_dev, rel_l2
build.build(debug=True)
out = {"lib": _lib.lib_path()}
dbg, st = moe_gpu.binding.moe_debug_selftest()
torch.cuda.synchronize()
out["selftest"] = [bool(dbg), int(st.item())]
for name, dt in (("bf16-train", "dsv3-bf16-train"), ("mxfp8-train", "dsv3-mxfp8-train")):
    w = W.BY_NAME[dt].scaled(T=384, E=32, d=512, f=512, name=name)
    x, W1, W2, lg = W.make_x(w, "cuda"), W.make_w1(w, "cuda"), W.make_w2(w, "cuda"), logits_dev(w)
    layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype=w.dtype, renormalize=w.renormalize,
                             training=True)
    y = layer.forward(x, lg)
    layer.backward(W.make_dy(w, "cuda"), lg)
    torch.cuda.synchronize()
    ref = om.layer_forward(f64(x), lg.cpu().numpy(), f64(W1), f64(W2), w.k, mxfp8_operands=w.dtype == "mxfp8")
    out[name] = [int(layer.dev_status.item()), float(rel_l2(f64(y), ref["y"]))]
w = W.BY_NAME["dsv3-nvfp4"].scaled(T=300, E=16, d=512, f=512, name="nvfp4")
x, W1, W2, lg = W.make_x(w, "cuda"), W.make_w1(w, "cuda"), W.make_w2(w, "cuda"), logits_dev(w)
layer = moe_gpu.MoELayer(w.T, w.d, w.E, w.k, w.f, W1, W2, dtype="nvfp4", renormalize=w.renormalize)
layer.forward(x, lg)
torch.cuda.synchronize()
out["nvfp4"] = [int(layer.dev_status.item())]
# the router split over clusters of 4 (50 tokens, d = 2048) and 2 (T = 2500, d = 1024)
for T, d in ((50, 2048), (2500, 1024)):
    xr = W.make_matrix(T, d, seed=T, dtype=torch.bfloat16, device="cuda")
    Wr = W.make_matrix(64, d, seed=T + 1, dtype=torch.bfloat16, device="cuda", scale=d ** -0.5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, wt, counts, lgt = moe_gpu.moe_route_topk_gemm(xr, Wr, 8, True, want_logits=True, dev_status=st)
    torch.cuda.synchronize()
    ri, _, _ = om.route_topk(lgt.cpu().numpy(), 8, True)
    out["router_%d" % T] = [int(st.item()), bool((idx.cpu().numpy() == ri).all()),
                            float(rel_l2(lgt.cpu().double().numpy(), om.router_logits(f64(xr), f64(Wr))))]
print("RESULT " + json.dumps(out))
"""


def test_selftest_matches_the_loaded_build():
    """The release build's check compiles to nothing; the MOE_DEBUG build's (loaded
    when the environment sets MOE_DEBUG=1) sets MOE_DEV_ASSERT."""
    need_gpu()
    want = os.environ.get("MOE_DEBUG") == "1"
    dbg, st = moe_gpu.binding.moe_debug_selftest()
    torch.cuda.synchronize()
    assert dbg == want
    assert int(st.item()) == (moe_gpu.binding._lib.MOE_DEV_ASSERT if want else 0)


def test_debug_build_runs_the_path_clean():
    need_gpu()
    env = dict(os.environ, MOE_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    out = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1][7:])
    assert out["lib"].endswith(os.path.join("debug", "libmoe.so"))
    assert out["selftest"] == [True, moe_gpu.binding._lib.MOE_DEV_ASSERT]
    assert out["bf16-train"][0] == 0 and out["bf16-train"][1] < 1e-2
    assert out["mxfp8-train"][0] == 0 and out["mxfp8-train"][1] < 5e-2
    assert out["nvfp4"] == [0]
    for T in (50, 2500):
        st, same, err = out["router_%d" % T]
        assert st == 0 and same and err < 1e-5
