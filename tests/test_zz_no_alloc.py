"""moe_permute_noalloc, the dispatch entry point for callers that cannot
allocate device memory (it keeps its scratch in a fixed array inside the
library), called through the C ABI and compared with moe_permute, which takes
a caller workspace.  Two calls in a row with different inputs: the second must
not see anything the first left in the shared scratch.

Collected last on purpose (file name), so a run that stops at the first failure
has already run every other test.
"""

import ctypes as C

import pytest
import torch

from ragged_grouped_gemm_topk_gb300 import _lib
from ragged_grouped_gemm_topk_gb300 import binding as B
from ragged_grouped_gemm_topk_gb300 import workloads as W
from _parity import need_gpu

pytestmark = pytest.mark.gpu


def _p(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(x, idx, counts, E, quant):
    T, k = idx.shape
    d = x.shape[1]
    dev = x.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    dest = torch.empty(T, k, dtype=torch.int32, device=dev)
    src = torch.empty(T * k, dtype=torch.int32, device=dev)
    xp = torch.empty(T * k, d, dtype=torch.uint8 if quant else x.dtype, device=dev)
    xs = torch.empty(T * k, d // 32, dtype=torch.uint8, device=dev) if quant else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lib = _lib.load()
    rc = lib.moe_permute_noalloc(_p(x), B._dt(x), T, d, _p(idx), k, E, _p(counts), _p(offsets),
                                 _p(dest), _p(src), _p(xp), _lib.MOE_E4M3 if quant else B._dt(x),
                                 _p(xs), _p(status), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.MOE_OK, lib.moe_last_error_string()
    return dict(offsets=offsets, dest_row=dest, src_pair=src, xp=xp, xp_scales=xs), status


@pytest.mark.parametrize("quant", [False, True], ids=["copy", "mxfp8"])
def test_noalloc_matches_workspace_entry_point_twice(quant):
    need_gpu()
    cases = [W.BY_NAME["dsv3-bf16-train"].scaled(T=3000, d=256, name="big"),
             W.BY_NAME["qwen3-235b-bf16"].scaled(T=333, E=64, k=4, d=128, name="small"),
             # the largest expert count, and a problem that fills the scratch exactly
             # (ceil(65536 / 256) * 1024 = 262144 entries, the last one included)
             W.BY_NAME["tiny-fp32"].scaled(T=300, E=1024, k=8, d=32, name="E1024"),
             W.BY_NAME["tiny-fp32"].scaled(T=65536, E=1024, k=1, d=32, name="at-bound")]
    for w in cases:
        x = W.make_x(w, "cuda")
        lg = torch.from_numpy(W.make_logits(w)).cuda()
        idx, _, counts = B.moe_route_topk(lg, w.k)
        want = B.moe_permute(x, idx, counts, w.E, xp_dtype="mxfp8" if quant else None)
        got, status = _noalloc(x, idx, counts, w.E, quant)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for key in ("offsets", "dest_row", "src_pair"):
            assert torch.equal(got[key], want[key]), key
        assert torch.equal(got["xp"].view(torch.uint8), want["xp"].view(torch.uint8))
        if quant:
            assert torch.equal(got["xp_scales"], want["xp_scales"])
        # the same entry point through the Python binding
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        got2 = B.moe_permute_noalloc(x, idx, counts, w.E, xp_dtype="mxfp8" if quant else None, dev_status=st2)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        for key in ("offsets", "dest_row", "src_pair", "xp") + (("xp_scales",) if quant else ()):
            assert torch.equal(got2[key].view(torch.uint8), want[key].view(torch.uint8)), key


def test_noalloc_rejects_problems_beyond_its_scratch():
    need_gpu()
    T, k, E = 65536 + 256, 1, 1024            # ceil(T/256) * E = 263168 > 262144
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    x = torch.zeros(T, 32, dtype=torch.bfloat16, device="cuda")
    lib = _lib.load()
    buf = torch.empty(T * k, dtype=torch.int32, device="cuda")
    rc = lib.moe_permute_noalloc(_p(x), _lib.MOE_BF16, T, 32, _p(idx), k, E, _p(counts),
                                 _p(torch.empty(E + 1, dtype=torch.int32, device="cuda")),
                                 _p(buf), _p(buf), None, _lib.MOE_BF16, None, None, None)
    assert rc == _lib.MOE_ERR_WORKSPACE
    assert b"scratch" in lib.moe_last_error_string()
