"""Helpers shared by the GPU parity tests: host copies, error measures, the
library handle, and inputs drawn from the seeded workload generators."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from ragged_grouped_gemm_topk_gb300 import workloads as W


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip(f"needs sm_103 (found sm_{major}{minor})")
    from ragged_grouped_gemm_topk_gb300 import build
    build.build()   # no-op when up to date; the kernels must be the in-tree library


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 host copy of a bf16/fp32 tensor."""
    return t.detach().to("cpu").double().numpy()


def i64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").numpy().astype(np.int64)


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


# Tolerances stated for the hot path: BF16 / TF32 outputs within rel-L2 1e-2 of
# the float64 oracle, MXFP8 GEMMs within 5e-2; integers and codes bit-exact;
# routing weights within 1e-6 absolute.
TOL_BF16 = 1e-2
TOL_MXFP8 = 5e-2
TOL_W = 1e-6


def logits_dev(w: W.Workload) -> torch.Tensor:
    return torch.from_numpy(W.make_logits(w)).cuda()


def ragged_offsets(counts) -> torch.Tensor:
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return torch.from_numpy(off).cuda()
