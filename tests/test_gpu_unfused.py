"""The unfused PyTorch baseline that bench.py times for context (separate
eager passes: RMSNorm, RoPE, blockwise scale and e4m3 cast, cache scatter)
against the oracle, at the same tolerances as the library's kernels, so the
context figure comes from a correct program."""
import os
import sys

import pytest

import workloads as wl
from gpu_cases import dsv4_parity, qk_parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [wl.QK_SMALL, wl.QK_LARGE], ids=lambda w: w.name)
def test_unfused_qk_matches_oracle(cuda_device, w, parity_log):
    rep = qk_parity(wl.make_qk_workload(w, device=cuda_device), slice_tokens=8192,
                    call=bench.unfused_qk)
    parity_log(rep)


@pytest.mark.parametrize("w", [wl.DSV4_DECODE, wl.DSV4_LARGE], ids=lambda w: w.name)
def test_unfused_dsv4_matches_oracle(cuda_device, w, parity_log):
    qrep, crep = dsv4_parity(wl.make_dsv4_workload(w, device=cuda_device), slice_tokens=1024,
                             call=bench.unfused_dsv4)
    assert crep.exp_mismatch_ties == 0
    parity_log(qrep, crep)
