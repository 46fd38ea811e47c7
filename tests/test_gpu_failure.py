"""Failure detection on the GPU without faulting it.

A pipeline wait that can never complete must end with MOE_DEVERR_TIMEOUT and a kernel
that returns, leaving the context usable; the wait runs on a barrier phase that no
thread completes (nothing traps, nothing reads a bad address)."""

import time

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import PARITY_WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    moe.moe_selftest_wait_timeout(flags, 20_000_000)   # 20 ms
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    assert flags.item() == moe.MOE_DEVERR_TIMEOUT
    # The context still runs the layer correctly afterwards.
    w = PARITY_WORKLOADS["decode"]
    r = tl.run_forward(w, tl.to_device(make_inputs(w, seed=0)))
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    ref = oracle.routed_reference(None, w.k, w.gate, None, g["logits"])
    np.testing.assert_array_equal(g["topk_idx"], ref["idx"])


def test_selftest_rejects_bad_arguments():
    flags = torch.zeros((1,), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(flags, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(flags, 10**12)
