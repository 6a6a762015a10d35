"""Failure detection on the GPU without a fault: a bounded barrier wait that can never complete
gives up after its limit, records the timeout in a device error word and returns; the context
stays usable for a normal layer step afterwards."""
import time

import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth

from .gpu_helpers import BF16_TOL, LayerRun, Inputs, rel_fro, to_np

pytestmark = pytest.mark.gpu

TIMEOUT = 2  # MOE_DEVERR_TIMEOUT


def test_bounded_wait_gives_up_and_reports_timeout(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    limit_ns = 50_000_000  # 50 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.moe_selftest_wait_timeout(err, limit_ns)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == TIMEOUT
    assert elapsed >= limit_ns * 1e-9
    # sticky: a second expiry keeps the first code, a cleared word records again
    err.fill_(7)
    g.moe_selftest_wait_timeout(err, 2_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == 7


def test_context_usable_after_a_timeout(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g.moe_selftest_wait_timeout(err, 5_000_000)
    cfg = synth.CONFIGS["tiny"]
    inp = Inputs(cfg)
    run = LayerRun(inp)
    assert int(err.item()) == TIMEOUT
    assert run.layer.device_error() == 0
    ref = inp.oracle(backward=False)
    assert rel_fro(to_np(run.y), ref.y) < BF16_TOL


def test_gemm_waits_give_up_and_context_recovers(lib):
    """A GEMM kernel's own bounded waits: the FC2 forward grouped GEMM of a routed BF16 layer
    (CTA pairs) runs with its TMA producer issuing no loads, so the MMA and epilogue waits of
    both CTAs of every pair run out after the limit. The kernel records the timeout in the
    workspace error word, frees TMEM and returns; after the word is cleared, a full layer step
    on the same context matches the oracle."""
    cfg = synth.CONFIGS["tiny"]
    inp = Inputs(cfg)
    run = LayerRun(inp, backward=False)
    L = run.layer
    assert L.device_error() == 0
    limit_ns = 5_000_000  # 5 ms
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.moe_selftest_gemm_timeout(L.desc, L.ws, L.ws_bytes, run.w2, limit_ns)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert L.device_error() == TIMEOUT
    assert elapsed >= limit_ns * 1e-9
    g.moe_clear_error(L.desc, L.ws)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    run.run(backward=True)
    assert L.device_error() == 0
    ref = inp.oracle()
    assert rel_fro(to_np(run.y), ref.y) < BF16_TOL
    assert rel_fro(to_np(run.dx), ref.dx) < BF16_TOL
