"""The allocation-free gradient-norm entry point, muon_adamw_grad_norm_noalloc.

Some callers of this library cannot call cudaMalloc: a host application
whose own pool allocator takes all device memory at start-up and forbids
later allocations, or a latency-critical loop that cannot accept
cudaMalloc's implicit device-wide synchronisation. This entry point gives
them the global gradient norm and clip coefficient without allocating: its
scratch is one fixed device array inside the library. The test calls it
through the C ABI, twice in a row on different gradients, and compares each
result with the norm and clip coefficient that muon_adamw_step computes on
the same gradients, within the parity suite's norm tolerance (1e-5 relative).

This file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest

import workloads
from harness import NORM_TOL, GpuSide

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    from muon_adamw_hybrid_grad_gb300 import build

    build.build()
    import muon_adamw_hybrid_grad_gb300 as m

    m.load_library()
    return m


def test_noalloc_norm_matches_step_on_two_calls(mx):
    import torch

    w = workloads.get_workload("tiny")
    gpu = GpuSide(w, workloads.master_weights(w))
    try:
        cfg = gpu.opt.cfg
        grads = [g for g in gpu.G if g is not None]
        ptrs = [g.data_ptr() for g in grads]
        numels = [g.numel() for g in grads]
        dtypes = [mx.MA_DT_BF16 if g.dtype == torch.bfloat16 else mx.MA_DT_F32 for g in grads]
        out = torch.empty(2, dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        for step, scale in ((1, 1.0), (2, 0.25)):
            gpu.load_grads(workloads.gradients(w, step, scale=scale))
            out.fill_(-1.0)  # a call that wrote nothing would leave -1
            mx.muon_adamw_grad_norm_noalloc(ptrs, numels, dtypes, cfg.max_grad_norm, cfg.clip_eps,
                                            out.data_ptr(), stream)
            torch.cuda.synchronize()
            total_na, coef_na = out.tolist()
            total_ref = gpu.step(w.lr)  # the existing entry point, same gradients
            _, coef_ref = mx.muon_adamw_last_norm(gpu.opt.handle)
            assert math.isclose(total_na, total_ref, rel_tol=NORM_TOL), (step, total_na, total_ref)
            assert math.isclose(coef_na, coef_ref, rel_tol=NORM_TOL), (step, coef_na, coef_ref)
        # a third call on the same (step 2) gradients reproduces the second exactly
        out2 = torch.empty(2, dtype=torch.float32, device="cuda")
        mx.muon_adamw_grad_norm_noalloc(ptrs, numels, dtypes, cfg.max_grad_norm, cfg.clip_eps,
                                        out2.data_ptr(), stream)
        torch.cuda.synchronize()
        assert out2.tolist() == [total_na, coef_na]
    finally:
        gpu.close()


def test_noalloc_rejects_too_many_tensors(mx):
    import torch

    n = mx.MA_NOALLOC_MAX_TENSORS + 1
    g = torch.zeros(n, 4, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(2, dtype=torch.float32, device="cuda")
    with pytest.raises(mx.MuonAdamWError) as ei:
        mx.muon_adamw_grad_norm_noalloc([g[i].data_ptr() for i in range(n)], [4] * n, [mx.MA_DT_BF16] * n,
                                        1.0, 1e-6, out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == mx.MA_ERR_ARG
    assert str(mx.MA_NOALLOC_MAX_TENSORS) in str(ei.value)
    torch.cuda.synchronize()
    assert out.tolist() == [0.0, 0.0]
