"""The allocation-free gradient-norm entry point, muon_adamw_grad_norm_noalloc.

Some callers of this library cannot call cudaMalloc: a host application
whose own pool allocator takes all device memory at start-up and forbids
later allocations, or a latency-critical loop that cannot accept
cudaMalloc's implicit device-wide synchronisation. This entry point gives
them the global gradient norm and clip coefficient without allocating: its
scratch is one fixed device array inside the library. The test calls it
through the C ABI, twice in a row on different gradients, and compares each
result with the norm and clip coefficient that muon_adamw_step computes on
the same gradients and with the fp64 oracle's, within the parity suite's
norm tolerance (1e-5 relative). A second case gives it more 64 Ki-element
chunks than the reduction has blocks (so blocks walk several chunks across
tensors), bf16 and fp32 gradients, empty tensors and a pointer that is not
16-byte aligned, and checks max_norm <= 0 (no clipping).

This file is named so that pytest collects it last.
"""
import math

import pytest

import oracle
import workloads
from harness import NORM_TOL, GpuSide
from workloads import TensorSpec

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
            host = workloads.gradients(w, step, scale=scale)
            gpu.load_grads(host)
            total_orc = oracle.global_grad_norm([g for g in host if g is not None])
            coef_orc = oracle.clip_coefficient(total_orc, cfg.max_grad_norm, cfg.clip_eps)
            out.fill_(-1.0)  # a call that wrote nothing would leave -1
            mx.muon_adamw_grad_norm_noalloc(ptrs, numels, dtypes, cfg.max_grad_norm, cfg.clip_eps,
                                            out.data_ptr(), stream)
            torch.cuda.synchronize()
            total_na, coef_na = out.tolist()
            total_ref = gpu.step(w.lr)  # the existing entry point, same gradients
            _, coef_ref = mx.muon_adamw_last_norm(gpu.opt.handle)
            assert math.isclose(total_na, total_ref, rel_tol=NORM_TOL), (step, total_na, total_ref)
            assert math.isclose(coef_na, coef_ref, rel_tol=NORM_TOL), (step, coef_na, coef_ref)
            assert math.isclose(total_na, total_orc, rel_tol=NORM_TOL), (step, total_na, total_orc)
            assert math.isclose(coef_na, coef_orc, rel_tol=NORM_TOL), (step, coef_na, coef_orc)
        # a third call on the same (step 2) gradients reproduces the second exactly
        out2 = torch.empty(2, dtype=torch.float32, device="cuda")
        mx.muon_adamw_grad_norm_noalloc(ptrs, numels, dtypes, cfg.max_grad_norm, cfg.clip_eps,
                                        out2.data_ptr(), stream)
        torch.cuda.synchronize()
        assert out2.tolist() == [total_na, coef_na]
    finally:
        gpu.close()


def test_noalloc_many_chunks_mixed_tensors(mx):
    import torch

    # 52 bf16 matrices (48 of 1024 x 1024, 4 of 4096 x 1024: 1016 chunks of
    # 64 Ki elements, more than the 4 x SMs blocks of the reduction), an
    # unaligned bf16 vector, fp32 vectors with ragged chunk tails, and two
    # empty tensors: 58 tensors
    shapes = [(1024, 1024)] * 48 + [(4096, 1024)] * 4
    wb = workloads.custom_workload("na_bf16", [TensorSpec(f"m{k}", s, rank8=True) for k, s in enumerate(shapes)] +
                                   [TensorSpec("u", (300001,))], grad_dtype="bf16")
    wf = workloads.custom_workload("na_f32", [TensorSpec(f"v{k}", (n,)) for k, n in
                                              enumerate((1000, 65537, 200003))], grad_dtype="fp32")
    dev = torch.device("cuda")
    out = torch.empty(2, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    keep = []
    for step in (1, 2):
        hb, hf = workloads.gradients(wb, step), workloads.gradients(wf, step)
        ptrs, numels, dtypes = [], [], []
        for g in hb[:-1]:
            t = torch.from_numpy(g).to(dev).to(torch.bfloat16)
            keep.append(t)
            ptrs.append(t.data_ptr()), numels.append(t.numel()), dtypes.append(mx.MA_DT_BF16)
        u = torch.zeros(hb[-1].size + 1, dtype=torch.bfloat16, device=dev)  # element 1 on: 2-byte aligned only
        u[1:].copy_(torch.from_numpy(hb[-1]).to(dev).to(torch.bfloat16))
        keep.append(u)
        ptrs.append(u.data_ptr() + 2), numels.append(hb[-1].size), dtypes.append(mx.MA_DT_BF16)
        for g in hf:
            t = torch.from_numpy(g).to(dev)
            keep.append(t)
            ptrs.append(t.data_ptr()), numels.append(t.numel()), dtypes.append(mx.MA_DT_F32)
        e = torch.zeros(4, dtype=torch.float32, device=dev)
        keep.append(e)
        for p in (e.data_ptr(), 0):  # empty tensors: numel 0, with a valid pointer and with NULL
            ptrs.append(p), numels.append(0), dtypes.append(mx.MA_DT_F32)
        assert len(ptrs) == 58
        total_orc = oracle.global_grad_norm(hb + hf)
        for max_norm in (1.0, 0.0, -1.0):
            out.fill_(-1.0)
            mx.muon_adamw_grad_norm_noalloc(ptrs, numels, dtypes, max_norm, 1e-6, out.data_ptr(), stream)
            torch.cuda.synchronize()
            total, coef = out.tolist()
            assert math.isclose(total, total_orc, rel_tol=NORM_TOL), (step, max_norm, total, total_orc)
            want = oracle.clip_coefficient(total_orc, max_norm, 1e-6)
            assert math.isclose(coef, want, rel_tol=NORM_TOL), (step, max_norm, coef, want)
        assert total_orc > 1.0  # the max_norm = 1 calls clipped
        keep.clear()


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
