"""dlo_op_gemm_noalloc: the GEMM entry point for callers that cannot allocate
device memory.  Its kernel scratch (the error word) lives in a static device
array inside the library.  Checked through the C ABI against dlo_op_gemm, the
entry point that takes caller-allocated scratch, on two calls in a row."""
import numpy as np
import pytest
import torch

from oracle import dit

dlo = pytest.importorskip("layerwise_weight_offload_slot_gb300")

pytestmark = pytest.mark.gpu


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def _rel(y, ref):
    y = y.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(y - ref) / np.linalg.norm(ref))


def test_noalloc_gemm_matches_allocating_entry_on_two_calls():
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(300, 272, 1152, dlo.EPI_BIAS), (2048, 1152, 1152, dlo.EPI_RESIDUAL)]
    for call, (M, N, K, epi) in enumerate(cases):
        g = np.random.default_rng(100 + call)
        A = _bf16(g.standard_normal((M, K)))
        W = _bf16(g.standard_normal((N, K)) * 0.05)
        b = _bf16(g.standard_normal(N) * 0.1)
        if epi == dlo.EPI_RESIDUAL:
            gate = torch.from_numpy(g.standard_normal((2, N)).astype(np.float32)).cuda()
            x0 = torch.from_numpy(g.standard_normal((M, N)).astype(np.float32)).cuda()
            ref, new = x0.clone(), x0.clone()
            args = (gate.data_ptr(), N, M // 2)
        else:
            ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            new = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
            args = (None, 0, 1)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dlo.dlo_op_gemm(A.data_ptr(), W.data_ptr(), dlo.DT_BF16, None, 0, b.data_ptr(), M, N, K,
                        epi, ref.data_ptr(), N, *args, err.data_ptr(), stream)
        dlo.dlo_op_gemm_noalloc(A.data_ptr(), W.data_ptr(), dlo.DT_BF16, None, 0, b.data_ptr(),
                                M, N, K, epi, new.data_ptr(), N, *args, stream)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        tol = 1e-5 if epi == dlo.EPI_RESIDUAL else 6e-3
        assert _rel(new, ref) <= tol
        # and both agree with the float64 oracle
        r = dit.linear(A.double().cpu().numpy(), W.double().cpu().numpy(), b.double().cpu().numpy())
        if epi == dlo.EPI_RESIDUAL:
            r = x0.double().cpu().numpy() + gate.double().cpu().numpy()[np.arange(M) // (M // 2)] * r
        y = new.double().cpu().numpy()
        assert np.linalg.norm(y - r) / np.linalg.norm(r) <= tol


def test_noalloc_gemm_rejects_bad_sizes():
    with pytest.raises(dlo.DloError):
        dlo.dlo_op_gemm_noalloc(16, 16, dlo.DT_BF16, None, 0, None, 10, 15, 16, 0, 16, 16, None, 0,
                                1, None)
