"""sdpa_bwd_noalloc: the backward for callers that may not allocate.

Some callers cannot call cudaMalloc -- code that a host framework hands only
its input and output buffers, and loops where an allocation (which can
synchronise the device) is not acceptable. For them the library keeps a
fixed scratch array and sdpa_bwd_noalloc uses it in place of the caller's
workspace. This test calls that entry point through the C ABI twice in a
row, on two different problems, and checks each result against the
ordinary sdpa_bwd with its own workspace, within the gradient tolerance of
the parity tests. The file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

from scaled_dot_product_07_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GRAD_RTOL_L2 = 3e-2


def _rel_l2(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def _noalloc_through_c_abi(sdpa, dout, q, k, v, out, lse, p, causal, seed, offset, scale):
    lib = sdpa.load_library()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    descs = [sdpa._desc(t) for t in (dout, q, k, v, out, dq, dk, dv)]
    r = [ctypes.byref(d) for d in descs]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.sdpa_bwd_noalloc(r[0], r[1], r[2], r[3], r[4], ctypes.c_void_p(lse.data_ptr()),
                              float(p), int(causal), seed, offset, float(scale), r[5], r[6], r[7],
                              stream)
    assert st == 0, sdpa.sdpa_status_string(st)
    return dq, dk, dv


def test_noalloc_backward_matches_the_workspace_backward_twice_in_a_row(cuda_lib):
    sdpa = cuda_lib
    problems = [
        W.Workload("noalloc_a", 2, 12, 1024, 1024, 64, True, 0.1, seed=1234, offset=0, input_seed=21),
        W.Workload("noalloc_b", 1, 4, 700, 900, 128, False, 0.0, input_seed=22, layouts=("BSHE",)),
    ]
    for w in problems:
        need = sdpa.sdpa_bwd_workspace_size(w.B, w.H, w.Sq, w.Sk, w.D)
        assert 0 < need <= sdpa.NOALLOC_SCRATCH_BYTES
        layout = w.layouts[0]
        q, k, v, do = (W.to_layout(x, layout).cuda() for x in W.draw_inputs(w))
        scale = 1.0 / np.sqrt(w.D)
        out, lse, seed, off = sdpa.sdpa_fwd(q, k, v, w.dropout_p, w.is_causal, scale, w.seed, w.offset)
        ref = sdpa.sdpa_bwd(do, q, k, v, out, lse, w.dropout_p, w.is_causal, seed, off, scale)
        got = _noalloc_through_c_abi(sdpa, do, q, k, v, out, lse, w.dropout_p, w.is_causal, seed,
                                     off, scale)
        torch.cuda.synchronize()
        assert sdpa.sdpa_check_device() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            e = _rel_l2(g, r)
            assert e <= GRAD_RTOL_L2, f"{w.name} {name}: rel L2 {e:.3g}"


def test_noalloc_rejects_problems_larger_than_its_scratch(cuda_lib):
    sdpa = cuda_lib
    B, H, S, D = 8, 16, 4096, 128  # needs ~272 MB of workspace
    assert sdpa.sdpa_bwd_workspace_size(B, H, S, S, D) > sdpa.NOALLOC_SCRATCH_BYTES
    x = torch.empty(B, H, S, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    with pytest.raises(sdpa.SdpaError) as ei:
        sdpa.sdpa_bwd_noalloc(x, x, x, x, x, lse)
    assert ei.value.status == 6
