"""GPU parity of the additive attention bias (sdpa_fwd_ex / sdpa_bwd_ex with
attn_bias and dbias) against the fp64 oracle.

The bias is read as torch's float attn_mask, added to the scaled scores
before the causal mask and the softmax (the forum thread's self-attention
with relative positional encoding; attn_bias support in the memory-efficient
kernel, PR 103704's priority-order discussion). Bounds as in the other
parity tests; dbias (= dS) within 3e-2 relative L2 per head.
"""

import numpy as np
import pytest
import torch

from scaled_dot_product_07_gb300 import workloads as W

from test_parity_gpu import compare, rel_l2, to_np

import oracle

pytestmark = pytest.mark.gpu


def run_case(sdpa, w, inputs, bias_cpu, layout="BHSE"):
    q, k, v, do = (W.to_layout(x, layout).cuda() for x in inputs)
    bias = W.padded_rows(bias_cpu.cuda())
    out, lse = sdpa.sdpa_fwd_ex(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset,
                                attn_bias=bias)
    dq, dk, dv, dbias = sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed,
                                         w.offset, attn_bias=bias, dbias=True)
    torch.cuda.synchronize()
    assert sdpa.sdpa_check_device() == 0
    return (out, lse, dq, dk, dv), dbias


def oracle_with_bias(w, inputs, bias_cpu, heads):
    q, k, v, do = (x.float().numpy().astype(np.float64) for x in inputs)
    b = bias_cpu.float().numpy().astype(np.float64)
    out, lse = oracle.sdpa_fwd(q, k, v, w.dropout_p, w.is_causal, None, w.seed, w.offset,
                               heads=heads, bias=b)
    dq, dk, dv, dbias = oracle.sdpa_bwd(do, q, k, v, out, lse, w.dropout_p, w.is_causal, w.seed,
                                        w.offset, None, heads=heads, bias=b)
    return (out, lse, dq, dk, dv), dbias


@pytest.mark.parametrize("D", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.0, 0.2])
@pytest.mark.parametrize("kind", ["random", "relpos"])
def test_bias_parity(cuda_lib, D, causal, p, kind):
    B, H = 2, 2
    Sq, Sk = (200, 330) if D != 96 else (333, 200)
    w = W.Workload("bias", B, H, Sq, Sk, D, causal, p, seed=31, offset=7, input_seed=1300 + D)
    inputs = W.draw_inputs(w)
    # a full [B, H, Sq, Sk] random bias; a relative-position bias shared by the batch
    shape = (B, H, Sq, Sk) if kind == "random" else (1, H, Sq, Sk)
    bias_cpu = W.draw_bias(shape, 40 + D, kind)
    gpu, gdb = run_case(cuda_lib, w, inputs, bias_cpu, "BSHE" if D == 96 else "BHSE")
    heads = [(b, h) for b in range(B) for h in range(H)]
    ref, rdb = oracle_with_bias(w, inputs, bias_cpu, heads)
    tag = f"bias {kind} D{D} c{int(causal)} p{p}"
    compare(gpu, ref, heads, tag)
    g = to_np(gdb)
    for b, h in heads:
        e = rel_l2(g[b, h], rdb[b, h])
        assert e <= 3e-2, f"{tag}: dbias head {(b, h)} rel L2 {e:.3g}"
    if causal:
        # positions hidden by the causal mask carry exactly zero gradient
        hidden = ~np.tril(np.ones((Sq, Sk), dtype=bool))
        assert (g[:, :, hidden] == 0).all()


def test_zero_bias_reproduces_the_unbiased_path(cuda_lib):
    w = W.Workload("bias0", 1, 2, 256, 256, 128, True, 0.1, seed=3, offset=1, input_seed=77)
    q, k, v, do = (x.cuda() for x in W.draw_inputs(w))
    zero = torch.zeros((1, 1, 256, 256), dtype=torch.bfloat16, device="cuda")
    out0, lse0, _, _ = cuda_lib.sdpa_fwd(q, k, v, 0.1, True, None, 3, 1)
    out1, lse1 = cuda_lib.sdpa_fwd_ex(q, k, v, 0.1, True, None, 3, 1, attn_bias=zero)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    # fixed-order dQ so that the two runs can be compared bit for bit
    g0 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out0, lse0, 0.1, True, 3, 1, deterministic=True)
    g1 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out1, lse1, 0.1, True, 3, 1, attn_bias=zero,
                              deterministic=True)
    torch.cuda.synchronize()
    for a, b in zip(g0, g1):
        assert torch.equal(a, b)
