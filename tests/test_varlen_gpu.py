"""GPU parity of packed variable-length batches (sdpa_fwd_varlen /
sdpa_bwd_varlen) against the fp64 oracle.

Reading (max_q / max_k of NVIDIA/Fuser issue 2278, "SdpaOpFwd / SdpaOpBwd
nodes"): sequence b is the top-left [len_q, len_k] block of a
[max_q, max_k] problem, so its dropout mask is that block of the padded
problem's mask. The oracle is run on exactly that padded problem -- zero
rows past each sequence and a -inf bias on the missing keys, which removes
them from the softmax -- and its rows and keys of the sequence are compared.
"""

import numpy as np
import pytest
import torch

import oracle
from scaled_dot_product_07_gb300 import workloads as W

from test_parity_gpu import GRAD_RTOL_L2, LSE_ATOL, OUT_ATOL, rel_l2, to_np

pytestmark = pytest.mark.gpu


def packed_inputs(lens_q, lens_k, H, D, seed):
    """Seeded packed bf16 tensors q, dout [total_q, H, D] and k, v [total_k, H, D]."""
    w = W.Workload("varlen", 1, H, sum(lens_q), sum(lens_k), D, False, 0.0, input_seed=seed)
    q, k, v, do = W.draw_inputs(w)  # logical [1, H, total, D]
    return tuple(x[0].permute(1, 0, 2).contiguous() for x in (q, k, v, do))


def oracle_sequence(q, k, v, do, b, H, Mq, Mk, lq, lk, p, causal, seed, offset):
    """Oracle results of sequence b: the top-left block of a [Mq, Mk] problem."""
    D = q.shape[2]
    scale = 1.0 / np.sqrt(D)
    res = {n: [] for n in ("out", "lse", "dq", "dk", "dv")}
    bias = np.zeros((Mq, Mk))
    bias[:, lk:] = -np.inf
    for h in range(H):
        qp, dop = np.zeros((Mq, D)), np.zeros((Mq, D))
        kp, vp = np.zeros((Mk, D)), np.zeros((Mk, D))
        qp[:lq], dop[:lq] = q[:, h], do[:, h]
        kp[:lk], vp[:lk] = k[:, h], v[:, h]
        out, lse = oracle.head_forward(qp, kp, vp, b, h, H, p, causal, scale, seed, offset, bias=bias)
        dq, dk, dv, _ = oracle.head_backward(dop, qp, kp, vp, out, lse, b, h, H, p, causal, scale,
                                             seed, offset, bias=bias)
        for n, x, m in (("out", out, lq), ("lse", lse, lq), ("dq", dq, lq), ("dk", dk, lk),
                        ("dv", dv, lk)):
            res[n].append(x[:m])
    return {n: np.stack(x, axis=1 if n != "lse" else 0) for n, x in res.items()}


def run_varlen(sdpa, lens_q, lens_k, Mq, Mk, H, D, p, causal, deterministic=False, seed=21, offset=4):
    q, k, v, do = packed_inputs(lens_q, lens_k, H, D, 4000 + D + sum(lens_q))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    gq, gk, gv, gdo = (x.cuda() for x in (q, k, v, do))
    out, lse, _, _ = sdpa.sdpa_fwd_varlen(gq, gk, gv, cu_q, cu_k, Mq, Mk, p, causal, None, seed, offset)
    dq, dk, dv = sdpa.sdpa_bwd_varlen(gdo, gq, gk, gv, out, lse, cu_q, cu_k, Mq, Mk, p, causal, seed,
                                      offset, deterministic=deterministic)
    torch.cuda.synchronize()
    assert sdpa.sdpa_check_device() == 0
    return (q, k, v, do), (out, lse, dq, dk, dv)


def check_against_oracle(inputs, gpu, lens_q, lens_k, Mq, Mk, H, p, causal, tag, seed=21, offset=4):
    q, k, v, do = (x.float().numpy().astype(np.float64) for x in inputs)
    out, lse, dq, dk, dv = (to_np(t) for t in gpu)
    oq = np.concatenate([[0], np.cumsum(lens_q)])
    ok = np.concatenate([[0], np.cumsum(lens_k)])
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        sq, sk = slice(oq[b], oq[b + 1]), slice(ok[b], ok[b + 1])
        if lq == 0 or lk == 0:
            continue
        ref = oracle_sequence(q[sq], k[sk], v[sk], do[sq], b, H, Mq, Mk, lq, lk, p, causal, seed,
                              offset)
        msg = f"{tag} seq {b} ({lq}x{lk})"
        assert np.abs(out[sq] - ref["out"]).max() <= OUT_ATOL, msg
        assert np.abs(lse[:, sq] - ref["lse"]).max() <= LSE_ATOL, msg
        for n, g in (("dq", dq[sq]), ("dk", dk[sk]), ("dv", dv[sk])):
            e = rel_l2(g, ref[n])
            assert e <= GRAD_RTOL_L2, f"{msg}: {n} rel L2 {e:.3g}"


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.0, 0.2])
def test_varlen_parity(cuda_lib, D, causal, p):
    # ragged lengths, a sequence without queries, lengths below the maxima
    lens_q, lens_k = [37, 0, 200, 129], [50, 10, 130, 300]
    Mq, Mk = 256, 320
    H = 2
    inputs, gpu = run_varlen(cuda_lib, lens_q, lens_k, Mq, Mk, H, D, p, causal)
    check_against_oracle(inputs, gpu, lens_q, lens_k, Mq, Mk, H, p, causal,
                         f"varlen D{D} c{int(causal)} p{p}")
    # a sequence without queries still owns its keys: their gradients are 0
    dk, dv = gpu[3], gpu[4]
    assert torch.count_nonzero(dk[50:60]) == 0 and torch.count_nonzero(dv[50:60]) == 0


def test_varlen_equals_the_fixed_length_call_when_all_lengths_match(cuda_lib):
    B, H, S, D = 3, 2, 200, 128
    lens = [S] * B
    inputs, gpu = run_varlen(cuda_lib, lens, lens, S, S, H, D, 0.1, True, seed=9, offset=2)
    q, k, v, do = (x.reshape(B, S, H, D).permute(0, 2, 1, 3).contiguous().cuda() for x in inputs)
    out, lse, _, _ = cuda_lib.sdpa_fwd(q, k, v, 0.1, True, None, 9, 2)
    torch.cuda.synchronize()
    assert torch.equal(gpu[0].reshape(B, S, H, D).permute(0, 2, 1, 3), out)
    assert torch.equal(gpu[1].reshape(H, B, S).permute(1, 0, 2), lse)


@pytest.mark.parametrize("D", [128, 200])
def test_varlen_deterministic_backward_is_reproducible(cuda_lib, D):
    lens_q, lens_k = [100, 260], [300, 90]
    runs = [run_varlen(cuda_lib, lens_q, lens_k, 260, 300, 2, D, 0.1, True, deterministic=True)
            for _ in range(2)]
    for a, b in zip(runs[0][1][2:], runs[1][1][2:]):
        assert torch.equal(a, b)
    check_against_oracle(runs[0][0], runs[0][1], lens_q, lens_k, 260, 300, 2, 0.1, True,
                         "varlen deterministic")


def test_varlen_sequence_without_keys(cuda_lib):
    lens_q, lens_k = [40, 30], [0, 70]
    inputs, gpu = run_varlen(cuda_lib, lens_q, lens_k, 64, 128, 2, 64, 0.0, False)
    out, lse, dq = gpu[0], gpu[1], gpu[2]
    assert torch.count_nonzero(out[:40]) == 0
    assert torch.isneginf(lse[:, :40]).all()
    assert torch.count_nonzero(dq[:40]) == 0
    check_against_oracle(inputs, gpu, lens_q, lens_k, 64, 128, 2, 0.0, False, "varlen no keys")
