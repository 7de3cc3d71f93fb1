"""GPU tests of the sdpa_options extensions (sdpa_fwd_ex / sdpa_bwd_ex).

- rng state in device memory: a CUDA graph of forward + backward, captured
  once, replayed with two different {seed, offset} values written into the
  device buffer, gives bit for bit what the host-seeded calls give for the
  same values (graph-safe rng passing, "REDO of dropout support for mem eff
  #102038", pytorch PR 103704, Summary);
- batch / head split: a block at (batch_offset, head_offset) of a problem
  with total_heads heads draws exactly its slice of the whole problem's
  dropout mask, and its forward and backward match the oracle run on the
  whole problem's heads with their global indices (the head split of
  test_sdpa_loop_split, "DID loop split for SDPA", NVIDIA/Fuser PR 3711);
- deterministic backward: dq, dk, dv are bitwise identical across runs and
  within the parity bounds of the oracle;
- kernel events: the pair the caller passes is recorded around the forward
  kernel and around the backward's main kernel, without changing results.
"""

import numpy as np
import pytest
import torch

import oracle
from scaled_dot_product_07_gb300 import workloads as W

from test_parity_gpu import compare, oracle_heads, to_np

pytestmark = pytest.mark.gpu


def _inputs(B, H, Sq, Sk, D, input_seed):
    w = W.Workload("opts", B, H, Sq, Sk, D, True, 0.0, input_seed=input_seed)
    return W.draw_inputs(w)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_graph_replay_with_device_rng_matches_host_seeded_calls(cuda_lib, D):
    sdpa = cuda_lib
    B, H, Sq, Sk, p = 1, 2, 300, 300, 0.2
    q, k, v, do = (x.cuda() for x in _inputs(B, H, Sq, Sk, D, 321 + D))
    states = [(1234567, 0), (98765, 4096)]

    def host_seeded(seed, off):
        out, lse, _, _ = sdpa.sdpa_fwd(q, k, v, p, True, None, seed, off)
        dq, dk, dv = sdpa.sdpa_bwd(do, q, k, v, out, lse, p, True, seed, off)
        return out, lse, dq, dk, dv

    refs = [host_seeded(*s) for s in states]
    torch.cuda.synchronize()

    rng = torch.tensor(states[0], dtype=torch.int64, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(sdpa.sdpa_bwd_workspace_size(B, H, Sq, Sk, D), dtype=torch.uint8, device="cuda")

    def step():
        sdpa.sdpa_fwd_ex(q, k, v, p, True, rng_state=rng, out=out, lse=lse)
        sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, p, True, rng_state=rng, dq=dq, dk=dk, dv=dv,
                         workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # outside capture first
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for s, ref in zip(states, refs):
        rng.copy_(torch.tensor(s, dtype=torch.int64))
        g.replay()
        torch.cuda.synchronize()
        for name, a, b in zip(("out", "lse", "dq", "dk", "dv"), (out, lse, dq, dk, dv), ref):
            assert torch.equal(a, b), f"{name} differs from the host-seeded call for {s}"
    assert sdpa.sdpa_check_device() == 0
    assert not torch.equal(refs[0][0], refs[1][0])  # the two states drop different weights


@pytest.mark.parametrize("B,H,Sq,Sk,b0,h0,Bs,Hs", [
    (2, 6, 37, 70, 1, 2, 1, 3), (3, 4, 130, 129, 0, 1, 2, 2), (2, 3, 64, 64, 1, 0, 1, 3)])
def test_shard_mask_is_the_slice_of_the_whole_mask(cuda_lib, B, H, Sq, Sk, b0, h0, Bs, Hs):
    p, seed, off = 0.3, 2024, 17
    whole = oracle.keep_mask(B, H, Sq, Sk, p, seed, off)
    part = cuda_lib.sdpa_dropout_mask_debug_ex(Bs, Hs, Sq, Sk, p, seed, off, batch_offset=b0,
                                               head_offset=h0, total_heads=H)
    assert np.array_equal(part.cpu().numpy().astype(bool), whole[b0:b0 + Bs, h0:h0 + Hs])
    # the same block keyed from device memory
    rng = torch.tensor([seed, off], dtype=torch.int64, device="cuda")
    part2 = cuda_lib.sdpa_dropout_mask_debug_ex(Bs, Hs, Sq, Sk, p, 0, 0, rng_state=rng,
                                                batch_offset=b0, head_offset=h0, total_heads=H)
    assert torch.equal(part, part2)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_sharded_call_matches_the_oracle_on_global_heads(cuda_lib, D, causal):
    B, H, Sq, Sk, p = 2, 4, 200, 330, 0.25
    w = W.Workload("shard", B, H, Sq, Sk, D, causal, p, seed=77, offset=5, input_seed=900 + D)
    inputs = W.draw_inputs(w)
    b0, h0, Bs, Hs = 1, 1, 1, 2
    q, k, v, do = (x[b0:b0 + Bs, h0:h0 + Hs].contiguous().cuda() for x in inputs)
    kw = dict(batch_offset=b0, head_offset=h0, total_heads=H)
    out, lse = cuda_lib.sdpa_fwd_ex(q, k, v, p, causal, None, w.seed, w.offset, **kw)
    dq, dk, dv = cuda_lib.sdpa_bwd_ex(do, q, k, v, out, lse, p, causal, w.seed, w.offset, **kw)
    torch.cuda.synchronize()
    assert cuda_lib.sdpa_check_device() == 0
    heads = [(b0 + b, h0 + h) for b in range(Bs) for h in range(Hs)]
    ref = oracle_heads(w, inputs, heads)
    # place the shard's results at its global position
    full = []
    for t, shape in ((out, (B, H, Sq, D)), (lse, (B, H, Sq)), (dq, (B, H, Sq, D)),
                     (dk, (B, H, Sk, D)), (dv, (B, H, Sk, D))):
        z = torch.zeros(shape, dtype=t.dtype)
        z[b0:b0 + Bs, h0:h0 + Hs] = t.cpu()
        full.append(z)
    compare(full, ref, heads, f"shard D{D} causal{int(causal)}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("p", [0.0, 0.2])
@pytest.mark.parametrize("Sq,Sk", [(300, 460), (460, 200)])
def test_deterministic_backward_is_reproducible_and_matches_the_oracle(cuda_lib, D, causal, p,
                                                                       Sq, Sk):
    w = W.Workload("det", 1, 3, Sq, Sk, D, causal, p, seed=11, offset=3,
                   input_seed=500 + Sq + Sk + D)
    inputs = W.draw_inputs(w)
    q, k, v, do = (x.cuda() for x in inputs)
    out, lse, _, _ = cuda_lib.sdpa_fwd(q, k, v, p, causal, None, w.seed, w.offset)
    runs = [cuda_lib.sdpa_bwd_ex(do, q, k, v, out, lse, p, causal, w.seed, w.offset,
                                 deterministic=True) for _ in range(3)]
    torch.cuda.synchronize()
    assert cuda_lib.sdpa_check_device() == 0
    for r in runs[1:]:
        for a, b in zip(r, runs[0]):
            assert torch.equal(a, b)
    heads = [(0, h) for h in range(w.H)]
    ref = oracle_heads(w, inputs, heads)
    compare((out, lse) + tuple(runs[0]), ref, heads, f"det D{D} c{int(causal)} p{p} {Sq}x{Sk}")
    # the default (reduce-add) path agrees with it up to summation order
    dq_a, _, _ = cuda_lib.sdpa_bwd(do, q, k, v, out, lse, p, causal, w.seed, w.offset)
    a, b = to_np(dq_a), to_np(runs[0][0])
    assert np.linalg.norm(a - b) <= 1e-2 * max(np.linalg.norm(b), 1e-30)


def test_kernel_events_bracket_the_main_kernels(cuda_lib):
    """kernel_events: the library records the pair around the forward kernel
    and around the backward's main kernel; the results are those of the plain
    calls, and each bracketed time is positive and inside its whole call."""
    sdpa = cuda_lib
    B, H, S, D, p = 2, 4, 1024, 128, 0.1
    q, k, v, do = (x.cuda() for x in _inputs(B, H, S, S, D, 77))
    out0, lse0, _, _ = sdpa.sdpa_fwd(q, k, v, p, True, None, 5, 8)
    dq0, dk0, dv0 = sdpa.sdpa_bwd(do, q, k, v, out0, lse0, p, True, 5, 8)
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    for e in ev:
        e.record(st)  # creates the CUDA events
    ev[0].record(st)
    out, lse = sdpa.sdpa_fwd_ex(q, k, v, p, True, None, 5, 8, kernel_events=(ev[1], ev[2]))
    ev[3].record(st)
    ev[4].record(st)
    dq, dk, dv = sdpa.sdpa_bwd_ex(do, q, k, v, out, lse, p, True, 5, 8,
                                  kernel_events=(ev[5], ev[6]))
    ev[7].record(st)
    torch.cuda.synchronize()
    assert sdpa.sdpa_check_device() == 0
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    a, b = to_np(dq), to_np(dq0)
    assert np.linalg.norm(a - b) <= 1e-2 * max(np.linalg.norm(b), 1e-30)
    fwd_k, fwd_all = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    bwd_k, bwd_all = ev[5].elapsed_time(ev[6]), ev[4].elapsed_time(ev[7])
    assert 0.0 < fwd_k <= fwd_all
    assert 0.0 < bwd_k < bwd_all  # the backward's preprocess and dQ kernels are outside
    with pytest.raises(ValueError):
        sdpa.sdpa_fwd_ex(q, k, v, p, True, kernel_events=(torch.cuda.Event(enable_timing=True),
                                                          ev[2]))
