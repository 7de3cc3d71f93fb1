"""Pins of the CPU oracle against things other than itself.

Each test ties one part of the oracle to a closed form worked by hand, an
invariant of the mathematics, a library routine that computes a special
case, central finite differences, or the statistics of the mask. Together
they are chosen so that a dropped term, a wrong sign, a transposed operand,
an off-by-one causal mask, a missing 1/(1-p) or a misplaced Philox word
fails at least one of them.
"""

import ctypes
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import philox

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- golden

def test_closed_form_cases():
    """Hand-derived forward and backward values (tests/golden)."""
    with open(os.path.join(HERE, "golden", "closed_form_cases.json")) as f:
        fx = json.load(f)
    for c in fx["cases"]:
        q, k, v, do = (np.array(c[n])[None, None] for n in ("q", "k", "v", "dout"))
        out, lse = oracle.sdpa_fwd(q, k, v, 0.0, c["is_causal"], c["scale"])
        np.testing.assert_allclose(out[0, 0], c["out"], rtol=0, atol=1e-13, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], c["lse"], rtol=0, atol=1e-13, err_msg=c["name"])
        dq, dk, dv = oracle.sdpa_bwd(do, q, k, v, out, lse, 0.0, c["is_causal"], scale=c["scale"])
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            np.testing.assert_allclose(got[0, 0], c[name], rtol=0, atol=1e-13,
                                       err_msg=f"{c['name']}:{name}")


# ---------------------------------------------------------------- philox

def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    return None


def _curand_host_philox(lib, seed, offset, n):
    """n words of curand's host-side PHILOX4_32_10 generator (runs on the CPU)."""
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


def test_philox_matches_curand_host_generator():
    """Philox4x32-10 against the library's own implementation of the same bijection.

    curand's host generator (it runs on the CPU, no GPU needed) emits, at
    stream position `offset`, word offset%4 of Philox(ctr, key) with
    key = (lo32(seed), hi32(seed)), ctr word 2 = (offset/4) mod 65536 and
    ctr words 0..1 = the 64-bit block (offset/4) div 65536. That pins the
    round function, both key words and counter words 0, 1 and 2.
    """
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not found")
    rng = np.random.default_rng(5)
    for _ in range(12):
        seed = int(rng.integers(0, 2**63)) | (int(rng.integers(0, 2)) << 63)
        c0 = int(rng.integers(0, 2**32))
        c1 = int(rng.integers(0, 2**12))
        c2 = int(rng.integers(0, 65536))
        block = (c1 << 32) | c0
        off = 4 * (block * 65536 + c2)
        got = _curand_host_philox(lib, seed, off, 4)
        mine = philox.philox4x32_10([c0, c1, c2, 0], (seed & 0xFFFFFFFF, seed >> 32))
        assert list(got) == list(mine), (seed, c0, c1, c2)


def test_uniform_words_select_word_n_mod_4():
    """u(n) is word n&3 of the block n>>2, for unaligned starts too."""
    seed, offset = 0x1122334455667788, 9
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for n0 in (0, 1, 2, 3, 4 * 1000 + 3, 2**33 + 1):
        u = philox.uniform_words(n0, 9, seed, offset)
        for t in range(9):
            n = n0 + t
            w = philox.philox4x32_10([n >> 2 & 0xFFFFFFFF, n >> 34, offset, 0], key)
            assert u[t] == w[n & 3]


def test_keep_rate_within_5_sigma():
    for p, shape in ((0.1, (512, 512)), (0.5, (64, 256)), (0.9, (128, 128))):
        m = philox.keep_mask_head(3, 5, 12, shape[0], shape[1], p, 1234, 0)
        n = m.size
        rate = m.mean()
        sigma = math.sqrt(p * (1 - p) / n)
        assert abs(rate - (1 - p)) < 5 * sigma, (p, rate)


def test_mask_reproducible_and_stream_separated():
    a = philox.keep_mask(2, 3, 40, 72, 0.3, 7, 4096)
    b = philox.keep_mask(2, 3, 40, 72, 0.3, 7, 4096)
    assert np.array_equal(a, b)
    # another offset or seed gives an independent stream: ~half the u bits flip
    n = 40 * 72
    u0 = philox.uniform_words(0, n, 7, 4096)
    for s, o in ((7, 4097), (8, 4096), (7, 4096 + (1 << 32))):
        u1 = philox.uniform_words(0, n, s, o)
        flips = np.unpackbits((u0 ^ u1).view(np.uint8)).mean()
        assert abs(flips - 0.5) < 0.02, (s, o, flips)


def test_mask_is_a_function_of_the_absolute_index():
    """Head (b,h) of the full mask uses the counters of its own index range."""
    B, H, Sq, Sk, p = 2, 3, 5, 11, 0.4
    full = philox.keep_mask(B, H, Sq, Sk, p, 99, 3)
    u = philox.uniform_words(0, B * H * Sq * Sk, 99, 3).reshape(B, H, Sq, Sk)
    assert np.array_equal(full, u >= philox.keep_threshold(p))


def test_threshold_edges():
    assert philox.keep_threshold(0.0) == 0
    assert philox.keep_threshold(0.5) == 2**31
    assert philox.keep_threshold(0.1) == 429496729
    assert philox.keep_mask_head(0, 0, 1, 8, 8, 0.0, 1, 2).all()
    with pytest.raises(ValueError):
        philox.keep_threshold(1.0)


# ---------------------------------------------------------------- forward

def test_softmax_rows_sum_to_one():
    """With V = I the output is the (dropout-free) probability matrix itself."""
    for causal in (False, True):
        q = rnd((1, 1, 9, 6), 1)
        k = rnd((1, 1, 6, 6), 2)
        v = np.eye(6)[None, None]
        out, _ = oracle.sdpa_fwd(q, k, v, 0.0, causal)
        np.testing.assert_allclose(out[0, 0].sum(axis=1), 1.0, atol=1e-14)
        assert (out >= 0).all()
        if causal:
            assert np.all(out[0, 0][np.triu_indices(6, 1)] == 0.0)


def test_causal_row_zero_is_v0():
    q = rnd((2, 3, 7, 4), 3)
    k = rnd((2, 3, 7, 4), 4)
    v = rnd((2, 3, 7, 4), 5)
    out, lse = oracle.sdpa_fwd(q, k, v, 0.0, True, 0.7)
    np.testing.assert_allclose(out[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], 0.7 * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-14)
    # with dropout, row 0 is V[0] times the dropout factor of element (0, 0)
    p = 0.5
    out, _ = oracle.sdpa_fwd(q, k, v, p, True, 0.7, seed=11, offset=0)
    keep = philox.keep_mask(2, 3, 7, 7, p, 11, 0)
    np.testing.assert_allclose(out[:, :, 0], v[:, :, 0] * keep[:, :, 0, 0, None] / (1 - p), atol=1e-14)


def test_identical_keys_give_mean_of_visible_values():
    B, H, Sq, Sk, D = 1, 2, 6, 6, 5
    q = rnd((B, H, Sq, D), 6)
    k = np.broadcast_to(rnd((B, H, 1, D), 7), (B, H, Sk, D))
    v = rnd((B, H, Sk, D), 8)
    scale = 0.3
    for causal in (False, True):
        out, lse = oracle.sdpa_fwd(q, k, v, 0.0, causal, scale)
        n = np.arange(1, Sq + 1) if causal else np.full(Sq, Sk)
        csum = np.cumsum(v, axis=2) if causal else np.broadcast_to(v.sum(2, keepdims=True), v.shape)
        np.testing.assert_allclose(out, csum / n[:, None], atol=1e-13)
        np.testing.assert_allclose(lse, scale * (q * k[:, :, :1]).sum(-1) + np.log(n), atol=1e-13)


def test_zero_queries_give_log_n():
    q = np.zeros((1, 1, 5, 3))
    k = rnd((1, 1, 9, 3), 9)
    v = rnd((1, 1, 9, 3), 10)
    _, lse = oracle.sdpa_fwd(q, k, v, 0.0, True)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, 6)), atol=1e-14)
    _, lse = oracle.sdpa_fwd(q, k, v, 0.0, False)
    np.testing.assert_allclose(lse[0, 0], np.log(9.0), atol=1e-14)


@pytest.mark.parametrize("causal,Sq,Sk,scale", [(False, 13, 13, None), (True, 13, 13, None),
                                                (False, 7, 19, 0.21), (True, 19, 7, 0.5)])
def test_matches_torch_math_sdpa_fp64(causal, Sq, Sk, scale):
    """Library special case: torch's CPU float64 SDPA and autograd (p = 0)."""
    B, H, D = 2, 3, 8
    q, k, v, do = (rnd((B, H, s, D), i) for i, s in enumerate((Sq, Sk, Sk, Sq)))
    out, lse = oracle.sdpa_fwd(q, k, v, 0.0, causal, scale)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    tout = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    np.testing.assert_allclose(out, tout.detach().numpy(), atol=1e-12)
    s = (1 / math.sqrt(D)) if scale is None else scale
    scores = s * tq.detach() @ tk.detach().transpose(-1, -2)
    if causal:
        scores = scores.masked_fill(~torch.ones(Sq, Sk, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(scores, dim=-1).numpy(), atol=1e-12)
    tout.backward(torch.tensor(do))
    dq, dk, dv = oracle.sdpa_bwd(do, q, k, v, out, lse, 0.0, causal, scale=scale)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_dropout_is_unbiased_over_seeds():
    """Averaged over masks, inverted dropout leaves the output unchanged."""
    B, H, Sq, Sk, D, p = 1, 1, 3, 6, 2, 0.5
    q, k, v = rnd((B, H, Sq, D), 20), rnd((B, H, Sk, D), 21), rnd((B, H, Sk, D), 22)
    ref, _ = oracle.sdpa_fwd(q, k, v)
    samples = np.stack([oracle.sdpa_fwd(q, k, v, p, False, None, seed=s)[0] for s in range(3000)])
    mean, sem = samples.mean(0), samples.std(0) / math.sqrt(len(samples))
    assert np.all(np.abs(mean - ref) < 5 * sem + 1e-12)


# ---------------------------------------------------------------- backward

@pytest.mark.parametrize("causal,p,Sq,Sk", [(False, 0.0, 5, 5), (True, 0.0, 6, 6),
                                             (False, 0.3, 4, 7), (True, 0.3, 7, 7),
                                             (True, 0.5, 8, 3)])
def test_backward_matches_central_differences(causal, p, Sq, Sk):
    """Gradients of L = sum(out * dO), with the dropout mask held fixed by (seed, offset)."""
    B, H, D = 1, 2, 3
    seed, off, scale = 77, 5, 0.8
    q, k, v, do = rnd((B, H, Sq, D), 30), rnd((B, H, Sk, D), 31), rnd((B, H, Sk, D), 32), rnd((B, H, Sq, D), 33)
    out, lse = oracle.sdpa_fwd(q, k, v, p, causal, scale, seed, off)
    grads = oracle.sdpa_bwd(do, q, k, v, out, lse, p, causal, seed, off, scale)

    def loss(qq, kk, vv):
        return (oracle.sdpa_fwd(qq, kk, vv, p, causal, scale, seed, off)[0] * do).sum()

    eps = 1e-6
    for which, g in enumerate(grads):
        args = [q, k, v]
        num = np.zeros_like(args[which])
        for idx in np.ndindex(*num.shape):
            a = [x.copy() for x in args]
            a[which][idx] += eps
            lp = loss(*a)
            a[which][idx] -= 2 * eps
            lm = loss(*a)
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, atol=2e-7, rtol=1e-6, err_msg=f"grad {which}")


def test_backward_invariants():
    """Softmax shift invariance: sum_j dK_j = 0; with p = 0, sum_j dV_j = sum_i dO_i."""
    B, H, Sq, Sk, D = 2, 2, 9, 12, 4
    q, k, v, do = rnd((B, H, Sq, D), 40), rnd((B, H, Sk, D), 41), rnd((B, H, Sk, D), 42), rnd((B, H, Sq, D), 43)
    for p in (0.0, 0.25):
        out, lse = oracle.sdpa_fwd(q, k, v, p, False, None, 3, 0)
        dq, dk, dv = oracle.sdpa_bwd(do, q, k, v, out, lse, p, False, 3, 0)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        if p == 0.0:
            np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


def test_head_subset_matches_full():
    q, k, v, do = rnd((2, 3, 5, 4), 50), rnd((2, 3, 6, 4), 51), rnd((2, 3, 6, 4), 52), rnd((2, 3, 5, 4), 53)
    out, lse = oracle.sdpa_fwd(q, k, v, 0.2, False, None, 1, 2)
    o2, l2 = oracle.sdpa_fwd(q, k, v, 0.2, False, None, 1, 2, heads=[(1, 2)])
    np.testing.assert_array_equal(o2[1, 2], out[1, 2])
    assert np.isnan(o2[0, 0]).all()


# ---------------------------------------------------------------- additive bias

@pytest.mark.parametrize("causal,Sq,Sk,shared", [(False, 11, 11, False), (False, 7, 13, True),
                                                 (True, 13, 9, False)])
def test_bias_matches_torch_math_sdpa_fp64(causal, Sq, Sk, shared):
    """Library special case: torch's CPU float64 SDPA with a float attn_mask,
    and autograd for every gradient including the bias's (p = 0)."""
    B, H, D, scale = 2, 3, 8, 0.3
    q, k, v, do = (rnd((B, H, s, D), 60 + i) for i, s in enumerate((Sq, Sk, Sk, Sq)))
    bias = rnd((1 if shared else B, H, Sq, Sk), 64)
    out, lse = oracle.sdpa_fwd(q, k, v, 0.0, causal, scale, bias=bias)
    tq, tk, tv, tb = (torch.tensor(x, requires_grad=True) for x in (q, k, v, bias))
    mask = tb
    if causal:
        mask = tb.masked_fill(~torch.ones(Sq, Sk, dtype=torch.bool).tril(), float("-inf"))
    tout = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(out, tout.detach().numpy(), atol=1e-12)
    scores = scale * tq.detach() @ tk.detach().transpose(-1, -2) + mask.detach()
    np.testing.assert_allclose(lse, torch.logsumexp(scores, dim=-1).numpy(), atol=1e-12)
    tout.backward(torch.tensor(do))
    dq, dk, dv, dbias = oracle.sdpa_bwd(do, q, k, v, out, lse, 0.0, causal, scale=scale, bias=bias)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)
    # the oracle returns the per-head dS; a shared bias's gradient is its sum
    got = dbias.sum(axis=0, keepdims=True) if shared else dbias
    np.testing.assert_allclose(got, tb.grad.numpy(), atol=1e-11)


def test_row_constant_bias_only_shifts_lse():
    """A bias constant along each row cancels in the softmax: out and every
    input gradient are unchanged, lse moves by the constant, and each row of
    dbias sums to zero."""
    B, H, Sq, Sk, D = 1, 2, 6, 9, 4
    q, k, v, do = rnd((B, H, Sq, D), 70), rnd((B, H, Sk, D), 71), rnd((B, H, Sk, D), 72), rnd((B, H, Sq, D), 73)
    c = rnd((B, H, Sq, 1), 74) * 5
    bias = np.broadcast_to(c, (B, H, Sq, Sk)).copy()
    for causal, p in ((False, 0.0), (True, 0.3)):
        out0, lse0 = oracle.sdpa_fwd(q, k, v, p, causal, None, 9, 1)
        out1, lse1 = oracle.sdpa_fwd(q, k, v, p, causal, None, 9, 1, bias=bias)
        np.testing.assert_allclose(out1, out0, atol=1e-12)
        np.testing.assert_allclose(lse1, lse0 + c[..., 0], atol=1e-12)
        g0 = oracle.sdpa_bwd(do, q, k, v, out0, lse0, p, causal, 9, 1)
        g1 = oracle.sdpa_bwd(do, q, k, v, out1, lse1, p, causal, 9, 1, bias=bias)
        for a, b in zip(g1[:3], g0):
            np.testing.assert_allclose(a, b, atol=1e-12)
        if p == 0.0:
            np.testing.assert_allclose(g1[3].sum(axis=3), 0.0, atol=1e-12)


def test_minus_infinity_bias_above_the_diagonal_is_the_causal_mask():
    """The bias is added before the softmax: -inf above the diagonal gives
    exactly the top-left causal result."""
    B, H, S, D = 1, 2, 7, 3
    q, k, v, do = (rnd((B, H, S, D), 80 + i) for i in range(4))
    tri = np.where(np.tril(np.ones((S, S), dtype=bool)), 0.0, -np.inf)[None, None]
    out_b, lse_b = oracle.sdpa_fwd(q, k, v, 0.2, False, None, 4, 0, bias=tri)
    out_c, lse_c = oracle.sdpa_fwd(q, k, v, 0.2, True, None, 4, 0)
    np.testing.assert_allclose(out_b, out_c, atol=1e-14)
    np.testing.assert_allclose(lse_b, lse_c, atol=1e-14)
    gb = oracle.sdpa_bwd(do, q, k, v, out_b, lse_b, 0.2, False, 4, 0, bias=tri)
    gc = oracle.sdpa_bwd(do, q, k, v, out_c, lse_c, 0.2, True, 4, 0)
    for a, b in zip(gb[:3], gc):
        np.testing.assert_allclose(a, b, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_padded_problem_with_masked_keys_is_the_shorter_problem(causal):
    """The reading behind the packed-batch tests: a sequence of lq queries
    and lk keys is the top-left block of a [Mq, Mk] problem whose extra keys
    get a -inf bias. Its rows of out and lse, its dq rows and its dk, dv rows
    are those of the [lq, lk] problem, and the padding keys get no gradient
    (no dropout: the padded problem's counters differ by design)."""
    H, D, lq, lk, Mq, Mk = 2, 4, 5, 6, 8, 9
    q, do = rnd((1, H, lq, D), 90), rnd((1, H, lq, D), 91)
    k, v = rnd((1, H, lk, D), 92), rnd((1, H, lk, D), 93)
    pad = lambda x, n: np.concatenate([x, np.zeros((1, H, n - x.shape[2], D))], axis=2)
    qp, dop, kp, vp = pad(q, Mq), pad(do, Mq), pad(k, Mk), pad(v, Mk)
    bias = np.zeros((1, 1, Mq, Mk))
    bias[..., lk:] = -np.inf
    out, lse = oracle.sdpa_fwd(q, k, v, 0.0, causal, None, 0, 0)
    out_p, lse_p = oracle.sdpa_fwd(qp, kp, vp, 0.0, causal, None, 0, 0, bias=bias)
    np.testing.assert_allclose(out_p[:, :, :lq], out, atol=1e-14)
    np.testing.assert_allclose(lse_p[:, :, :lq], lse, atol=1e-14)
    dq, dk, dv = oracle.sdpa_bwd(do, q, k, v, out, lse, 0.0, causal, 0, 0)
    dq_p, dk_p, dv_p, _ = oracle.sdpa_bwd(dop, qp, kp, vp, out_p, lse_p, 0.0, causal, 0, 0,
                                          bias=bias)
    np.testing.assert_allclose(dq_p[:, :, :lq], dq, atol=1e-13)
    np.testing.assert_allclose(dk_p[:, :, :lk], dk, atol=1e-13)
    np.testing.assert_allclose(dv_p[:, :, :lk], dv, atol=1e-13)
    assert not dk_p[:, :, lk:].any() and not dv_p[:, :, lk:].any()


@pytest.mark.parametrize("causal,p", [(False, 0.0), (True, 0.3)])
def test_bias_gradient_matches_central_differences(causal, p):
    """dbias of L = sum(out * dO), the dropout mask held fixed by (seed, offset)."""
    B, H, Sq, Sk, D = 1, 1, 5, 6, 3
    seed, off, scale = 12, 3, 0.7
    q, k, v, do = rnd((B, H, Sq, D), 90), rnd((B, H, Sk, D), 91), rnd((B, H, Sk, D), 92), rnd((B, H, Sq, D), 93)
    bias = rnd((B, H, Sq, Sk), 94)
    out, lse = oracle.sdpa_fwd(q, k, v, p, causal, scale, seed, off, bias=bias)
    dbias = oracle.sdpa_bwd(do, q, k, v, out, lse, p, causal, seed, off, scale, bias=bias)[3]

    def loss(bb):
        return (oracle.sdpa_fwd(q, k, v, p, causal, scale, seed, off, bias=bb)[0] * do).sum()

    eps = 1e-6
    num = np.zeros_like(bias)
    for idx in np.ndindex(*bias.shape):
        a = bias.copy()
        a[idx] += eps
        lp = loss(a)
        a[idx] -= 2 * eps
        num[idx] = (lp - loss(a)) / (2 * eps)
    np.testing.assert_allclose(dbias, num, atol=2e-7, rtol=1e-6)
