"""Dropout keep bits carried from the forward to the backward (dropout_bits).

The forward writes the keep bits of the score tiles it computes into a
caller's buffer; a backward given that buffer reads them instead of drawing
them again. The stored words must hold exactly the oracle's mask (Philox4x32-10
of the absolute element index, "REDO of dropout support for mem eff
#102038", pytorch PR 103704), and both calls must return bit for bit what
the calls that draw the mask themselves return.
"""

import numpy as np
import pytest
import torch

import oracle


def ceil128(n):
    return (n + 127) // 128 * 128


def unpack(bits, B, H, Sq, Sk):
    """[B, H, Sq, Sk] keep flags from the buffer's words: word
    ((b*H + h)*ceil128(Sk)/32 + w)*ceil128(Sq) + i holds keys 32w .. 32w+31 of
    row i, bit e for key 32w + e."""
    Sq_p, Sk_p = ceil128(Sq), ceil128(Sk)
    w = bits.cpu().numpy().view(np.uint32).reshape(B * H, Sk_p // 32, Sq_p)
    b = ((w[..., None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)  # [BH, W, Sq_p, 32]
    m = b.transpose(0, 2, 1, 3).reshape(B, H, Sq_p, Sk_p)
    return m[:, :, :Sq, :Sk]


def visible(Sq, Sk, causal):
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    return (j <= i) if causal else np.ones((Sq, Sk), dtype=bool)


def inputs(B, H, Sq, Sk, D, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda S: torch.randn(B, H, S, D, generator=g).bfloat16().cuda()
    return mk(Sq), mk(Sk), mk(Sk), mk(Sq)


# several 128-key tiles and ragged tails; Sk not a multiple of 4 (a word
# straddles Philox groups); Sq != Sk both ways; head dims 64, 96 (padded to
# the 128-wide kernels) and 128
CASES = [(2, 3, 300, 260, 64, True), (1, 2, 200, 333, 128, True), (2, 2, 257, 384, 128, False),
         (1, 1, 128, 128, 96, True), (1, 2, 129, 131, 64, False), (1, 2, 520, 390, 128, True)]


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Sq,Sk,D,causal", CASES)
def test_stored_bits_are_the_oracle_mask_and_change_no_result(cuda_lib, B, H, Sq, Sk, D, causal):
    p, seed, offset = 0.15, 1234, 77
    q, k, v, do = inputs(B, H, Sq, Sk, D, 11 + Sq + Sk)
    bits = torch.zeros(cuda_lib.sdpa_dropout_bits_size(B, H, Sq, Sk) // 4, dtype=torch.int32,
                       device="cuda")
    out0, lse0 = cuda_lib.sdpa_fwd_ex(q, k, v, p, causal, None, seed, offset)
    out1, lse1 = cuda_lib.sdpa_fwd_ex(q, k, v, p, causal, None, seed, offset, dropout_bits=bits)
    torch.cuda.synchronize()
    assert cuda_lib.sdpa_check_device() == 0
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    vis = visible(Sq, Sk, causal)
    got = unpack(bits, B, H, Sq, Sk)
    want = oracle.keep_mask(B, H, Sq, Sk, p, seed, offset)
    assert np.array_equal(got[:, :, vis], want[:, :, vis])
    g0 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out0, lse0, p, causal, seed, offset, deterministic=True)
    g1 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out0, lse0, p, causal, seed, offset, deterministic=True,
                              dropout_bits=bits)
    torch.cuda.synchronize()
    assert cuda_lib.sdpa_check_device() == 0
    for a, b, name in zip(g0, g1, ("dq", "dk", "dv")):
        assert torch.equal(a, b), name


@pytest.mark.gpu
def test_stored_bits_with_device_rng_state_and_a_head_slice(cuda_lib):
    """A slice of heads [3, 5) of a 5-head problem with the seed and offset
    read from device memory: the stored words are that slice of the whole
    problem's mask, and the backward that reads them matches the one that
    draws."""
    B, H, Sq, Sk, D, Ht, h0 = 2, 2, 256, 200, 64, 5, 3
    p, seed, offset = 0.3, 987654321, 4242
    q, k, v, do = inputs(B, H, Sq, Sk, D, 5)
    rng = torch.tensor([seed, offset], dtype=torch.int64, device="cuda")
    bits = torch.zeros(cuda_lib.sdpa_dropout_bits_size(B, H, Sq, Sk) // 4, dtype=torch.int32,
                       device="cuda")
    kw = dict(rng_state=rng, head_offset=h0, total_heads=Ht)
    out, lse = cuda_lib.sdpa_fwd_ex(q, k, v, p, True, None, 0, 0, dropout_bits=bits, **kw)
    torch.cuda.synchronize()
    got = unpack(bits, B, H, Sq, Sk)
    want = oracle.keep_mask(B, Ht, Sq, Sk, p, seed, offset)[:, h0:h0 + H]
    vis = visible(Sq, Sk, True)
    assert np.array_equal(got[:, :, vis], want[:, :, vis])
    g0 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out, lse, p, True, 0, 0, deterministic=True, **kw)
    g1 = cuda_lib.sdpa_bwd_ex(do, q, k, v, out, lse, p, True, 0, 0, deterministic=True,
                              dropout_bits=bits, **kw)
    torch.cuda.synchronize()
    assert cuda_lib.sdpa_check_device() == 0
    for a, b, name in zip(g0, g1, ("dq", "dk", "dv")):
        assert torch.equal(a, b), name


@pytest.mark.gpu
def test_bits_buffer_is_ignored_without_dropout(cuda_lib):
    B, H, S, D = 1, 2, 200, 64
    q, k, v, do = inputs(B, H, S, S, D, 3)
    bits = torch.full((cuda_lib.sdpa_dropout_bits_size(B, H, S, S) // 4,), 7, dtype=torch.int32,
                      device="cuda")
    out, lse = cuda_lib.sdpa_fwd_ex(q, k, v, 0.0, True, None, 1, 0, dropout_bits=bits)
    ref, _ = cuda_lib.sdpa_fwd_ex(q, k, v, 0.0, True, None, 1, 0)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert bool((bits == 7).all())
