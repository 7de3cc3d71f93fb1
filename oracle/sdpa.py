"""Plain fp64 scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. This is the CPU oracle that the CUDA path is
checked against. Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it;
the library never calls it and it never calls the library.

It materialises the whole score matrix of one (batch, head) at a time, in
float64, with numpy matmuls as the only library steps. There is no tiling,
no online softmax and no fusion: every quantity is the textbook definition.

What is computed, and where it comes from
-----------------------------------------
* "Scaled_dot_product_attention" (discuss.pytorch.org thread): the
  operation is ``torch.nn.functional.scaled_dot_product_attention``; its
  plain reading is ``out = dropout(softmax(scale * Q K^T + causal)) V``.
  The pages never print the formula; that reading is taken here.
* "DID loop split for SDPA" (NVIDIA/Fuser PR 3711), test_sdpa_loop_split:
  the forward ``sdpfa_fwd(q, k, v, dropout_p, is_causal, scale)`` returns
  (attn, log_sumexp, seed, offset) and the backward
  ``sdpfa_bwd(out_grad, q, k, v, attn, log_sumexp, dropout_p, is_causal,
  seed, offset, scale)`` returns (q_grad, k_grad, v_grad); ``scale=None``
  means the default, read as 1/sqrt(D); ``is_causal`` is read as top-left
  aligned (key j visible to query i iff j <= i).
* Issue "SdpaOpFwd / SdpaOpBwd nodes" (NVIDIA/Fuser issue 2278): the
  softmax statistic that is stashed for the backward is the log-sum-exp of
  each score row (natural log); the backward recomputes the probabilities
  from it instead of storing them.
* "REDO of dropout support for mem eff #102038" (pytorch PR 103704),
  Summary: dropout inside the fused kernel, with the mask regenerated in
  the backward from (seed, offset) and the absolute element index (see
  ``oracle.philox``). Dropout is read as inverted dropout applied to the
  probabilities after the softmax: P~ = P * keep / (1 - p); the
  log-sum-exp is that of the undropped scores.

* Additive attention bias: the forum thread asks for self-attention with
  relative positional encoding through scaled_dot_product_attention, and
  the priority-order discussion of PR 103704 mentions adding attn_bias
  support to the memory-efficient kernel. It is read as torch's float
  ``attn_mask``: a bias B_ij added to the scaled scores before the softmax,
  ``S = scale * Q K^T + B`` (then the causal mask), and the log-sum-exp is
  that of these biased scores. Its gradient is ``dB = dS``.

Backward (the standard derivative of the forward above)::

    dV = P~^T dO
    dP = (dO V^T) * keep / (1 - p)
    Delta_i = sum_e dO_ie * out_ie      (= sum_j P_ij dP_ij)
    dS = P * (dP - Delta)
    dQ = scale * dS K,   dK = scale * dS^T Q
"""

import math

import numpy as np

from .philox import keep_mask_head


def default_scale(D):
    """The softmax scale used when the caller passes none: 1/sqrt(head dim)."""
    return 1.0 / math.sqrt(D)


def _visible(Sq, Sk, is_causal):
    """Boolean [Sq, Sk]: key j is visible to query i (top-left causal)."""
    if not is_causal:
        return np.ones((Sq, Sk), dtype=bool)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    return j <= i


def _dropout_factor(b, h, H, Sq, Sk, p, seed, offset):
    """Z = keep / (1 - p) as float64 [Sq, Sk] (all ones when p == 0)."""
    if p == 0.0:
        return np.ones((Sq, Sk))
    keep = keep_mask_head(b, h, H, Sq, Sk, p, seed, offset)
    return keep.astype(np.float64) / (1.0 - p)


def _heads(B, H, heads):
    return [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)


def head_forward(qh, kh, vh, b, h, H, dropout_p, is_causal, scale, seed, offset, bias=None):
    """Forward of one head. qh [Sq,D], kh [Sk,D], vh [Sk,D] (float64);
    bias: optional additive bias [Sq,Sk] of this head.

    Returns (out [Sq,D], lse [Sq]).
    """
    Sq, Sk = qh.shape[0], kh.shape[0]
    S = scale * (qh @ kh.T)
    if bias is not None:
        S = S + bias
    S = np.where(_visible(Sq, Sk, is_causal), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
    P = np.exp(S - lse[:, None])
    Z = _dropout_factor(b, h, H, Sq, Sk, dropout_p, seed, offset)
    out = (P * Z) @ vh
    return out, lse


def head_backward(doh, qh, kh, vh, outh, lseh, b, h, H, dropout_p, is_causal,
                  scale, seed, offset, check_delta=True, bias=None):
    """Backward of one head; returns (dq [Sq,D], dk [Sk,D], dv [Sk,D]), and
    dbias [Sq,Sk] as a fourth item when ``bias`` is given."""
    Sq, Sk = qh.shape[0], kh.shape[0]
    S = scale * (qh @ kh.T)
    if bias is not None:
        S = S + bias
    S = np.where(_visible(Sq, Sk, is_causal), S, -np.inf)
    P = np.exp(S - lseh[:, None])
    Z = _dropout_factor(b, h, H, Sq, Sk, dropout_p, seed, offset)
    dv = (P * Z).T @ doh
    dP = (doh @ vh.T) * Z
    delta = (doh * outh).sum(axis=1)
    if check_delta:
        # The two expressions of Delta agree when out/lse are this forward's.
        alt = (P * dP).sum(axis=1)
        tol = 1e-9 * (1.0 + np.abs(doh).sum(axis=1) * np.abs(outh).sum(axis=1))
        if not np.all(np.abs(alt - delta) <= tol):
            raise AssertionError("rowsum(dO*out) != rowsum(P*dP): out/lse are not this forward's")
    dS = P * (dP - delta[:, None])
    dq = scale * (dS @ kh)
    dk = scale * (dS.T @ qh)
    if bias is not None:
        return dq, dk, dv, dS
    return dq, dk, dv


def _bias_of(bias, b, h):
    """The [Sq,Sk] bias of head (b, h) from a [B or 1, H or 1, Sq, Sk] array."""
    if bias is None:
        return None
    return bias[b if bias.shape[0] > 1 else 0, h if bias.shape[1] > 1 else 0]


def sdpa_fwd(q, k, v, dropout_p=0.0, is_causal=False, scale=None, seed=0, offset=0,
             heads=None, bias=None):
    """Forward over logical [B,H,S,D] float64 arrays.

    ``heads``: optional iterable of (b, h) pairs; only those heads are
    computed (the others are left NaN). ``bias``: optional additive bias
    [B or 1, H or 1, Sq, Sk] (a size-1 dim is shared by every batch / head).
    Returns (out [B,H,Sq,D], lse [B,H,Sq]).
    """
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, Sq, D = q.shape
    if scale is None:
        scale = default_scale(D)
    out = np.full((B, H, Sq, v.shape[3]), np.nan)
    lse = np.full((B, H, Sq), np.nan)
    if bias is not None:
        bias = np.asarray(bias, dtype=np.float64)
    for b, h in _heads(B, H, heads):
        out[b, h], lse[b, h] = head_forward(q[b, h], k[b, h], v[b, h], b, h, H,
                                            dropout_p, is_causal, scale, seed, offset,
                                            bias=_bias_of(bias, b, h))
    return out, lse


def sdpa_bwd(dout, q, k, v, out, lse, dropout_p=0.0, is_causal=False, seed=0, offset=0,
             scale=None, heads=None, check_delta=True, bias=None):
    """Backward over logical [B,H,S,D] float64 arrays; returns (dq, dk, dv),
    and dbias [B,H,Sq,Sk] (per head, not summed over shared dims) as a
    fourth item when ``bias`` is given."""
    dout, q, k, v, out, lse = (np.asarray(t, dtype=np.float64)
                               for t in (dout, q, k, v, out, lse))
    B, H, Sq, D = q.shape
    if scale is None:
        scale = default_scale(D)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    if bias is not None:
        bias = np.asarray(bias, dtype=np.float64)
        dbias = np.full((B, H, q.shape[2], k.shape[2]), np.nan)
    for b, h in _heads(B, H, heads):
        r = head_backward(dout[b, h], q[b, h], k[b, h], v[b, h], out[b, h], lse[b, h], b, h, H,
                          dropout_p, is_causal, scale, seed, offset, check_delta,
                          bias=_bias_of(bias, b, h))
        dq[b, h], dk[b, h], dv[b, h] = r[:3]
        if bias is not None:
            dbias[b, h] = r[3]
    if bias is not None:
        return dq, dk, dv, dbias
    return dq, dk, dv
