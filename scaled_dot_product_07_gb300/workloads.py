"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out in memory; it holds
none of the attention arithmetic, so both the CUDA path (tests, bench) and
the CPU oracle can consume its tensors without sharing any of the method.

Workloads
---------
``tiny``            B1 H2 S128 D64, causal, p=0
``pages_test``      B2 H12 S1024 D64 (model width 768), causal, p=0, in the
                    BHSE and BSHE layouts -- the shape and the two stride
                    orders of test_sdpa_loop_split ("DID loop split for
                    SDPA", NVIDIA/Fuser PR 3711)
``encoder_dropout`` B32 H12 S512 D64, non-causal, p=0.1, seed 1234, offset 0
``decoder_long``    B8 H16 S4096 D128, causal, p=0, dO ~ N(0, 0.1^2)
``cross_attn``      B4 H16 Sq1024 Sk8192 D128, non-causal, p=0.1, seed 7,
                    offset 4096, K drawn N(0,1) then multiplied by 3

Recipe: q, k, v, dout are drawn in that order from one CPU
``torch.Generator`` seeded with the workload's input seed, as float32
``randn`` of the logical shape [B, H, S, D], multiplied by their scale
factor, and rounded to bfloat16 (round to nearest even). The layout only
decides the memory order of the same logical values.
"""

from dataclasses import dataclass, field

import torch

# stride_order of test_sdpa_loop_split: entry k is the rank of dim k's stride
# (higher = outer) over the logical dims (B, H, S, D).
STRIDE_ORDER = {"BHSE": (3, 2, 1, 0), "BSHE": (3, 1, 2, 0)}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    is_causal: bool
    dropout_p: float = 0.0
    seed: int = 0          # Philox seed of the dropout mask
    offset: int = 0        # Philox offset of the dropout mask
    input_seed: int = 0    # seed of the input generator
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    do_std: float = 1.0
    layouts: tuple = field(default=("BHSE",))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 128, 64, True, input_seed=0),
    "pages_test": Workload("pages_test", 2, 12, 1024, 1024, 64, True, input_seed=1,
                           layouts=("BHSE", "BSHE")),
    "encoder_dropout": Workload("encoder_dropout", 32, 12, 512, 512, 64, False, 0.1,
                                seed=1234, offset=0, input_seed=2),
    "decoder_long": Workload("decoder_long", 8, 16, 4096, 4096, 128, True, input_seed=3,
                             do_std=0.1),
    "cross_attn": Workload("cross_attn", 4, 16, 1024, 8192, 128, False, 0.1, seed=7,
                           offset=4096, input_seed=4, k_std=3.0),
}


def make_workload(name, **overrides):
    """A named workload, optionally with fields replaced (e.g. smaller B)."""
    w = WORKLOADS[name]
    if overrides:
        d = dict(w.__dict__)
        d.update(overrides)
        w = Workload(**d)
    return w


def draw_inputs(w):
    """Seeded logical-[B,H,S,D] bfloat16 CPU tensors (q, k, v, dout), contiguous."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.input_seed)
    out = []
    for shape, std in (((w.B, w.H, w.Sq, w.D), w.q_std),
                       ((w.B, w.H, w.Sk, w.D), w.k_std),
                       ((w.B, w.H, w.Sk, w.D), w.v_std),
                       ((w.B, w.H, w.Sq, w.D), w.do_std)):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def to_layout(x, layout):
    """Same logical [B,H,S,D] values stored in the given memory order.

    Returns a view with logical shape [B,H,S,D] whose strides follow the
    layout's stride order (BHSE: contiguous; BSHE: physical [B,S,H,D]).
    """
    if layout == "BHSE":
        return x.contiguous()
    if layout == "BSHE":
        return x.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
    raise ValueError(f"unknown layout {layout}")


def draw_bias(shape, seed, kind="random"):
    """Seeded bfloat16 additive-bias input of logical shape [Bb, Hb, Sq, Sk]
    (CPU, contiguous).

    ``random``: float32 ``randn`` from a CPU generator seeded with ``seed``,
    times 1.5. ``relpos``: a relative-position pattern, -slope_h * |i - j|
    with slope_h = 2^(-(h + 1) / Hb) (distance penalties of different
    strength per head), plus the same random draw times 0.1. Both are
    rounded to bfloat16; only inputs are made here.
    """
    Bb, Hb, Sq, Sk = shape
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    noise = torch.randn(shape, generator=g, dtype=torch.float32)
    if kind == "random":
        x = noise * 1.5
    elif kind == "relpos":
        dist = (torch.arange(Sq)[:, None] - torch.arange(Sk)[None, :]).abs().float()
        slope = torch.pow(2.0, -(torch.arange(Hb, dtype=torch.float32) + 1.0) / Hb)
        x = -slope[None, :, None, None] * dist[None, None] + 0.1 * noise
    else:
        raise ValueError(f"unknown bias kind {kind}")
    return x.to(torch.bfloat16)


def padded_rows(x, multiple=8):
    """The same logical [.., Sk] values in a buffer whose key rows are padded
    to a multiple of ``multiple`` elements (a view with a larger row stride),
    as the bias loads of the kernels require 16-byte aligned rows."""
    Sk = x.shape[-1]
    pad = (Sk + multiple - 1) // multiple * multiple
    buf = torch.zeros(x.shape[:-1] + (pad,), dtype=x.dtype, device=x.device)
    buf[..., :Sk] = x
    return buf[..., :Sk]
