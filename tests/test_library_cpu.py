"""Host-side checks of the C-ABI library that need no GPU.

The library is built (nvcc cross-compiles sm_103a here), loaded, and every
entry point declared in include/sdpa.h must be exported. Argument checks
run entirely on the host before any CUDA call, so their status codes are
tested here with fake pointers that are never dereferenced.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from scaled_dot_product_07_gb300 import _build
    _build.build()
    import scaled_dot_product_07_gb300 as sdpa
    return sdpa.load_library()


def declared_functions():
    with open(os.path.join(ROOT, "include", "sdpa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(sdpa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sdpa_fwd", "sdpa_bwd", "sdpa_bwd_workspace_size", "sdpa_dropout_mask_debug",
              "sdpa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import scaled_dot_product_07_gb300 as sdpa
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/sdpa.h but not exported"
    assert set(names) == set(sdpa.EXPORTED_SYMBOLS)


def test_status_strings(lib):
    import scaled_dot_product_07_gb300 as sdpa
    for code, name in sdpa.STATUS_NAMES.items():
        assert sdpa.sdpa_status_string(code).startswith(name)
    assert "UNKNOWN" in sdpa.sdpa_status_string(99)


def test_workspace_size(lib):
    import scaled_dot_product_07_gb300 as sdpa
    # fp32 dQ accumulator + two fp32 row vectors, Sq rounded up to 128
    assert sdpa.sdpa_bwd_workspace_size(2, 3, 200, 77, 64) == 2 * 3 * 256 * (64 + 2) * 4
    assert sdpa.sdpa_bwd_workspace_size(8, 16, 4096, 4096, 128) == 8 * 16 * 4096 * 130 * 4
    assert sdpa.sdpa_bwd_workspace_size(0, 3, 200, 77, 64) == 0
    # head dims up to 64 keep 64-wide accumulator rows, up to 128 128-wide
    # rows (the 128-wide tiles of the backward), above 128 256-wide rows
    assert sdpa.sdpa_bwd_workspace_size(2, 3, 200, 77, 40) == 2 * 3 * 256 * (64 + 2) * 4
    assert sdpa.sdpa_bwd_workspace_size(2, 3, 200, 77, 96) == 2 * 3 * 256 * (128 + 2) * 4
    assert sdpa.sdpa_bwd_workspace_size(2, 3, 200, 77, 136) == 2 * 3 * 256 * (256 + 2) * 4
    assert sdpa.sdpa_bwd_workspace_size(2, 3, 200, 77, 256) == 2 * 3 * 256 * (256 + 2) * 4
    assert sdpa.sdpa_bwd_workspace_size(1, 1, 0, 77, 64) == 0


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced


def test_workspace_size_saturates_instead_of_wrapping(lib):
    import scaled_dot_product_07_gb300 as sdpa
    size_max = 2**64 - 1
    # 2^62 fp32 rows would wrap a 64-bit byte count; no workspace satisfies it
    assert sdpa.sdpa_bwd_workspace_size(2**30, 2**20, 2**20, 1, 128) == size_max
    assert sdpa.sdpa_bwd_workspace_size_ex(2**10, 2**10, 2**20, 2**30, 128, True) == size_max
    # the largest sizes below the limit are exact
    assert sdpa.sdpa_bwd_workspace_size(2**20, 2**10, 2**12, 1, 128) == 2**42 * 130 * 4


def desc(B, H, S, D, layout="BHSE", data=FAKE, stride=None):
    import scaled_dot_product_07_gb300 as sdpa
    t = sdpa.SdpaTensor()
    t.data = data
    for i, s in enumerate((B, H, S, D)):
        t.size[i] = s
    if stride is None:
        stride = (H * S * D, S * D, D, 1) if layout == "BHSE" else (S * H * D, D, H * D, 1)
    for i, s in enumerate(stride):
        t.stride[i] = s
    return t


def fwd_status(lib, q, k, v, o, p=0.0, causal=0, scale=0.125, lse=FAKE):
    r = ctypes.byref
    return lib.sdpa_fwd(r(q), r(k), r(v), p, causal, scale, 1, 0, r(o), ctypes.c_void_p(lse), None)


def test_forward_argument_errors(lib):
    B, H, S, D = 2, 3, 100, 64
    ok = lambda: desc(B, H, S, D)
    # head dims: multiples of 8 up to 256
    for bad in (100, 264, 4, 130):
        assert fwd_status(lib, desc(B, H, S, bad), desc(B, H, S, bad), desc(B, H, S, bad),
                          desc(B, H, S, bad)) == 2
    # E != Ev
    assert fwd_status(lib, ok(), ok(), desc(B, H, S, 128), ok()) == 1
    # K and V disagree on Sk; batch mismatch
    assert fwd_status(lib, ok(), ok(), desc(B, H, S + 1, D), ok()) == 1
    assert fwd_status(lib, ok(), desc(B + 1, H, S, D), desc(B + 1, H, S, D), ok()) == 1
    # out shape
    assert fwd_status(lib, ok(), ok(), ok(), desc(B, H, S + 1, D)) == 1
    # dropout probability and scale
    assert fwd_status(lib, ok(), ok(), ok(), ok(), p=1.0) == 1
    assert fwd_status(lib, ok(), ok(), ok(), ok(), p=-0.1) == 1
    assert fwd_status(lib, ok(), ok(), ok(), ok(), scale=0.0) == 1
    assert fwd_status(lib, ok(), ok(), ok(), ok(), scale=float("nan")) == 1
    # D not innermost
    assert fwd_status(lib, desc(B, H, S, D, stride=(H * S * D, S * D, 1, S)), ok(), ok(), ok()) == 2
    # misaligned base pointer, misaligned stride
    assert fwd_status(lib, desc(B, H, S, D, data=FAKE + 2), ok(), ok(), ok()) == 3
    assert fwd_status(lib, desc(B, H, S, D, stride=(H * S * 72, S * 72, 68, 1)), ok(), ok(), ok()) == 3
    # null data, null / misaligned lse
    assert fwd_status(lib, desc(B, H, S, D, data=None), ok(), ok(), ok()) == 1
    assert fwd_status(lib, ok(), ok(), ok(), ok(), lse=0) == 1
    assert fwd_status(lib, ok(), ok(), ok(), ok(), lse=FAKE + 2) == 1
    # a key length of zero with queries present
    assert fwd_status(lib, ok(), desc(B, H, 0, D), desc(B, H, 0, D), ok()) == 1


def test_launch_grid_and_counter_limits(lib):
    # views with overlapping strides can describe problems whose grids of
    # 128-row tiles do not fit in int, or whose dropout counter does not fit
    # in 64 bits; both are refused on the host
    D = 64
    small = (D, D, D, 1)
    big = desc(2**15, 2**15, 2**20, D, stride=small)        # 2^43 query tiles
    assert fwd_status(lib, big, big, big, big) == 2
    wide = desc(2**7, 1, 2**30, D, stride=small)            # 2^30 tiles, counter 2^67
    assert fwd_status(lib, wide, wide, wide, wide) == 1
    r = ctypes.byref
    assert lib.sdpa_bwd(r(big), r(big), r(big), r(big), r(big), ctypes.c_void_p(FAKE), 0.0, 0, 0,
                        0, 0.125, r(big), r(big), r(big), ctypes.c_void_p(FAKE), 2**40, None) == 2


def test_empty_problems_are_no_ops(lib):
    D = 64
    # Sq == 0 and B == 0 succeed without touching the device (no GPU here)
    assert fwd_status(lib, desc(2, 3, 0, D), desc(2, 3, 5, D), desc(2, 3, 5, D), desc(2, 3, 0, D)) == 0
    assert fwd_status(lib, desc(0, 3, 9, D), desc(0, 3, 5, D), desc(0, 3, 5, D), desc(0, 3, 9, D)) == 0
    r = ctypes.byref
    z = desc(0, 2, 4, D)
    assert lib.sdpa_bwd(r(z), r(z), r(z), r(z), r(z), None, 0.0, 0, 0, 0, 0.125, r(z), r(z), r(z),
                        None, 0, None) == 0
    assert lib.sdpa_dropout_mask_debug(0, 2, 3, 4, 0.1, 1, 2, None, None) == 0


def test_backward_argument_errors(lib):
    B, H, Sq, Sk, D = 1, 2, 100, 70, 128
    q, kk = desc(B, H, Sq, D), desc(B, H, Sk, D)
    r = ctypes.byref

    def st(ws=FAKE, ws_bytes=1 << 30, dk=None, p=0.0):
        return lib.sdpa_bwd(r(q), r(q), r(kk), r(kk), r(q), ctypes.c_void_p(FAKE), p, 1, 0, 0,
                            0.1, r(q), r(dk or kk), r(kk), ctypes.c_void_p(ws), ws_bytes, None)

    need = lib.sdpa_bwd_workspace_size(B, H, Sq, Sk, D)
    assert st(ws=0) == 6
    assert st(ws_bytes=need - 1) == 6
    assert st(ws=FAKE + 16) == 6  # workspace must be 256-byte aligned
    assert st(dk=desc(B, H, Sk + 1, D)) == 1
    assert st(p=1.5) == 1


def test_mask_debug_argument_errors(lib):
    assert lib.sdpa_dropout_mask_debug(1, 1, 4, 4, 1.0, 0, 0, ctypes.c_void_p(FAKE), None) == 1
    assert lib.sdpa_dropout_mask_debug(1, 1, 4, 4, 0.5, 0, 0, None, None) == 1
    assert lib.sdpa_dropout_mask_debug(-1, 1, 4, 4, 0.5, 0, 0, ctypes.c_void_p(FAKE), None) == 1


def test_binding_refuses_cpu_tensors():
    import torch
    import scaled_dot_product_07_gb300 as sdpa
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sdpa.sdpa_fwd(x, x, x)


def test_noalloc_backward_rejects_oversize_problems_on_the_host(lib):
    import scaled_dot_product_07_gb300 as sdpa
    B, H, S, D = 8, 16, 4096, 128
    assert lib.sdpa_bwd_workspace_size(B, H, S, S, D) > sdpa.NOALLOC_SCRATCH_BYTES
    t = desc(B, H, S, D)
    r = ctypes.byref
    st = lib.sdpa_bwd_noalloc(r(t), r(t), r(t), r(t), r(t), ctypes.c_void_p(FAKE), 0.0, 1, 0, 0,
                              0.1, r(t), r(t), r(t), None)
    assert st == 6


def options(**kw):
    import scaled_dot_product_07_gb300 as sdpa
    o = sdpa.SdpaOptions()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def test_deterministic_workspace_holds_one_dq_slice_per_key_tile(lib):
    import scaled_dot_product_07_gb300 as sdpa
    # one fp32 [B*H, ceil128(Sq), D] slice per 128-key tile, plus lse2 and delta
    assert sdpa.sdpa_bwd_workspace_size_ex(2, 3, 200, 300, 64, True) == 2 * 3 * 256 * (64 * 3 + 2) * 4
    assert (sdpa.sdpa_bwd_workspace_size_ex(8, 16, 4096, 4096, 128, True)
            == 8 * 16 * 4096 * (128 * 32 + 2) * 4)
    # without the flag (or with no options at all) it is the plain workspace
    assert (sdpa.sdpa_bwd_workspace_size_ex(2, 3, 200, 300, 64, False)
            == sdpa.sdpa_bwd_workspace_size(2, 3, 200, 300, 64))
    assert lib.sdpa_bwd_workspace_size_ex(2, 3, 200, 300, 64, None) == lib.sdpa_bwd_workspace_size(
        2, 3, 200, 300, 64)


def test_option_errors_are_reported_before_any_launch(lib):
    B, H, S, D = 2, 4, 300, 64  # three key tiles
    t = desc(B, H, S, D)
    r = ctypes.byref

    def fwd(o):
        return lib.sdpa_fwd_ex(r(t), r(t), r(t), 0.1, 1, 0.125, 1, 0, r(t), ctypes.c_void_p(FAKE),
                               r(o), None)

    # head slice past the problem's heads; negative offsets; misaligned rng pointer
    assert fwd(options(head_offset=1)) == 1                       # total_heads 0 means H
    assert fwd(options(head_offset=3, total_heads=6)) == 1       # 3 + 4 > 6
    assert fwd(options(batch_offset=-1)) == 1
    assert fwd(options(total_heads=-2)) == 1
    assert fwd(options(rng_state=FAKE + 4)) == 3
    # kernel events need both handles (checked before anything is recorded)
    handles = (ctypes.c_void_p * 2)(FAKE, None)
    assert fwd(options(kernel_events=ctypes.addressof(handles))) == 1
    # the global counter must fit in 64 bits
    assert fwd(options(batch_offset=2**30, total_heads=2**30)) == 1

    def bwd(o, ws_bytes):
        return lib.sdpa_bwd_ex(r(t), r(t), r(t), r(t), r(t), ctypes.c_void_p(FAKE), 0.0, 1, 0, 0,
                               0.125, r(t), r(t), r(t), ctypes.c_void_p(FAKE), ws_bytes, r(o), None)

    # deterministic mode needs its larger workspace
    plain = lib.sdpa_bwd_workspace_size(B, H, S, S, D)
    det = lib.sdpa_bwd_workspace_size_ex(B, H, S, S, D, r(options(deterministic=1)))
    assert det > plain
    assert bwd(options(deterministic=1), det - 1) == 6
    assert bwd(options(head_offset=2, total_heads=5), plain) == 1
    assert lib.sdpa_dropout_mask_debug_ex(B, H, S, S, 0.1, 0, 0, r(options(head_offset=9)),
                                          ctypes.c_void_p(FAKE), None) == 1


def test_bias_argument_errors(lib):
    B, H, Sq, Sk, D = 2, 4, 100, 130, 64
    q, kk = desc(B, H, Sq, D), desc(B, H, Sk, D)
    r = ctypes.byref
    keep = []  # descriptors must outlive the calls that point at them

    def bias(Bb=B, Hb=H, S1=Sq, S2=Sk, row=136, data=FAKE, key_stride=1):
        d = desc(Bb, Hb, S1, S2, data=data, stride=(Hb * S1 * row, S1 * row, row, key_stride))
        keep.append(d)
        return ctypes.addressof(d)

    def fwd(o):
        return lib.sdpa_fwd_ex(r(q), r(kk), r(kk), 0.0, 1, 0.125, 1, 0, r(q), ctypes.c_void_p(FAKE),
                               r(o), None)

    assert fwd(options(attn_bias=bias(Bb=3))) == 1           # batch 3 vs 2
    assert fwd(options(attn_bias=bias(S2=Sk + 1))) == 1      # key length
    assert fwd(options(attn_bias=bias(row=130))) == 3        # rows not 16-byte aligned
    assert fwd(options(attn_bias=bias(data=FAKE + 2))) == 3  # base not aligned
    assert fwd(options(attn_bias=bias(key_stride=2))) == 2   # keys not contiguous

    def bwd(o):
        return lib.sdpa_bwd_ex(r(q), r(q), r(kk), r(kk), r(q), ctypes.c_void_p(FAKE), 0.0, 1, 0, 0,
                               0.125, r(q), r(kk), r(kk), ctypes.c_void_p(FAKE), 1 << 40, r(o), None)

    # a gradient needs the bias, and must have the full [B, H, Sq, Sk] shape
    assert bwd(options(dbias=bias())) == 1
    assert bwd(options(attn_bias=bias(Bb=1, Hb=1), dbias=bias(Bb=1))) == 1


def test_varlen_argument_errors(lib):
    import scaled_dot_product_07_gb300 as sdpa
    H, Tq, Tk, D = 2, 300, 400, 64
    r = ctypes.byref
    q, kk = desc(1, H, Tq, D, layout="BSHE"), desc(1, H, Tk, D, layout="BSHE")

    def seqs(cq=FAKE, ck=FAKE, batch=3, mq=128, mk=256):
        v = sdpa.SdpaVarlen()
        v.cu_seqlens_q, v.cu_seqlens_k = cq, ck
        v.batch, v.max_seqlen_q, v.max_seqlen_k = batch, mq, mk
        return v

    def fwd(vl, qq=q, o=None):
        return lib.sdpa_fwd_varlen(r(qq), r(kk), r(kk), r(vl), 0.0, 1, 0.125, 0, 0, r(qq),
                                   ctypes.c_void_p(FAKE), o, None)

    assert fwd(seqs(cq=None)) == 1                       # offsets missing
    assert fwd(seqs(ck=FAKE + 2)) == 3                   # offsets not 4-byte aligned
    assert fwd(seqs(batch=0)) == 1
    assert fwd(seqs(mq=0)) == 1
    assert fwd(seqs(), qq=desc(2, H, Tq, D)) == 1        # packed tensors are [1, H, total, D]
    keep = desc(1, H, Tq, Tk, stride=(H * Tq * 408, Tq * 408, 408, 1))
    assert fwd(seqs(), o=r(options(attn_bias=ctypes.addressof(keep)))) == 2  # no bias when packed
    assert lib.sdpa_bwd_varlen_workspace_size(None, H, D, None) == 0
    vl = seqs()
    # workspace as for a [batch, H, max_q] problem
    assert (lib.sdpa_bwd_varlen_workspace_size(r(vl), H, D, None)
            == lib.sdpa_bwd_workspace_size(3, H, 128, 256, D))


def test_dropout_bits_size(lib):
    import scaled_dot_product_07_gb300 as sdpa
    # one bit per score of the 128-padded [Sq, Sk] block of every (batch, head)
    assert sdpa.sdpa_dropout_bits_size(2, 3, 200, 300) == 2 * 3 * 256 * 384 // 8
    assert sdpa.sdpa_dropout_bits_size(8, 16, 4096, 4096) == 8 * 16 * 4096 * 4096 // 8
    assert sdpa.sdpa_dropout_bits_size(1, 1, 1, 1) == 128 * 128 // 8
    assert sdpa.sdpa_dropout_bits_size(0, 3, 200, 300) == 0
    assert sdpa.sdpa_dropout_bits_size(2, 3, -1, 300) == 0
    assert sdpa.sdpa_dropout_bits_size(2**30, 2**30, 2**20, 2**20) == 2**64 - 1


def test_dropout_bits_argument_errors(lib):
    import scaled_dot_product_07_gb300 as sdpa
    B, H, S, D = 2, 4, 300, 64
    t = desc(B, H, S, D)
    r = ctypes.byref
    need = sdpa.sdpa_dropout_bits_size(B, H, S, S)

    def fwd(o, tt=t, p=0.1):
        return lib.sdpa_fwd_ex(r(tt), r(tt), r(tt), p, 1, 0.125, 1, 0, r(tt),
                               ctypes.c_void_p(FAKE), r(o), None)

    assert fwd(options(dropout_bits=FAKE + 2, dropout_bits_bytes=need)) == 3  # not 4-byte aligned
    assert fwd(options(dropout_bits=FAKE, dropout_bits_bytes=need - 4)) == 1  # short
    # head dims above 128 and an attention bias have no stored-bits path
    wide = desc(B, H, S, 192)
    assert fwd(options(dropout_bits=FAKE, dropout_bits_bytes=need), tt=wide) == 2
    keep = desc(B, H, S, S, stride=(H * S * 304, S * 304, 304, 1))
    o = options(dropout_bits=FAKE, dropout_bits_bytes=need, attn_bias=ctypes.addressof(keep))
    assert fwd(o) == 2

    def bwd(o, p=0.1):
        return lib.sdpa_bwd_ex(r(t), r(t), r(t), r(t), r(t), ctypes.c_void_p(FAKE), p, 1, 0, 0,
                               0.125, r(t), r(t), r(t), ctypes.c_void_p(FAKE), 1 << 40, r(o), None)

    assert bwd(options(dropout_bits=FAKE, dropout_bits_bytes=need - 1)) == 1
    assert bwd(options(dropout_bits=FAKE + 1, dropout_bits_bytes=need)) == 3
    # a packed batch has no stored-bits path
    vl = sdpa.SdpaVarlen()
    vl.cu_seqlens_q, vl.cu_seqlens_k, vl.batch, vl.max_seqlen_q, vl.max_seqlen_k = FAKE, FAKE, 2, 128, 128
    q = desc(1, H, 200, D, layout="BSHE")
    st = lib.sdpa_fwd_varlen(r(q), r(q), r(q), r(vl), 0.1, 1, 0.125, 0, 0, r(q),
                             ctypes.c_void_p(FAKE),
                             r(options(dropout_bits=FAKE, dropout_bits_bytes=1 << 30)), None)
    assert st == 2
