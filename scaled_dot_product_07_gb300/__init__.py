"""Fused scaled-dot-product attention for training on GB300 (sm_103a).

Python binding of the C ABI declared in ``include/sdpa.h``. Every function
here only marshals arguments (torch tensors -> pointers, sizes and strides,
torch's current CUDA stream) and calls the shared library built from
``csrc/``; all computation happens in the library's CUDA kernels. PyTorch
provides device memory and streams. There is no CPU fallback: if the
library is missing or no GPU is present the calls raise.

    out, lse, seed, offset = sdpa_fwd(q, k, v, dropout_p, is_causal, scale)
    dq, dk, dv = sdpa_bwd(dout, q, k, v, out, lse, dropout_p, is_causal,
                          seed, offset, scale)

Tensors have the logical shape [B, H, S, D] (D a multiple of 8 up to 256,
innermost and contiguous) in bfloat16, in any dense order of B, H, S with 16-byte aligned
strides -- e.g. BHSE or BSHE ("DID loop split for SDPA", NVIDIA/Fuser PR
3711, test_sdpa_loop_split). ``lse`` is float32 [B, H, Sq].
"""

import ctypes
import math
import os

__all__ = [
    "SdpaError", "load_library", "library_path", "sdpa_fwd", "sdpa_bwd",
    "sdpa_bwd_workspace_size", "sdpa_dropout_mask_debug", "sdpa_check_device",
    "sdpa_selftest_wait_timeout", "sdpa_status_string", "SDPAFunction", "EXPORTED_SYMBOLS",
    "sdpa_bwd_noalloc", "NOALLOC_SCRATCH_BYTES", "sdpa_fwd_ex", "sdpa_bwd_ex",
    "sdpa_bwd_workspace_size_ex", "sdpa_dropout_mask_debug_ex", "SdpaOptions",
    "sdpa_fwd_varlen", "sdpa_bwd_varlen", "sdpa_bwd_varlen_workspace_size", "SdpaVarlen",
    "sdpa_dropout_bits_size",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libsdpa_gb300.so")
_LIB = None

# Every entry point of include/sdpa.h.
EXPORTED_SYMBOLS = (
    "sdpa_fwd", "sdpa_bwd_workspace_size", "sdpa_bwd", "sdpa_dropout_mask_debug",
    "sdpa_check_device", "sdpa_selftest_wait_timeout", "sdpa_status_string", "sdpa_bwd_noalloc",
    "sdpa_fwd_ex", "sdpa_bwd_workspace_size_ex", "sdpa_bwd_ex", "sdpa_dropout_mask_debug_ex",
    "sdpa_fwd_varlen", "sdpa_bwd_varlen_workspace_size", "sdpa_bwd_varlen", "sdpa_dropout_bits_size",
)

# SDPA_BWD_NOALLOC_SCRATCH_BYTES of include/sdpa.h
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024

SDPA_OK = 0
STATUS_NAMES = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARG", 2: "SDPA_ERR_UNSUPPORTED",
                3: "SDPA_ERR_ALIGNMENT", 4: "SDPA_ERR_CUDA", 5: "SDPA_ERR_DEVICE_TIMEOUT",
                6: "SDPA_ERR_WORKSPACE"}


class SdpaError(RuntimeError):
    """A library call returned a non-zero status."""

    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {sdpa_status_string(status)}")


class SdpaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("size", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4)]


class SdpaVarlen(ctypes.Structure):
    """sdpa_varlen of include/sdpa.h."""
    _fields_ = [("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("batch", ctypes.c_int64), ("max_seqlen_q", ctypes.c_int64),
                ("max_seqlen_k", ctypes.c_int64)]


class SdpaOptions(ctypes.Structure):
    """sdpa_options of include/sdpa.h."""
    _fields_ = [("rng_state", ctypes.c_void_p), ("batch_offset", ctypes.c_int64),
                ("head_offset", ctypes.c_int64), ("total_heads", ctypes.c_int64),
                ("deterministic", ctypes.c_int), ("attn_bias", ctypes.c_void_p),
                ("dbias", ctypes.c_void_p), ("kernel_events", ctypes.c_void_p),
                ("dropout_bits", ctypes.c_void_p), ("dropout_bits_bytes", ctypes.c_size_t)]


def library_path():
    return _LIB_PATH


def load_library(path=None):
    """Load the CUDA library (once). Raises if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    lib = ctypes.CDLL(p)
    P = ctypes.POINTER(SdpaTensor)
    i64, u64, dbl, flt, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_double,
                              ctypes.c_float, ctypes.c_void_p)
    lib.sdpa_fwd.argtypes = [P, P, P, dbl, ctypes.c_int, flt, u64, u64, P, vp, vp]
    lib.sdpa_fwd.restype = ctypes.c_int
    lib.sdpa_bwd_workspace_size.argtypes = [i64, i64, i64, i64, i64]
    lib.sdpa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.sdpa_bwd.argtypes = [P, P, P, P, P, vp, dbl, ctypes.c_int, u64, u64, flt, P, P, P, vp,
                             ctypes.c_size_t, vp]
    lib.sdpa_bwd.restype = ctypes.c_int
    lib.sdpa_bwd_noalloc.argtypes = [P, P, P, P, P, vp, dbl, ctypes.c_int, u64, u64, flt, P, P, P,
                                     vp]
    lib.sdpa_bwd_noalloc.restype = ctypes.c_int
    lib.sdpa_dropout_mask_debug.argtypes = [i64, i64, i64, i64, dbl, u64, u64, vp, vp]
    lib.sdpa_dropout_mask_debug.restype = ctypes.c_int
    lib.sdpa_fwd_ex.argtypes = [P, P, P, dbl, ctypes.c_int, flt, u64, u64, P, vp, vp, vp]
    lib.sdpa_fwd_ex.restype = ctypes.c_int
    lib.sdpa_bwd_workspace_size_ex.argtypes = [i64, i64, i64, i64, i64, vp]
    lib.sdpa_bwd_workspace_size_ex.restype = ctypes.c_size_t
    lib.sdpa_bwd_ex.argtypes = [P, P, P, P, P, vp, dbl, ctypes.c_int, u64, u64, flt, P, P, P, vp,
                                ctypes.c_size_t, vp, vp]
    lib.sdpa_bwd_ex.restype = ctypes.c_int
    lib.sdpa_dropout_mask_debug_ex.argtypes = [i64, i64, i64, i64, dbl, u64, u64, vp, vp, vp]
    lib.sdpa_dropout_mask_debug_ex.restype = ctypes.c_int
    lib.sdpa_fwd_varlen.argtypes = [P, P, P, vp, dbl, ctypes.c_int, flt, u64, u64, P, vp, vp, vp]
    lib.sdpa_fwd_varlen.restype = ctypes.c_int
    lib.sdpa_bwd_varlen_workspace_size.argtypes = [vp, i64, i64, vp]
    lib.sdpa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.sdpa_bwd_varlen.argtypes = [P, P, P, P, P, vp, vp, dbl, ctypes.c_int, u64, u64, flt, P, P,
                                    P, vp, ctypes.c_size_t, vp, vp]
    lib.sdpa_bwd_varlen.restype = ctypes.c_int
    lib.sdpa_dropout_bits_size.argtypes = [i64, i64, i64, i64]
    lib.sdpa_dropout_bits_size.restype = ctypes.c_size_t
    lib.sdpa_check_device.argtypes = [vp]
    lib.sdpa_check_device.restype = ctypes.c_int
    lib.sdpa_selftest_wait_timeout.argtypes = [u64, vp]
    lib.sdpa_selftest_wait_timeout.restype = ctypes.c_int
    lib.sdpa_status_string.argtypes = [ctypes.c_int]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    if path is None:
        _LIB = lib
    return lib


def sdpa_status_string(status):
    return load_library().sdpa_status_string(int(status)).decode()


def _check(status, where):
    if status != SDPA_OK:
        raise SdpaError(status, where)


def _desc(t):
    """Descriptor of a logical [B,H,S,D] tensor (pointer, sizes, element strides)."""
    if t.dim() != 4:
        raise ValueError("expected a 4-D tensor [B, H, S, D]")
    d = SdpaTensor()
    d.data = t.data_ptr() if t.numel() else None
    for i in range(4):
        d.size[i] = t.size(i)
        d.stride[i] = t.stride(i)
    return d


def _stream(device):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_tensor(t, name):
    import torch
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")


def _default_scale(D, scale):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def sdpa_fwd(q, k, v, dropout_p=0.0, is_causal=False, scale=None, seed=None, offset=None,
             out=None, lse=None):
    """Forward. Returns (out, lse, seed, offset).

    ``scale=None`` uses 1/sqrt(D). When dropout is on and ``seed``/``offset``
    are not given, the seed is drawn from torch's default CPU generator and
    the offset is 0; pass the returned values to :func:`sdpa_bwd`.
    """
    import torch
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    B, H, Sq, D = q.shape
    if seed is None:
        seed = int(torch.randint(0, 2**62, (1,)).item()) if dropout_p > 0 else 0
    if offset is None:
        offset = 0
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    dq_, dk_, dv_, do_ = _desc(q), _desc(k), _desc(v), _desc(out)
    st = lib.sdpa_fwd(ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_), float(dropout_p),
                      int(bool(is_causal)), _default_scale(D, scale), int(seed), int(offset),
                      ctypes.byref(do_), ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                      _stream(q.device))
    _check(st, "sdpa_fwd")
    return out, lse, seed, offset


def sdpa_bwd_workspace_size(B, H, Sq, Sk, D):
    return int(load_library().sdpa_bwd_workspace_size(B, H, Sq, Sk, D))


def sdpa_bwd(dout, q, k, v, out, lse, dropout_p=0.0, is_causal=False, seed=0, offset=0,
             scale=None, dq=None, dk=None, dv=None, workspace=None):
    """Backward. Returns (dq, dk, dv) in the layouts of q, k, v."""
    import torch
    lib = load_library()
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_tensor(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = sdpa_bwd_workspace_size(B, H, Sq, Sk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    descs = [_desc(t) for t in (dout, q, k, v, out, dq, dk, dv)]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.sdpa_bwd(refs[0], refs[1], refs[2], refs[3], refs[4],
                      ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                      float(dropout_p), int(bool(is_causal)), int(seed), int(offset),
                      _default_scale(D, scale), refs[5], refs[6], refs[7],
                      ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                      _stream(q.device))
    _check(st, "sdpa_bwd")
    return dq, dk, dv


def sdpa_bwd_noalloc(dout, q, k, v, out, lse, dropout_p=0.0, is_causal=False, seed=0, offset=0,
                     scale=None, dq=None, dk=None, dv=None):
    """Backward without a caller workspace: the library's built-in scratch
    array (NOALLOC_SCRATCH_BYTES) is used instead. For callers that may not
    allocate device memory; the output tensors must still be provided (or
    are allocated here by torch when omitted, for convenience in Python).
    Calls that overlap on the GPU share the scratch and race; keep them on
    one stream."""
    import torch
    lib = load_library()
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_tensor(t, n)
    D = q.shape[3]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    descs = [_desc(t) for t in (dout, q, k, v, out, dq, dk, dv)]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.sdpa_bwd_noalloc(refs[0], refs[1], refs[2], refs[3], refs[4],
                              ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                              float(dropout_p), int(bool(is_causal)), int(seed), int(offset),
                              _default_scale(D, scale), refs[5], refs[6], refs[7],
                              _stream(q.device))
    _check(st, "sdpa_bwd_noalloc")
    return dq, dk, dv


def sdpa_dropout_mask_debug(B, H, Sq, Sk, dropout_p, seed, offset, device="cuda"):
    """uint8 keep mask [B,H,Sq,Sk] from the device Philox routine of the kernels."""
    import torch
    lib = load_library()
    mask = torch.empty((B, H, Sq, Sk), dtype=torch.uint8, device=device)
    st = lib.sdpa_dropout_mask_debug(B, H, Sq, Sk, float(dropout_p), int(seed), int(offset),
                                     ctypes.c_void_p(mask.data_ptr() if mask.numel() else None),
                                     _stream(mask.device))
    _check(st, "sdpa_dropout_mask_debug")
    return mask


def _bias_desc(t, name):
    import torch
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4:
        raise ValueError(f"{name} must be a 4-D bfloat16 CUDA tensor [B or 1, H or 1, Sq, Sk]")
    d = SdpaTensor()
    d.data = t.data_ptr() if t.numel() else None
    for i in range(4):
        d.size[i] = t.size(i)
        d.stride[i] = t.stride(i)
    return d


def _event_handle(e):
    """The cudaEvent_t of a torch.cuda.Event (created by its first record)."""
    h = int(getattr(e, "cuda_event", 0) or 0)
    if h == 0:
        raise ValueError("kernel_events: record each torch.cuda.Event once before passing it "
                         "(torch creates the CUDA event on its first record)")
    return h


def _options(rng_state=None, batch_offset=0, head_offset=0, total_heads=0, deterministic=False,
             attn_bias=None, dbias=None, kernel_events=None, dropout_bits=None):
    """sdpa_options (by pointer) for the *_ex calls; rng_state is a device
    tensor holding {seed, offset} as two 64-bit integers, or None; attn_bias
    and dbias are bfloat16 tensors or None; kernel_events is None or a pair of
    torch.cuda.Event (timing enabled, each recorded once already) that the
    library records around the call's main kernel; dropout_bits is None or a
    contiguous CUDA tensor of sdpa_dropout_bits_size() bytes that carries the
    dropout keep mask from the forward to the backward."""
    o = SdpaOptions()
    o._keep = []
    if dropout_bits is not None:
        if not dropout_bits.is_cuda or not dropout_bits.is_contiguous():
            raise ValueError("dropout_bits must be a contiguous CUDA tensor")
        o.dropout_bits = dropout_bits.data_ptr()
        o.dropout_bits_bytes = dropout_bits.numel() * dropout_bits.element_size()
    if kernel_events is not None:
        a, b = kernel_events
        handles = (ctypes.c_void_p * 2)(_event_handle(a), _event_handle(b))
        o._keep.append(handles)
        o.kernel_events = ctypes.addressof(handles)
    if attn_bias is not None:
        bd = _bias_desc(attn_bias, "attn_bias")
        o._keep.append(bd)
        o.attn_bias = ctypes.addressof(bd)
    if dbias is not None:
        dd = _bias_desc(dbias, "dbias")
        o._keep.append(dd)
        o.dbias = ctypes.addressof(dd)
    if rng_state is not None:
        if not rng_state.is_cuda or rng_state.numel() < 2 or rng_state.element_size() != 8:
            raise ValueError("rng_state must be a CUDA tensor of two 64-bit integers {seed, offset}")
        o.rng_state = rng_state.data_ptr()
    o.batch_offset = int(batch_offset)
    o.head_offset = int(head_offset)
    o.total_heads = int(total_heads)
    o.deterministic = int(bool(deterministic))
    return o


def sdpa_dropout_bits_size(B, H, Sq, Sk):
    """Bytes of the buffer that carries the dropout keep bits of a [B, H, Sq,
    Sk] problem from the forward to the backward (``dropout_bits``)."""
    return int(load_library().sdpa_dropout_bits_size(B, H, Sq, Sk))


def sdpa_fwd_ex(q, k, v, dropout_p=0.0, is_causal=False, scale=None, seed=0, offset=0,
                rng_state=None, batch_offset=0, head_offset=0, total_heads=0, attn_bias=None,
                out=None, lse=None, kernel_events=None, dropout_bits=None):
    """Forward with options: ``rng_state`` (device {seed, offset}, read by the
    kernels when they run, e.g. inside a replayed CUDA graph), the batch /
    head position of this call in a larger split problem, an additive
    bfloat16 ``attn_bias`` [B or 1, H or 1, Sq, Sk] of the scaled scores,
    ``kernel_events`` (a pair of torch.cuda.Event recorded around the forward
    kernel, for timing it alone) and ``dropout_bits`` (a device buffer of
    :func:`sdpa_dropout_bits_size` bytes into which the forward writes its
    dropout keep bits, for a backward given the same buffer). Returns (out,
    lse)."""
    import torch
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    B, H, Sq, D = q.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    opt = _options(rng_state, batch_offset, head_offset, total_heads, attn_bias=attn_bias,
                   kernel_events=kernel_events, dropout_bits=dropout_bits)
    dq_, dk_, dv_, do_ = _desc(q), _desc(k), _desc(v), _desc(out)
    st = lib.sdpa_fwd_ex(ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_), float(dropout_p),
                         int(bool(is_causal)), _default_scale(D, scale), int(seed), int(offset),
                         ctypes.byref(do_), ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                         ctypes.byref(opt), _stream(q.device))
    _check(st, "sdpa_fwd_ex")
    return out, lse


def sdpa_bwd_workspace_size_ex(B, H, Sq, Sk, D, deterministic=False):
    opt = _options(deterministic=deterministic)
    return int(load_library().sdpa_bwd_workspace_size_ex(B, H, Sq, Sk, D, ctypes.byref(opt)))


def sdpa_bwd_ex(dout, q, k, v, out, lse, dropout_p=0.0, is_causal=False, seed=0, offset=0,
                scale=None, rng_state=None, batch_offset=0, head_offset=0, total_heads=0,
                deterministic=False, attn_bias=None, dbias=None, dq=None, dk=None, dv=None,
                workspace=None, kernel_events=None, dropout_bits=None):
    """Backward with options (see :func:`sdpa_fwd_ex`); ``deterministic``
    selects the fixed-order dQ accumulation. ``dbias``: None, True (allocate)
    or a bfloat16 [B, H, Sq, Sk] tensor that receives the bias gradient dS.
    ``kernel_events`` are recorded around the backward's main kernel.
    ``dropout_bits``: the buffer a forward of the same problem filled; the
    backward reads the keep bits from it instead of drawing them.
    Returns (dq, dk, dv), or (dq, dk, dv, dbias) when dbias is requested."""
    import torch
    lib = load_library()
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_tensor(t, n)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dbias is True:
        # key rows padded to 8 elements: the gradient tiles are stored by TMA
        pad = (Sk + 7) // 8 * 8
        dbias = torch.empty((B, H, Sq, pad), dtype=torch.bfloat16, device=q.device)[..., :Sk]
    opt = _options(rng_state, batch_offset, head_offset, total_heads, deterministic, attn_bias,
                   dbias, kernel_events, dropout_bits)
    need = int(lib.sdpa_bwd_workspace_size_ex(B, H, Sq, Sk, D, ctypes.byref(opt)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    descs = [_desc(t) for t in (dout, q, k, v, out, dq, dk, dv)]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.sdpa_bwd_ex(refs[0], refs[1], refs[2], refs[3], refs[4],
                         ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                         float(dropout_p), int(bool(is_causal)), int(seed), int(offset),
                         _default_scale(D, scale), refs[5], refs[6], refs[7],
                         ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                         ctypes.byref(opt), _stream(q.device))
    _check(st, "sdpa_bwd_ex")
    if dbias is not None:
        return dq, dk, dv, dbias
    return dq, dk, dv


def sdpa_dropout_mask_debug_ex(B, H, Sq, Sk, dropout_p, seed=0, offset=0, rng_state=None,
                               batch_offset=0, head_offset=0, total_heads=0, device="cuda"):
    """Keep mask [B,H,Sq,Sk] of a block at (batch_offset, head_offset) of a
    problem with total_heads heads, optionally keyed from device memory."""
    import torch
    lib = load_library()
    mask = torch.empty((B, H, Sq, Sk), dtype=torch.uint8, device=device)
    opt = _options(rng_state, batch_offset, head_offset, total_heads)
    st = lib.sdpa_dropout_mask_debug_ex(B, H, Sq, Sk, float(dropout_p), int(seed), int(offset),
                                        ctypes.byref(opt),
                                        ctypes.c_void_p(mask.data_ptr() if mask.numel() else None),
                                        _stream(mask.device))
    _check(st, "sdpa_dropout_mask_debug_ex")
    return mask


def _packed(t, name):
    """Descriptor of a packed [total, H, D] tensor as the logical [1, H, total, D]."""
    if t.dim() != 3:
        raise ValueError(f"{name} must be a packed [total, H, D] tensor")
    return _desc(t.permute(1, 0, 2).unsqueeze(0))


def _varlen(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k):
    import torch
    for c, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        if not c.is_cuda or c.dtype != torch.int32 or c.dim() != 1:
            raise ValueError(f"{n} must be a 1-D int32 CUDA tensor of batch + 1 offsets")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold batch + 1 offsets")
    vl = SdpaVarlen()
    vl.cu_seqlens_q = cu_seqlens_q.data_ptr()
    vl.cu_seqlens_k = cu_seqlens_k.data_ptr()
    vl.batch = cu_seqlens_q.numel() - 1
    vl.max_seqlen_q = int(max_seqlen_q)
    vl.max_seqlen_k = int(max_seqlen_k)
    return vl


def sdpa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    dropout_p=0.0, is_causal=False, scale=None, seed=None, offset=None,
                    rng_state=None, batch_offset=0, head_offset=0, total_heads=0, out=None,
                    lse=None):
    """Forward of a packed batch: q [total_q, H, D], k, v [total_k, H, D];
    sequence b is rows cu_seqlens_q[b]:cu_seqlens_q[b+1] (queries) and
    cu_seqlens_k[b]:cu_seqlens_k[b+1] (keys). Returns (out [total_q, H, D],
    lse [H, total_q], seed, offset)."""
    import torch
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n)
    Tq, H, D = q.shape
    if seed is None:
        seed = int(torch.randint(0, 2**62, (1,)).item()) if dropout_p > 0 else 0
    if offset is None:
        offset = 0
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, Tq), dtype=torch.float32, device=q.device) if lse is None else lse
    vl = _varlen(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    opt = _options(rng_state, batch_offset, head_offset, total_heads)
    dq_, dk_, dv_, do_ = _packed(q, "q"), _packed(k, "k"), _packed(v, "v"), _packed(out, "out")
    st = lib.sdpa_fwd_varlen(ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_),
                             ctypes.byref(vl), float(dropout_p), int(bool(is_causal)),
                             _default_scale(D, scale), int(seed), int(offset), ctypes.byref(do_),
                             ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                             ctypes.byref(opt), _stream(q.device))
    _check(st, "sdpa_fwd_varlen")
    return out, lse, seed, offset


def sdpa_bwd_varlen_workspace_size(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, H, D,
                                   deterministic=False):
    vl = _varlen(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    opt = _options(deterministic=deterministic)
    return int(load_library().sdpa_bwd_varlen_workspace_size(ctypes.byref(vl), H, D,
                                                             ctypes.byref(opt)))


def sdpa_bwd_varlen(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                    max_seqlen_k, dropout_p=0.0, is_causal=False, seed=0, offset=0, scale=None,
                    rng_state=None, batch_offset=0, head_offset=0, total_heads=0,
                    deterministic=False, dq=None, dk=None, dv=None, workspace=None):
    """Backward of a packed batch (see :func:`sdpa_fwd_varlen`). Returns
    (dq, dk, dv) in the packed layouts of q, k, v."""
    import torch
    lib = load_library()
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _check_tensor(t, n)
    Tq, H, D = q.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    vl = _varlen(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    opt = _options(rng_state, batch_offset, head_offset, total_heads, deterministic)
    need = int(lib.sdpa_bwd_varlen_workspace_size(ctypes.byref(vl), H, D, ctypes.byref(opt)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    descs = [_packed(t, n) for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out"),
                                        (dq, "dq"), (dk, "dk"), (dv, "dv"))]
    refs = [ctypes.byref(d) for d in descs]
    st = lib.sdpa_bwd_varlen(refs[0], refs[1], refs[2], refs[3], refs[4],
                             ctypes.c_void_p(lse.data_ptr() if lse.numel() else None),
                             ctypes.byref(vl), float(dropout_p), int(bool(is_causal)), int(seed),
                             int(offset), _default_scale(D, scale), refs[5], refs[6], refs[7],
                             ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                             ctypes.byref(opt), _stream(q.device))
    _check(st, "sdpa_bwd_varlen")
    return dq, dk, dv


def sdpa_check_device(device="cuda"):
    """Synchronise and return the status of the library's bounded waits (int)."""
    return int(load_library().sdpa_check_device(_stream(device)))


def sdpa_selftest_wait_timeout(limit_ns=50_000_000, device="cuda"):
    """Run the bounded-wait self test; returns the status (5 = timed out as designed)."""
    return int(load_library().sdpa_selftest_wait_timeout(int(limit_ns), _stream(device)))


def _make_function():
    import torch

    class SDPAFunction(torch.autograd.Function):
        """autograd wrapper: forward = sdpa_fwd, backward = sdpa_bwd."""

        @staticmethod
        def forward(ctx, q, k, v, dropout_p=0.0, is_causal=False, scale=None, seed=None):
            out, lse, seed, offset = sdpa_fwd(q, k, v, dropout_p, is_causal, scale, seed)
            ctx.save_for_backward(q, k, v, out, lse)
            ctx.args = (dropout_p, is_causal, seed, offset, scale)
            return out

        @staticmethod
        def backward(ctx, dout):
            q, k, v, out, lse = ctx.saved_tensors
            p, causal, seed, offset, scale = ctx.args
            dq, dk, dv = sdpa_bwd(dout.contiguous(), q, k, v, out, lse, p, causal, seed, offset,
                                  scale)
            return dq, dk, dv, None, None, None, None

    return SDPAFunction


class _LazyFunction:
    _fn = None

    def __getattr__(self, name):
        if _LazyFunction._fn is None:
            _LazyFunction._fn = _make_function()
        return getattr(_LazyFunction._fn, name)


SDPAFunction = _LazyFunction()
