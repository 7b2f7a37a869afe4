"""Thin Python binding of the C ABI in include/mx.h (ctypes, argument marshalling
only).  Every step of the MX path runs in the CUDA library; if the library is
not built, the first call raises.

PyTorch supplies device memory and the current stream: tensors are passed by
``data_ptr()``; outputs and workspaces the caller does not pass are allocated
here with ``torch.empty`` (the library itself allocates nothing).
"""
import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmx_gb300.so")

MX_OK = 0
MX_ERR_SHAPE, MX_ERR_ALIGN, MX_ERR_ARG, MX_ERR_NOT_BLOCK32, MX_ERR_SCALE = 1, 2, 3, 4, 5
MX_ERR_WORKSPACE, MX_ERR_EXPERT_ID, MX_ERR_CUDA, MX_ERR_UNSUPPORTED, MX_ERR_TIMEOUT = 6, 7, 8, 9, 10
MX_ERR_INEXACT = 11
MX_FMT_E4M3, MX_FMT_E2M1 = 0, 1
MX_SCALE_BLOCK32X32, MX_SCALE_ROW1X32 = 0, 1
MX_PACK_FOLD, MX_PACK_REQUIRE_BLOCK, MX_PACK_GATE_UP = 1, 2, 4
MX_LAYOUT_PLAIN, MX_LAYOUT_GATE_UP = 0, 1
MX_LINEAR_NO_FUSED_QUANT = 1
MX_LINEAR_CLUSTER_GEMV = 1 << 14
MX_GEMV_MAX_M = 32
MX_MAX_EXPERTS = 512

EXPORTED = ("mx_last_error", "mx_check_device_errors", "mx_pack_size", "mx_pack_weights",
            "mx_quantize_act", "mx_dequant", "mxfp8_linear_workspace_size", "mxfp8_linear",
            "mx_route_experts", "mxfp4_moe_workspace_size", "mxfp4_moe_linear", "mxfp4_moe_linear_w4a8",
            "mxfp8_linear_noalloc", "mxfp4_moe_expert_workspace_size", "mxfp4_moe_expert",
            "mxfp8_linear_q_workspace_size", "mxfp8_linear_q", "mx_e4m3_from_dequant",
            "mx_selftest_bounded_wait", "mx_measure_mxf8_peak")


class MxError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class MxPackedWeightC(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("scale_mode", ctypes.c_int32), ("E", ctypes.c_int32),
                ("N", ctypes.c_int32), ("K", ctypes.c_int32), ("Kp", ctypes.c_int32),
                ("bytes", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p),
                ("neg_zero_count", ctypes.c_int64), ("layout", ctypes.c_int32)]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load_library(path: str = None) -> ctypes.CDLL:
    """Load the shared library and declare its signatures (no GPU needed)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"the MX CUDA library is not built ({p}); run "
                           "`python -m mxfp4_quantized_linear_gb300.build`")
    L = ctypes.CDLL(p)
    vp, i32, sz, u = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
    pw = ctypes.POINTER(MxPackedWeightC)
    sig = {
        "mx_last_error": (ctypes.c_char_p, []),
        "mx_check_device_errors": (i32, []),
        "mx_pack_size": (sz, [i32, i32, i32, i32]),
        "mx_pack_weights": (i32, [vp, vp, i32, i32, i32, i32, i32, u, vp, sz, pw, vp]),
        "mx_quantize_act": (i32, [vp, i32, i32, vp, vp, vp]),
        "mx_dequant": (i32, [vp, vp, i32, i32, i32, i32, vp, vp]),
        "mxfp8_linear_workspace_size": (sz, [i32, pw]),
        "mxfp8_linear": (i32, [vp, i32, pw, vp, vp, u, vp, sz, vp]),
        "mx_route_experts": (i32, [vp, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]),
        "mxfp4_moe_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "mxfp4_moe_linear": (i32, [vp, vp, i32, i32, pw, vp, vp, sz, vp, vp]),
        "mxfp4_moe_linear_w4a8": (i32, [vp, vp, i32, i32, pw, vp, vp, sz, vp, vp]),
        "mxfp8_linear_noalloc": (i32, [vp, i32, pw, vp, vp, vp]),
        "mxfp4_moe_expert_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
        "mxfp8_linear_q_workspace_size": (sz, [i32, pw]),
        "mx_selftest_bounded_wait": (i32, [i32, vp, vp]),
        "mx_measure_mxf8_peak": (i32, [i32, i32, ctypes.POINTER(ctypes.c_double), vp]),
        "mx_e4m3_from_dequant": (i32, [vp, vp, i32, i32, i32, vp, vp, ctypes.POINTER(ctypes.c_int64), vp]),
        "mxfp8_linear_q": (i32, [vp, vp, i32, pw, vp, vp, u, vp, sz, vp]),
        "mxfp4_moe_expert": (i32, [vp, vp, vp, i32, i32, pw, pw, vp, vp, sz, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = L
    return L


def _check(rc: int):
    if rc != MX_OK:
        raise MxError(rc, load_library().mx_last_error().decode())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    if _raw_stream is not None:
        return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _stream_int() -> int:
    """The current stream as a plain int (the decode hot path)."""
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_BF16 = torch.bfloat16


def _ok(t, dtype) -> bool:
    """The common case of _need, without building an error message."""
    return type(t) is torch.Tensor and t.dtype is dtype and t.is_cuda and t.is_contiguous()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class PackedWeight:
    """A packed weight: the device buffer (kept alive here) plus its descriptor."""

    def __init__(self, buf: torch.Tensor, desc: MxPackedWeightC):
        self.buf = buf
        self.desc = desc
        self.ref = ctypes.byref(desc)  # passed to every call

    fmt = property(lambda self: self.desc.fmt)
    scale_mode = property(lambda self: self.desc.scale_mode)
    E = property(lambda self: self.desc.E)
    N = property(lambda self: self.desc.N)
    K = property(lambda self: self.desc.K)
    Kp = property(lambda self: self.desc.Kp)
    neg_zero_count = property(lambda self: int(self.desc.neg_zero_count))

    def _region(self, ptr, n):
        off = ptr - self.buf.data_ptr()
        return self.buf[off: off + n]

    def bytes_tensor(self) -> torch.Tensor:
        """E4M3: [E, N, Kp]; E2M1: tiles [E, ceil(N/128), Kp/128, 128, 64]."""
        d = self.desc
        if d.fmt == MX_FMT_E4M3:
            return self._region(d.bytes, d.E * d.N * d.Kp).view(d.E, d.N, d.Kp)
        rt, kt = (d.N + 127) // 128, d.Kp // 128
        return self._region(d.bytes, d.E * rt * kt * 8192).view(d.E, rt, kt, 128, 64)

    def codes_tensor(self) -> torch.Tensor:
        d = self.desc
        rows = d.N // 32 if d.scale_mode == MX_SCALE_BLOCK32X32 else d.N
        return self._region(d.codes, d.E * rows * (d.Kp // 32)).view(d.E, rows, d.Kp // 32)

    def sf_tensor(self) -> torch.Tensor:
        d = self.desc
        if not d.sf:
            return None
        rt, kt = (d.N + 127) // 128, d.Kp // 128
        return self._region(d.sf, d.E * rt * kt * 512).view(d.E, rt, kt, 512)


def _fmt_code(fmt):
    return {"e4m3": MX_FMT_E4M3, "e2m1": MX_FMT_E2M1, MX_FMT_E4M3: MX_FMT_E4M3,
            MX_FMT_E2M1: MX_FMT_E2M1}[fmt]


def mx_pack_size(fmt, E: int, N: int, K: int) -> int:
    return int(load_library().mx_pack_size(_fmt_code(fmt), E, N, K))


def mx_pack_weights(w_bytes: torch.Tensor, codes: torch.Tensor, fmt="e4m3",
                    flags: int = MX_PACK_FOLD) -> PackedWeight:
    """w_bytes: e4m3 [N, K] / [E, N, K] or fp4x2 [E, N, K/2] (uint8, CUDA);
    codes: [E, rows, K/32] or [rows, K/32] uint8, rows = N or N/32."""
    f = _fmt_code(fmt)
    _need(w_bytes, torch.uint8, "w_bytes")
    _need(codes, torch.uint8, "codes")
    wb = w_bytes if w_bytes.dim() == 3 else w_bytes.unsqueeze(0)
    cb = codes if codes.dim() == 3 else codes.unsqueeze(0)
    E, N, kk = wb.shape
    K = kk if f == MX_FMT_E4M3 else 2 * kk
    size = mx_pack_size(f, E, N, K)
    if size == 0:
        raise MxError(MX_ERR_SHAPE, f"invalid packed shape E={E} N={N} K={K}")
    buf = torch.empty(size, dtype=torch.uint8, device=w_bytes.device)
    desc = MxPackedWeightC()
    _check(load_library().mx_pack_weights(_ptr(wb), _ptr(cb), f, E, N, K, cb.shape[1], flags,
                                          _ptr(buf), size, ctypes.byref(desc), _stream()))
    return PackedWeight(buf, desc)


def mx_quantize_act(x: torch.Tensor):
    """x bf16 [M, K] -> (q uint8 [M, K] e4m3, codes uint8 [M, K/32])."""
    _need(x, torch.bfloat16, "x")
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    c = torch.empty((M, K // 32), dtype=torch.uint8, device=x.device)
    _check(load_library().mx_quantize_act(_ptr(x), M, K, _ptr(q), _ptr(c), _stream()))
    return q, c


def mx_e4m3_from_dequant(w: torch.Tensor, codes: torch.Tensor, scale_mode: int = MX_SCALE_BLOCK32X32,
                         strict: bool = True):
    """bf16 weight [N, K] dequantized as e4m3 x 2^(code - 127), codes [N/32, K/32]
    (or [N, K/32] with MX_SCALE_ROW1X32) -> its e4m3 bytes uint8 [N, K]; raises
    MxError(MX_ERR_INEXACT) when some value is not given back exactly.  With
    ``strict=False`` returns (bytes, number of values not given back) instead."""
    _need(w, torch.bfloat16, "w")
    _need(codes, torch.uint8, "codes")
    N, K = w.shape
    out = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scratch = torch.empty(1, dtype=torch.int64, device=w.device)
    bad = ctypes.c_int64(0)
    rc = load_library().mx_e4m3_from_dequant(_ptr(w), _ptr(codes), scale_mode, N, K, _ptr(out), _ptr(scratch),
                                             ctypes.byref(bad), _stream())
    if not strict and rc == MX_ERR_INEXACT:
        return out, int(bad.value)
    _check(rc)
    return out if strict else (out, 0)


def mx_dequant(w_bytes: torch.Tensor, codes: torch.Tensor, fmt="e4m3",
               scale_mode: int = MX_SCALE_ROW1X32) -> torch.Tensor:
    """e4m3 [N, K] or fp4x2 [N, K/2] bytes with codes -> bf16 [N, K]."""
    f = _fmt_code(fmt)
    _need(w_bytes, torch.uint8, "w_bytes")
    _need(codes, torch.uint8, "codes")
    N = w_bytes.shape[0]
    K = w_bytes.shape[1] * (1 if f == MX_FMT_E4M3 else 2)
    out = torch.empty((N, K), dtype=torch.bfloat16, device=w_bytes.device)
    _check(load_library().mx_dequant(_ptr(w_bytes), _ptr(codes), f, scale_mode, N, K, _ptr(out), _stream()))
    return out


def mxfp8_linear_workspace_size(M: int, w: PackedWeight) -> int:
    return int(load_library().mxfp8_linear_workspace_size(M, ctypes.byref(w.desc)))


def mxfp8_linear(x: torch.Tensor, w: PackedWeight, bias: torch.Tensor = None, out: torch.Tensor = None,
                 flags: int = 0, workspace: torch.Tensor = None) -> torch.Tensor:
    """bf16 x [M, K] @ w^T (+ bias) -> bf16 [M, N]."""
    if not _ok(x, _BF16):
        _need(x, _BF16, "x")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, w.desc.N), dtype=_BF16, device=x.device)
    elif not _ok(out, _BF16):
        _need(out, _BF16, "out")
    if bias is not None and not _ok(bias, _BF16):
        _need(bias, _BF16, "bias")
    if workspace is None:  # the library reports a too-small workspace itself
        need = mxfp8_linear_workspace_size(M, w)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    lib = _lib if _lib is not None else load_library()
    rc = lib.mxfp8_linear(x.data_ptr(), M, w.ref, None if bias is None else bias.data_ptr(), out.data_ptr(),
                          flags, None if workspace is None else workspace.data_ptr(),
                          0 if workspace is None else workspace.numel(), _stream_int())
    if rc != MX_OK:
        _check(rc)
    return out


def mxfp8_linear_q(xq: torch.Tensor, xcodes: torch.Tensor, w: PackedWeight, bias: torch.Tensor = None,
                   out: torch.Tensor = None, workspace: torch.Tensor = None) -> torch.Tensor:
    """Pre-quantized activation: e4m3 bytes xq uint8 [M, K] and row-major E8M0
    codes uint8 [M, K/32] @ w^T (+ bias) -> bf16 [M, N]."""
    _need(xq, torch.uint8, "xq")
    _need(xcodes, torch.uint8, "xcodes")
    M = xq.shape[0]
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.bfloat16, device=xq.device)
    _need(out, torch.bfloat16, "out")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias")
    if workspace is None:
        need = int(load_library().mxfp8_linear_q_workspace_size(M, ctypes.byref(w.desc)))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(load_library().mxfp8_linear_q(_ptr(xq), _ptr(xcodes), M, ctypes.byref(w.desc), _ptr(bias), _ptr(out), 0,
                                         _ptr(workspace), ws_bytes, _stream()))
    return out


def mxfp8_linear_noalloc(x: torch.Tensor, w: PackedWeight, bias: torch.Tensor = None,
                         out: torch.Tensor = None) -> torch.Tensor:
    """mxfp8_linear for M <= 32 without a workspace: the library keeps the
    quantized activation in its own fixed device array, for callers that may
    not allocate (see include/mx.h).  Pass ``out`` to avoid the allocation this
    Python wrapper would otherwise make for the result."""
    _need(x, torch.bfloat16, "x")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias")
    _check(load_library().mxfp8_linear_noalloc(_ptr(x), M, ctypes.byref(w.desc), _ptr(bias), _ptr(out),
                                               _stream()))
    return out


def mx_route_experts(topk_ids: torch.Tensor, E: int, dev_status: torch.Tensor = None) -> dict:
    """topk_ids int32 [T, topk] -> dict of int32 device tensors (see include/mx.h)."""
    _need(topk_ids, torch.int32, "topk_ids")
    T, topk = topk_ids.shape
    dev = topk_ids.device
    r = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
         "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "pairs": torch.empty(max(T * topk, 1), dtype=torch.int32, device=dev),
         "active": torch.full((E,), -1, dtype=torch.int32, device=dev),
         "n_active": torch.empty(1, dtype=torch.int32, device=dev),
         "status": dev_status if dev_status is not None else torch.empty(1, dtype=torch.int32, device=dev)}
    _check(load_library().mx_route_experts(_ptr(topk_ids), T, topk, E, _ptr(r["counts"]), _ptr(r["offsets"]),
                                           _ptr(r["pairs"]), _ptr(r["active"]), _ptr(r["n_active"]),
                                           _ptr(r["status"]), _stream()))
    return r


def mxfp4_moe_workspace_size(T: int, topk: int, E: int, N: int, K: int) -> int:
    return int(load_library().mxfp4_moe_workspace_size(T, topk, E, N, K))


def mxfp4_moe_linear(x: torch.Tensor, topk_ids: torch.Tensor, w: PackedWeight, out: torch.Tensor = None,
                     workspace: torch.Tensor = None, dev_status: torch.Tensor = None) -> torch.Tensor:
    """bf16 x [T, K], int32 topk_ids [T, topk] -> bf16 [T, topk, N]."""
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    T, topk = topk_ids.shape
    if out is None:
        out = torch.empty((T, topk, w.N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    need = mxfp4_moe_workspace_size(T, topk, w.E, w.N, w.K)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(load_library().mxfp4_moe_linear(_ptr(x), _ptr(topk_ids), T, topk, ctypes.byref(w.desc), _ptr(out),
                                           _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream()))
    return out


def mxfp4_moe_linear_w4a8(x: torch.Tensor, topk_ids: torch.Tensor, w: PackedWeight, out: torch.Tensor = None,
                          workspace: torch.Tensor = None, dev_status: torch.Tensor = None) -> torch.Tensor:
    """bf16 x [T, K] (quantized per token to MXFP8 inside the call), int32
    topk_ids [T, topk] -> bf16 [T, topk, N]."""
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    T, topk = topk_ids.shape
    if out is None:
        out = torch.empty((T, topk, w.N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    need = mxfp4_moe_workspace_size(T, topk, w.E, w.N, w.K)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(load_library().mxfp4_moe_linear_w4a8(_ptr(x), _ptr(topk_ids), T, topk, ctypes.byref(w.desc),
                                                _ptr(out), _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                                _stream()))
    return out


def mxfp4_moe_expert_workspace_size(T: int, topk: int, E: int, K: int, I: int, H: int) -> int:
    return int(load_library().mxfp4_moe_expert_workspace_size(T, topk, E, K, I, H))


def mxfp4_moe_expert(x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, w13: PackedWeight,
                     w2: PackedWeight, out: torch.Tensor = None, workspace: torch.Tensor = None,
                     dev_status: torch.Tensor = None) -> torch.Tensor:
    """The routed expert MLP: bf16 x [T, K], int32 topk_ids [T, topk], f32
    topk_weights [T, topk], w13 packed with MX_PACK_GATE_UP, w2 [E, H, I] ->
    bf16 [T, H] (see include/mx.h)."""
    _need(x, torch.bfloat16, "x")
    _need(topk_ids, torch.int32, "topk_ids")
    _need(topk_weights, torch.float32, "topk_weights")
    T, topk = topk_ids.shape
    if out is None:
        out = torch.empty((T, w2.N), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        need = mxfp4_moe_expert_workspace_size(T, topk, w13.E, w13.K, w13.N // 2, w2.N)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(load_library().mxfp4_moe_expert(_ptr(x), _ptr(topk_ids), _ptr(topk_weights), T, topk,
                                           ctypes.byref(w13.desc), ctypes.byref(w2.desc), _ptr(out),
                                           _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream()))
    return out


def mx_measure_mxf8_peak(iters: int = 2000, reps: int = 5) -> float:
    """Dense MXFP8 tensor TFLOP/s of the current device, measured by an
    MMA-only loop on every SM (see include/mx.h); synchronizes."""
    v = ctypes.c_double(0.0)
    _check(load_library().mx_measure_mxf8_peak(iters, reps, ctypes.byref(v), _stream()))
    return float(v.value)


def mx_check_device_errors() -> None:
    _check(load_library().mx_check_device_errors())
