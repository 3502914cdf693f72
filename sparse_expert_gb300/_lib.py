"""ctypes binding of libmoe_gb300.so: argument marshalling only.

Every function here allocates its outputs with torch on the inputs' device,
passes raw pointers, sizes and the current CUDA stream to the C entry point
of the same name, and raises MoEError on a non-OK status.  All arithmetic
runs in the library's CUDA kernels.  There is no fallback: if the library
is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_BAD_INDEX", 6: "MOE_ERR_WORKSPACE", 7: "MOE_ERR_NO_DEVICE"}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {detail}")
        self.status = status


class ForwardLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("topk_idx", "topk_w", "counts", "offsets", "src_token", "dest_row", "row_w",
                 "x_perm", "h", "y", "total")]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run sparse_expert_gb300/build.py (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_S = ctypes.c_int  # moe_status_t

SIGNATURES = {
    "moe_abi_version": (ctypes.c_int, []),
    "moe_status_string": (ctypes.c_char_p, [_S]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_route_topk": (_S, [_P, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "moe_route_topk_grouped": (_S, [_P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "moe_router_packed_bytes": (_SZ, [_I32, _I32]),
    "moe_pack_router_weights": (_S, [_P, _I32, _I32, _P, _P]),
    "moe_router_topk": (_S, [_P, _P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "moe_forward_routed": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "moe_dispatch_scan": (_S, [_P, _P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_dispatch_scan_noalloc": (_S, [_P, _P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "moe_permute": (_S, [_P, _I64, _I32, _P, _I32, _P, _P]),
    "moe_packed_weight_bytes": (_SZ, [_I32, _I32, _I32]),
    "moe_pack_weights": (_S, [_P, _P, _P, _I32, _I32, _I32, _P, _P]),
    "moe_quantize_fp8_blockwise": (_S, [_P, _I64, _P, _P, _P]),
    "moe_dequantize_fp8_blockwise": (_S, [_P, _P, _I64, _P, _P]),
    "moe_fp8_packed_weight_bytes": (_SZ, [_I32, _I32, _I32]),
    "moe_pack_weights_fp8": (_S, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P]),
    "moe_forward_fp8": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_fp8_timed": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "moe_grouped_swiglu_workspace_bytes": (_SZ, []),
    "moe_grouped_swiglu": (_S, [_P, _P, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_S, [_P, _P, _P, _I64, _I32, _I32, _P, _P]),
    "moe_combine_backward": (_S, [_P, _P, _P, _P, _I64, _I32, _I32, _P, _P, _P]),
    "moe_route_backward": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _P, _P]),
    "moe_forward_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_forward_layout": (_S, [_I64, _I32, _I32, _I32, _I32, ctypes.POINTER(ForwardLayout)]),
    "moe_forward": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_timed": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "moe_forward_gathered": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_gathered_timed": (_S, [_P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _SZ, _P, _P]),
    "moe_forward_host": (_S, [_P, _P, _P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _SZ, _P]),
    "moe_read_device_status": (_S, [_P, _P, ctypes.POINTER(_I32)]),
    "moe_get_device_status": (_S, [_P, _P]),
    "moe_dispatch_noalloc_status": (_S, [_P, ctypes.POINTER(_I32)]),
    "moe_selftest_wait_timeout": (_S, [_P, _SZ, _I64, _P]),
    "moe_selftest_activation": (_S, [_P, _I64, _P, _P, _P]),
    "moe_set_tile_schedule": (_S, [_I32]),
    "moe_occupy_sms": (_S, [_I32, _I64, _P]),
    "moe_forward_host_stream": (_S, [_P, _P, _P, _I32, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _SZ,
                                     _P, _P, _P]),
    "moe_grouped_gate_up_save": (_S, [_P, _P, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_swiglu_backward": (_S, [_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                         _SZ, _P]),
    "moe_backward_workspace_bytes": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_backward": (_S, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_backward_timed": (_S, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                _P]),
}
for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoEError(status, where, lib.moe_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _event_handles(events, stream):
    """cudaEvent_t handles of torch events (None: no event at that boundary)."""
    for ev in events:
        if ev is not None and ev.cuda_event == 0:
            ev.record(stream)  # materialise the handle
    return (ctypes.c_void_p * len(events))(*[0 if ev is None else ev.cuda_event for ev in events])


def _contig(t, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def abi_version() -> int:
    return lib.moe_abi_version()


# --------------------------------------------------------------- stage 1
def moe_route_topk(logits, k, renormalize=True, n_groups=1, stream=None):
    """topk_idx int32 [T,k], topk_w fp32 [T,k] of fp32 router logits [T,E];
    n_groups > 1 takes k/n_groups experts from each group of consecutive experts."""
    _contig(logits, torch.float32, "logits")
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    if n_groups == 1:
        _check(lib.moe_route_topk(_ptr(logits), T, E, k, int(bool(renormalize)), _ptr(idx), _ptr(w),
                                  _stream(stream)), "moe_route_topk")
    else:
        _check(lib.moe_route_topk_grouped(_ptr(logits), T, E, k, n_groups, int(bool(renormalize)), _ptr(idx),
                                          _ptr(w), _stream(stream)), "moe_route_topk_grouped")
    return idx, w


def moe_pack_router_weights(w_router, stream=None):
    """Router weights [d, E] bf16 in the fused router's layout (uint8 buffer)."""
    _contig(w_router, torch.bfloat16, "w_router")
    d, E = w_router.shape
    packed = torch.empty(lib.moe_router_packed_bytes(d, E), dtype=torch.uint8, device=w_router.device)
    _check(lib.moe_pack_router_weights(_ptr(w_router), d, E, _ptr(packed), _stream(stream)), "moe_pack_router_weights")
    return packed


def moe_router_topk(x, router_packed, E, k, renormalize=True, stream=None):
    """Fused router: topk_idx [T,k], topk_w [T,k] of logits x @ w_router, never materialised."""
    _contig(x, torch.bfloat16, "x")
    T, d = x.shape
    idx = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    ws = torch.empty(256, dtype=torch.uint8, device=x.device)
    _check(lib.moe_router_topk(_ptr(x), _ptr(router_packed), T, d, E, k, int(bool(renormalize)), _ptr(idx), _ptr(w),
                               _ptr(ws), ws.numel(), _stream(stream)), "moe_router_topk")
    return idx, w


# ------------------------------------------------------------ stages 2-3
def moe_dispatch_workspace_bytes(T, E, k) -> int:
    return lib.moe_dispatch_workspace_bytes(T, E, k)


def moe_dispatch_scan(topk_idx, E, topk_w=None, row_w=True, workspace=None, stream=None):
    """counts [E], offsets [E+1], src_token [P], dest_row [P], row_w [P] (or None)."""
    _contig(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    dev = topk_idx.device
    P = T * k
    if topk_w is not None:
        _contig(topk_w, torch.float32, "topk_w")
    need = lib.moe_dispatch_workspace_bytes(T, E, k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    src = torch.empty(P, dtype=torch.int32, device=dev)
    dst = torch.empty(P, dtype=torch.int32, device=dev)
    rw = torch.empty(P, dtype=torch.float32, device=dev) if (row_w and topk_w is not None) else None
    _check(lib.moe_dispatch_scan(_ptr(topk_idx), _ptr(topk_w), T, E, k, _ptr(counts), _ptr(offsets), _ptr(src),
                                 _ptr(dst), _ptr(rw), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_dispatch_scan")
    return dict(counts=counts, offsets=offsets, src_token=src, dest_row=dst, row_w=rw, workspace=workspace)


def moe_dispatch_scan_noalloc(topk_idx, E, topk_w=None, row_w=True, stream=None):
    """moe_dispatch_scan without a workspace, for callers that cannot
    allocate device memory at call time (the library's fixed 4 MiB device
    scratch is used instead; overlapping calls race on it)."""
    _contig(topk_idx, torch.int32, "topk_idx")
    T, k = topk_idx.shape
    dev = topk_idx.device
    P = T * k
    if topk_w is not None:
        _contig(topk_w, torch.float32, "topk_w")
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    src = torch.empty(P, dtype=torch.int32, device=dev)
    dst = torch.empty(P, dtype=torch.int32, device=dev)
    rw = torch.empty(P, dtype=torch.float32, device=dev) if (row_w and topk_w is not None) else None
    _check(lib.moe_dispatch_scan_noalloc(_ptr(topk_idx), _ptr(topk_w), T, E, k, _ptr(counts), _ptr(offsets),
                                         _ptr(src), _ptr(dst), _ptr(rw), _stream(stream)),
           "moe_dispatch_scan_noalloc")
    return dict(counts=counts, offsets=offsets, src_token=src, dest_row=dst, row_w=rw)


# ---------------------------------------------------------- stage 4 / 5
def moe_permute(x, dest_row, k, stream=None):
    """x_perm [T*k, d] with x_perm[dest_row[t*k+j]] = x[t]."""
    _contig(x, torch.bfloat16, "x")
    _contig(dest_row, torch.int32, "dest_row")
    T, d = x.shape
    out = torch.empty(T * k, d, dtype=torch.bfloat16, device=x.device)
    _check(lib.moe_permute(_ptr(x), T, d, _ptr(dest_row), k, _ptr(out), _stream(stream)), "moe_permute")
    return out


def moe_packed_weight_bytes(E, d, f) -> int:
    return lib.moe_packed_weight_bytes(E, d, f)


def moe_pack_weights(w_gate, w_up, w_down, stream=None):
    """Packed expert weights (uint8 buffer) for moe_grouped_swiglu / moe_forward."""
    for t, n in ((w_gate, "w_gate"), (w_up, "w_up"), (w_down, "w_down")):
        _contig(t, torch.bfloat16, n)
    E, d, f = w_gate.shape
    packed = torch.empty(lib.moe_packed_weight_bytes(E, d, f), dtype=torch.uint8, device=w_gate.device)
    _check(lib.moe_pack_weights(_ptr(w_gate), _ptr(w_up), _ptr(w_down), E, d, f, _ptr(packed), _stream(stream)),
           "moe_pack_weights")
    return packed


def moe_quantize_fp8_blockwise(w, stream=None):
    """(codes uint8 [n], scales fp32 [n/128]) of a bf16 tensor, blocks of 128 in memory order."""
    _contig(w, torch.bfloat16, "w")
    n = w.numel()
    codes = torch.empty(n, dtype=torch.uint8, device=w.device)
    scales = torch.empty(n // 128, dtype=torch.float32, device=w.device)
    _check(lib.moe_quantize_fp8_blockwise(_ptr(w), n, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8_blockwise")
    return codes, scales


def moe_dequantize_fp8_blockwise(codes, scales, shape=None, stream=None):
    """bf16 weights (of ``shape``, flat by default) from codes and per-block scales."""
    _contig(codes, torch.uint8, "codes")
    _contig(scales, torch.float32, "scales")
    n = codes.numel()
    out = torch.empty(n, dtype=torch.bfloat16, device=codes.device)
    _check(lib.moe_dequantize_fp8_blockwise(_ptr(codes), _ptr(scales), n, _ptr(out), _stream(stream)),
           "moe_dequantize_fp8_blockwise")
    return out if shape is None else out.view(shape)


def moe_fp8_packed_weight_bytes(E, d, f) -> int:
    return lib.moe_fp8_packed_weight_bytes(E, d, f)


def moe_pack_weights_fp8(gate, up, down, E, d, f, stream=None):
    """FP8 weights (uint8 buffer) for moe_forward_fp8 from three (codes, scales)
    pairs as moe_quantize_fp8_blockwise returns them for w_gate, w_up [E,d,f]
    and w_down [E,f,d]."""
    for (c, sc), n in ((gate, "gate"), (up, "up"), (down, "down")):
        _contig(c, torch.uint8, n + " codes")
        _contig(sc, torch.float32, n + " scales")
    dev = gate[0].device
    packed = torch.empty(lib.moe_fp8_packed_weight_bytes(E, d, f), dtype=torch.uint8, device=dev)
    _check(lib.moe_pack_weights_fp8(_ptr(gate[0]), _ptr(gate[1]), _ptr(up[0]), _ptr(up[1]), _ptr(down[0]),
                                    _ptr(down[1]), E, d, f, _ptr(packed), _stream(stream)), "moe_pack_weights_fp8")
    return packed


def moe_forward_fp8(x, logits, packed_fp8, E, k, f, renormalize=True, workspace=None, out=None, topk_idx=None,
                    topk_w=None, stream=None):
    """moe_forward with FP8 weights packed by moe_pack_weights_fp8."""
    _contig(x, torch.bfloat16, "x")
    _contig(logits, torch.float32, "logits")
    T, d = x.shape
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_forward_fp8(_ptr(x), _ptr(logits), _ptr(packed_fp8), T, d, E, k, f, int(bool(renormalize)),
                               _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                               _stream(stream)),
           "moe_forward_fp8")
    return out


def moe_forward_fp8_timed(x, logits, packed_fp8, E, k, f, workspace, out, events, renormalize=True, stream=None):
    """moe_forward_fp8 recording events[0..6] at the stage boundaries."""
    T, d = x.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    handles = _event_handles(events, s)
    _check(lib.moe_forward_fp8_timed(_ptr(x), _ptr(logits), _ptr(packed_fp8), T, d, E, k, f, int(bool(renormalize)),
                                     _ptr(out), _ptr(workspace), workspace.numel(), _stream(s), handles),
           "moe_forward_fp8_timed")
    return out


def moe_grouped_swiglu(x_perm, offsets, E, f, packed, row_scale=None, workspace=None, stream=None):
    """(h [P,f], y [P,d]) of the grouped SwiGLU expert MLP."""
    _contig(x_perm, torch.bfloat16, "x_perm")
    _contig(offsets, torch.int32, "offsets")
    P, d = x_perm.shape
    dev = x_perm.device
    if row_scale is not None:
        _contig(row_scale, torch.float32, "row_scale")
    if workspace is None:
        workspace = torch.empty(lib.moe_grouped_swiglu_workspace_bytes(), dtype=torch.uint8, device=dev)
    h = torch.empty(P, f, dtype=torch.bfloat16, device=dev)
    y = torch.empty(P, d, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_grouped_swiglu(_ptr(x_perm), _ptr(offsets), P, E, d, f, _ptr(packed), _ptr(row_scale), _ptr(h),
                                  _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_grouped_swiglu")
    return h, y


def moe_grouped_gate_up_save(x_perm, offsets, E, f, packed, workspace=None, stream=None):
    """(h [P,f], gu [P,2f]): the gate/up GEMM keeping G and U, interleaved per gate/up tile."""
    _contig(x_perm, torch.bfloat16, "x_perm")
    _contig(offsets, torch.int32, "offsets")
    P, d = x_perm.shape
    dev = x_perm.device
    if workspace is None:
        workspace = torch.empty(lib.moe_grouped_swiglu_workspace_bytes(), dtype=torch.uint8, device=dev)
    h = torch.empty(P, f, dtype=torch.bfloat16, device=dev)
    gu = torch.empty(P, 2 * f, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_grouped_gate_up_save(_ptr(x_perm), _ptr(offsets), P, E, d, f, _ptr(packed), _ptr(h), _ptr(gu),
                                        _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_grouped_gate_up_save")
    return h, gu


def gu_split(gu, f):
    """(G [P,f], U [P,f]) from the interleaved [P,2f] layout (a view reshuffle, for checks)."""
    h_t = 64
    t = gu.reshape(gu.shape[0], f // h_t, 2, h_t)
    return t[:, :, 0, :].reshape(gu.shape[0], f), t[:, :, 1, :].reshape(gu.shape[0], f)


def moe_grouped_swiglu_backward(x_perm, h, gu, dy, offsets, E, f, packed, workspace=None, stream=None):
    """dict(dgu, dx_perm, dw_gate, dw_up, dw_down) of the expert MLP backward."""
    for t, name in ((x_perm, "x_perm"), (h, "h"), (gu, "gu"), (dy, "dy")):
        _contig(t, torch.bfloat16, name)
    _contig(offsets, torch.int32, "offsets")
    P, d = x_perm.shape
    dev = x_perm.device
    if workspace is None:
        workspace = torch.empty(lib.moe_grouped_swiglu_workspace_bytes(), dtype=torch.uint8, device=dev)
    r = dict(dgu=torch.empty(P, 2 * f, dtype=torch.bfloat16, device=dev),
             dx_perm=torch.empty(P, d, dtype=torch.bfloat16, device=dev),
             dw_gate=torch.empty(E, d, f, dtype=torch.bfloat16, device=dev),
             dw_up=torch.empty(E, d, f, dtype=torch.bfloat16, device=dev),
             dw_down=torch.empty(E, f, d, dtype=torch.bfloat16, device=dev))
    _check(lib.moe_grouped_swiglu_backward(_ptr(x_perm), _ptr(h), _ptr(gu), _ptr(dy), _ptr(offsets), P, E, d, f,
                                           _ptr(packed), _ptr(r["dgu"]), _ptr(r["dx_perm"]), _ptr(r["dw_gate"]),
                                           _ptr(r["dw_up"]), _ptr(r["dw_down"]), _ptr(workspace), workspace.numel(),
                                           _stream(stream)),
           "moe_grouped_swiglu_backward")
    return r


def _backward_outputs(T, d, E, f, dev):
    return dict(dx=torch.empty(T, d, dtype=torch.bfloat16, device=dev),
                d_logits=torch.empty(T, E, dtype=torch.float32, device=dev),
                dw_gate=torch.empty(E, d, f, dtype=torch.bfloat16, device=dev),
                dw_up=torch.empty(E, d, f, dtype=torch.bfloat16, device=dev),
                dw_down=torch.empty(E, f, d, dtype=torch.bfloat16, device=dev))


def moe_backward(x, logits, packed, dout, E, k, f, renormalize=True, workspace=None, grads=None, stream=None):
    """dict(dx, d_logits, dw_gate, dw_up, dw_down): the layer backward (forward recomputed)."""
    _contig(x, torch.bfloat16, "x")
    _contig(logits, torch.float32, "logits")
    _contig(dout, torch.bfloat16, "dout")
    T, d = x.shape
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib.moe_backward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device=dev)
    g = grads if grads is not None else _backward_outputs(T, d, E, f, dev)
    _check(lib.moe_backward(_ptr(x), _ptr(logits), _ptr(packed), _ptr(dout), T, d, E, k, f, int(bool(renormalize)),
                            _ptr(g["dx"]), _ptr(g["d_logits"]), _ptr(g["dw_gate"]), _ptr(g["dw_up"]),
                            _ptr(g["dw_down"]), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_backward")
    return g


BACKWARD_STAGES = ("recompute_route_index_permute", "recompute_gate_up", "output_grad_rows", "dgrad_down",
                   "dgrad_gate_up", "gate_grad_route_bwd", "wgrad_down", "wgrad_gate_up", "unpermute")


def moe_backward_timed(x, logits, packed, dout, E, k, f, workspace, grads, events, renormalize=True, stream=None):
    """moe_backward recording events[0..9] at the stage boundaries (BACKWARD_STAGES); a None entry records nothing."""
    T, d = x.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    handles = _event_handles(events, s)
    g = grads
    _check(lib.moe_backward_timed(_ptr(x), _ptr(logits), _ptr(packed), _ptr(dout), T, d, E, k, f,
                                  int(bool(renormalize)), _ptr(g["dx"]), _ptr(g["d_logits"]), _ptr(g["dw_gate"]),
                                  _ptr(g["dw_up"]), _ptr(g["dw_down"]), _ptr(workspace), workspace.numel(), _stream(s),
                                  handles),
           "moe_backward_timed")
    return g


def moe_combine(y, dest_row, T, k, topk_w=None, stream=None):
    """out [T, d] = sum_j w[t,j] * y[dest_row[t*k+j]] (w = 1 when topk_w is None)."""
    _contig(y, torch.bfloat16, "y")
    _contig(dest_row, torch.int32, "dest_row")
    if topk_w is not None:
        _contig(topk_w, torch.float32, "topk_w")
    d = y.shape[1]
    out = torch.empty(T, d, dtype=torch.bfloat16, device=y.device)
    _check(lib.moe_combine(_ptr(y), _ptr(dest_row), _ptr(topk_w), T, k, d, _ptr(out), _stream(stream)),
           "moe_combine")
    return out


def moe_combine_backward(dout, mlp_out, dest_row, topk_w, stream=None):
    """(d_mlp_out [T*k, d] bf16, d_topk_w [T, k] fp32) of the output reduction."""
    _contig(dout, torch.bfloat16, "dout")
    _contig(mlp_out, torch.bfloat16, "mlp_out")
    _contig(dest_row, torch.int32, "dest_row")
    _contig(topk_w, torch.float32, "topk_w")
    T, d = dout.shape
    k = topk_w.shape[1]
    dy = torch.empty(T * k, d, dtype=torch.bfloat16, device=dout.device)
    dw = torch.empty(T, k, dtype=torch.float32, device=dout.device)
    _check(lib.moe_combine_backward(_ptr(dout), _ptr(mlp_out), _ptr(dest_row), _ptr(topk_w), T, k, d, _ptr(dy),
                                    _ptr(dw), _stream(stream)), "moe_combine_backward")
    return dy, dw


def moe_route_backward(logits, topk_idx, d_topk_w, renormalize=True, stream=None):
    """d_logits [T, E] fp32 from the gates' gradient (selection held fixed)."""
    _contig(logits, torch.float32, "logits")
    _contig(topk_idx, torch.int32, "topk_idx")
    _contig(d_topk_w, torch.float32, "d_topk_w")
    T, E = logits.shape
    k = topk_idx.shape[1]
    out = torch.empty(T, E, dtype=torch.float32, device=logits.device)
    _check(lib.moe_route_backward(_ptr(logits), _ptr(topk_idx), _ptr(d_topk_w), T, E, k, int(bool(renormalize)),
                                  _ptr(out), _stream(stream)), "moe_route_backward")
    return out


# ------------------------------------------------------------ the layer
def moe_forward_workspace_bytes(T, E, k, d, f) -> int:
    return lib.moe_forward_workspace_bytes(T, E, k, d, f)


def moe_backward_workspace_bytes(T, E, k, d, f) -> int:
    return lib.moe_backward_workspace_bytes(T, E, k, d, f)


def moe_forward_layout(T, E, k, d, f) -> ForwardLayout:
    lay = ForwardLayout()
    _check(lib.moe_forward_layout(T, E, k, d, f, ctypes.byref(lay)), "moe_forward_layout")
    return lay


def moe_forward(x, logits, packed, E, k, f, renormalize=True, workspace=None, out=None, topk_idx=None,
                topk_w=None, stream=None):
    """out [T, d] of the whole layer.  The workspace keeps every intermediate."""
    _contig(x, torch.bfloat16, "x")
    _contig(logits, torch.float32, "logits")
    T, d = x.shape
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_forward(_ptr(x), _ptr(logits), _ptr(packed), T, d, E, k, f, int(bool(renormalize)), _ptr(out),
                           _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward")
    return out


FORWARD_STAGES = ("route", "index", "permute", "gate_up", "down", "combine")


def moe_forward_gathered(x, logits, packed, E, k, f, renormalize=True, workspace=None, out=None, topk_idx=None,
                         topk_w=None, stream=None):
    """moe_forward with the gate/up GEMM gathering its rows from x (no x_perm)."""
    _contig(x, torch.bfloat16, "x")
    _contig(logits, torch.float32, "logits")
    T, d = x.shape
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_forward_gathered(_ptr(x), _ptr(logits), _ptr(packed), T, d, E, k, f, int(bool(renormalize)),
                                    _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                                    _stream(stream)),
           "moe_forward_gathered")
    return out


def moe_forward_gathered_timed(x, logits, packed, E, k, f, workspace, out, events, renormalize=True, stream=None):
    """moe_forward_gathered recording events[0..6] at the stage boundaries."""
    T, d = x.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    handles = _event_handles(events, s)
    _check(lib.moe_forward_gathered_timed(_ptr(x), _ptr(logits), _ptr(packed), T, d, E, k, f, int(bool(renormalize)),
                                          _ptr(out), _ptr(workspace), workspace.numel(), _stream(s), handles),
           "moe_forward_gathered_timed")
    return out


def moe_forward_routed(x, router_packed, packed, E, k, f, renormalize=True, workspace=None, out=None, stream=None):
    """out [T, d] of the whole layer from the tokens and the packed router weights."""
    _contig(x, torch.bfloat16, "x")
    T, d = x.shape
    dev = x.device
    if workspace is None:
        workspace = torch.empty(lib.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device=dev)
    if out is None:
        out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    _check(lib.moe_forward_routed(_ptr(x), _ptr(router_packed), _ptr(packed), T, d, E, k, f, int(bool(renormalize)),
                                  _ptr(out), None, None, _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward_routed")
    return out


def moe_forward_timed(x, logits, packed, E, k, f, workspace, out, events, renormalize=True, stream=None):
    """moe_forward that records events[0..6] (torch.cuda.Event, timing enabled)
    at the stage boundaries on the launching stream; a None entry records
    nothing at its boundary."""
    T, d = x.shape
    s = stream if stream is not None else torch.cuda.current_stream()
    handles = _event_handles(events, s)
    _check(lib.moe_forward_timed(_ptr(x), _ptr(logits), _ptr(packed), T, d, E, k, f, int(bool(renormalize)),
                                 _ptr(out), _ptr(workspace), workspace.numel(), _stream(s), handles),
           "moe_forward_timed")
    return out


def moe_forward_host(x_host, logits_host, out_host, x_dev, logits_dev, out_dev, packed, E, k, f, workspace,
                     renormalize=True, stream=None):
    """moe_forward from host tensors (pinned for full-speed copies); waits for the stream."""
    T, d = x_host.shape
    _check(lib.moe_forward_host(_ptr(x_host), _ptr(logits_host), _ptr(out_host), _ptr(x_dev), _ptr(logits_dev),
                                _ptr(out_dev), _ptr(packed), T, d, E, k, f, int(bool(renormalize)),
                                _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_forward_host")
    return out_host


def moe_forward_host_stream(x_hosts, logits_hosts, out_hosts, x_dev, logits_dev, out_dev, packed, E, k, f,
                            workspace, renormalize=True, stream=None, copy_in=None, copy_out=None):
    """moe_forward over host batches with overlapped copies; *_dev are pairs of device slots."""
    n = len(x_hosts)
    T, d = x_hosts[0].shape
    stream = stream if stream is not None else torch.cuda.current_stream()
    copy_in = copy_in if copy_in is not None else torch.cuda.Stream()
    copy_out = copy_out if copy_out is not None else torch.cuda.Stream()

    def arr(ts):
        return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    _check(lib.moe_forward_host_stream(arr(x_hosts), arr(logits_hosts), arr(out_hosts), n, arr(x_dev),
                                       arr(logits_dev), arr(out_dev), _ptr(packed), T, d, E, k, f,
                                       int(bool(renormalize)), _ptr(workspace), workspace.numel(), _stream(stream),
                                       _stream(copy_in), _stream(copy_out)),
           "moe_forward_host_stream")
    return out_hosts


def moe_selftest_wait_timeout(workspace, limit_ns, stream=None):
    """Runs the bounded-wait check; read the status with moe_read_device_status."""
    _check(lib.moe_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_selftest_activation(z, stream=None):
    """Silu(z) and sigmoid(z), fp32, computed by the device functions of the expert-GEMM epilogues."""
    z = _contig(z, torch.float32, "z")
    silu = torch.empty_like(z)
    sig = torch.empty_like(z)
    _check(lib.moe_selftest_activation(_ptr(z), z.numel(), _ptr(silu), _ptr(sig), _stream(stream)),
           "moe_selftest_activation")
    return silu, sig


TILE_SCHEDULE_DYNAMIC = 0
TILE_SCHEDULE_STATIC = 1


def moe_set_tile_schedule(mode):
    """The paired expert GEMMs' tile schedule for the rest of the process (measurement)."""
    _check(lib.moe_set_tile_schedule(int(mode)), "moe_set_tile_schedule")


def moe_occupy_sms(n_sms, duration_ns, stream=None):
    """A kernel holding n_sms SMs for duration_ns on `stream` (measurement)."""
    _check(lib.moe_occupy_sms(int(n_sms), int(duration_ns), _stream(stream)), "moe_occupy_sms")


def forward_intermediates(workspace, T, E, k, d, f):
    """Views of the intermediates that moe_forward leaves in its workspace."""
    lay = moe_forward_layout(T, E, k, d, f)
    P = T * k

    def view(off, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return workspace[off:off + nbytes].view(dtype)
    return dict(
        counts=view(lay.counts, E, torch.int32),
        offsets=view(lay.offsets, E + 1, torch.int32),
        topk_idx=view(lay.topk_idx, P, torch.int32).view(T, k),
        topk_w=view(lay.topk_w, P, torch.float32).view(T, k),
        src_token=view(lay.src_token, P, torch.int32),
        dest_row=view(lay.dest_row, P, torch.int32),
        row_w=view(lay.row_w, P, torch.float32),
        x_perm=view(lay.x_perm, P * d, torch.bfloat16).view(P, d),
        h=view(lay.h, P * f, torch.bfloat16).view(P, f),
        y=view(lay.y, P * d, torch.bfloat16).view(P, d),
    )


def moe_read_device_status(workspace, stream=None) -> int:
    st = _I32(0)
    _check(lib.moe_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(st)), "moe_read_device_status")
    return st.value


def moe_get_device_status(workspace, stream=None) -> int:
    """The workspace's device status as the C call returns it (0 = MOE_OK,
    4 = MOE_ERR_TIMEOUT, 5 = MOE_ERR_BAD_INDEX); raises only when the read
    itself fails."""
    s = lib.moe_get_device_status(_ptr(workspace), _stream(stream))
    if s in (1, 3):  # MOE_ERR_INVALID_ARG, MOE_ERR_CUDA: the read failed
        _check(s, "moe_get_device_status")
    return s


def moe_dispatch_noalloc_status(stream=None) -> int:
    """Device status of the latest moe_dispatch_scan_noalloc on this device."""
    st = _I32(0)
    _check(lib.moe_dispatch_noalloc_status(_stream(stream), ctypes.byref(st)), "moe_dispatch_noalloc_status")
    return st.value
