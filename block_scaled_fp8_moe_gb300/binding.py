"""Thin ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function takes torch tensors, checks dtype/device/contiguity/size on the host, and calls
the C entry point of the same name on the current CUDA stream. There is no fallback: if libmoe.so
is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
lib = ctypes.CDLL(LIB_PATH)

(MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT,
 MOE_ERR_DEVICE_INPUT) = range(7)

EXPORTED = [
    "moe_status_string", "moe_workspace_bytes", "moe_packed_w13_bytes", "moe_packed_w2_bytes",
    "moe_quant_mxfp4", "moe_pack_w13", "moe_pack_w2", "moe_route_topk", "moe_quant_mxfp8",
    "moe_w13_swiglu_grouped", "moe_w2_combine_grouped", "moe_forward", "moe_check_device_status",
    "moe_route_topk_noalloc", "moe_selftest_timeout", "moe_route_topk_anchored", "moe_forward_anchored",
    "moe_packed_shared_w13_bytes", "moe_packed_shared_w2_bytes", "moe_pack_shared_w13", "moe_pack_shared_w2",
    "moe_shared_workspace_bytes", "moe_forward_shared", "moe_dead_from_survival", "moe_w2_grouped", "moe_combine",
    "moe_probe_mma_rate", "moe_quant_mxfp8_plan", "moe_experts_grouped",
]

MOE_FLAG_SWIGLU_DEBUG = 1
MOE_FLAG_X_PLAN_ORDER = 2


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("flags", ctypes.c_int32)]


class MoeSharedExpert(ctypes.Structure):
    _fields_ = [("I", ctypes.c_int32), ("w13", ctypes.c_void_p), ("w13_s", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("w2_s", ctypes.c_void_p), ("ws", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t)]


class MoeIntermediates(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_idx", "topk_w", "expert_counts", "expert_offsets", "xq", "xs", "hq", "hs", "swiglu")]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_SHP = ctypes.POINTER(MoeShape)

lib.moe_status_string.restype = ctypes.c_char_p
lib.moe_status_string.argtypes = [ctypes.c_int]
lib.moe_workspace_bytes.restype = _SZ
lib.moe_workspace_bytes.argtypes = [_SHP]
lib.moe_packed_w13_bytes.restype = _SZ
lib.moe_packed_w13_bytes.argtypes = [_SHP, ctypes.POINTER(_SZ)]
lib.moe_packed_w2_bytes.restype = _SZ
lib.moe_packed_w2_bytes.argtypes = [_SHP, ctypes.POINTER(_SZ)]
lib.moe_quant_mxfp4.argtypes = [_I32, _I32, _P, _P, _P, _P]
lib.moe_quant_mxfp8.argtypes = [_I32, _I32, _P, _P, _P, _P]
lib.moe_quant_mxfp8_plan.argtypes = [_SHP] + [_P] * 6 + [_P]
lib.moe_experts_grouped.argtypes = [_SHP] + [_P] * 12 + [_P, _SZ, _P]
lib.moe_dead_from_survival.argtypes = [_I32, _P, ctypes.c_float, _P, _P]
lib.moe_pack_w13.argtypes = [_SHP, _P, _P, _P, _P, _P]
lib.moe_pack_w2.argtypes = [_SHP, _P, _P, _P, _P, _P]
lib.moe_route_topk.argtypes = [_SHP] + [_P] * 10 + [_P, _SZ, _P]
lib.moe_w13_swiglu_grouped.argtypes = [_SHP] + [_P] * 9 + [_P, _SZ, _P]
lib.moe_w2_combine_grouped.argtypes = [_SHP] + [_P] * 10 + [_P, _SZ, _P]
lib.moe_w2_grouped.argtypes = [_SHP] + [_P] * 7 + [_P, _SZ, _P]
lib.moe_combine.argtypes = [_SHP] + [_P] * 5 + [_P, _SZ, _P]
lib.moe_probe_mma_rate.argtypes = [_I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(ctypes.c_int64), _P, _SZ, _P]
lib.moe_forward.argtypes = [_SHP] + [_P] * 9 + [ctypes.POINTER(MoeIntermediates), _P, _SZ, _P]
lib.moe_check_device_status.argtypes = [_P, _P]
lib.moe_route_topk_noalloc.argtypes = [_SHP] + [_P] * 10 + [_P]
lib.moe_selftest_timeout.argtypes = [_P, ctypes.c_uint64, _P]
lib.moe_route_topk_anchored.argtypes = [_SHP] + [_P] * 11 + [_P, _SZ, _P]
lib.moe_forward_anchored.argtypes = [_SHP] + [_P] * 10 + [ctypes.POINTER(MoeIntermediates), _P, _SZ, _P]
lib.moe_packed_shared_w13_bytes.restype = _SZ
lib.moe_packed_shared_w13_bytes.argtypes = [_SHP, ctypes.POINTER(_SZ)]
lib.moe_packed_shared_w2_bytes.restype = _SZ
lib.moe_packed_shared_w2_bytes.argtypes = [_SHP, ctypes.POINTER(_SZ)]
lib.moe_pack_shared_w13.argtypes = [_SHP, _P, _P, _P, _P, _P]
lib.moe_pack_shared_w2.argtypes = [_SHP, _P, _P, _P, _P, _P]
lib.moe_shared_workspace_bytes.restype = _SZ
lib.moe_shared_workspace_bytes.argtypes = [_SHP, _I32]
lib.moe_forward_shared.argtypes = ([_SHP] + [_P] * 9 + [ctypes.POINTER(MoeSharedExpert), _P,
                                   ctypes.POINTER(MoeIntermediates), _P, _SZ, _P, _P])
for _n in EXPORTED:
    if _n not in ("moe_status_string", "moe_workspace_bytes", "moe_packed_w13_bytes", "moe_packed_w2_bytes",
                  "moe_packed_shared_w13_bytes", "moe_packed_shared_w2_bytes", "moe_shared_workspace_bytes"):
        getattr(lib, _n).restype = ctypes.c_int


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {lib.moe_status_string(code).decode()} ({code})")
        self.code = code


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


def shape(T, H, E, k, I, flags=0) -> MoeShape:
    return MoeShape(int(T), int(H), int(E), int(k), int(I), int(flags))


def _ptr(t: torch.Tensor | None, dtype=None, numel=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} needs {numel} elements, has {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def hs_pitch(I: int) -> int:
    return (I + 127) // 128 * 128 // 32


def moe_workspace_bytes(shp: MoeShape) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(shp)))


def alloc_workspace(shp: MoeShape, device="cuda") -> torch.Tensor:
    n = moe_workspace_bytes(shp)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def moe_packed_w13_bytes(shp: MoeShape) -> tuple[int, int]:
    sb = _SZ(0)
    n = lib.moe_packed_w13_bytes(ctypes.byref(shp), ctypes.byref(sb))
    return int(n), int(sb.value)


def moe_packed_w2_bytes(shp: MoeShape) -> tuple[int, int]:
    sb = _SZ(0)
    n = lib.moe_packed_w2_bytes(ctypes.byref(shp), ctypes.byref(sb))
    return int(n), int(sb.value)


def moe_quant_mxfp4(w: torch.Tensor, q: torch.Tensor | None = None, s: torch.Tensor | None = None, stream=None):
    rows, cols = w.reshape(-1, w.shape[-1]).shape
    q = torch.empty(rows * cols // 2, dtype=torch.uint8, device=w.device) if q is None else q
    s = torch.empty(rows * cols // 32, dtype=torch.uint8, device=w.device) if s is None else s
    _check(lib.moe_quant_mxfp4(rows, cols, _ptr(w, torch.float32, name="w"), _ptr(q, torch.uint8, rows * cols // 2),
                               _ptr(s, torch.uint8, rows * cols // 32), _stream(stream)), "moe_quant_mxfp4")
    return q.view(*w.shape[:-1], cols // 2), s.view(*w.shape[:-1], cols // 32)


def moe_quant_mxfp8(x: torch.Tensor, q: torch.Tensor | None = None, s: torch.Tensor | None = None, stream=None):
    rows, cols = x.reshape(-1, x.shape[-1]).shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device) if q is None else q
    s = torch.empty(rows, cols // 32, dtype=torch.uint8, device=x.device) if s is None else s
    _check(lib.moe_quant_mxfp8(rows, cols, _ptr(x, torch.bfloat16, name="x"), _ptr(q, torch.uint8, rows * cols),
                               _ptr(s, torch.uint8, rows * cols // 32), _stream(stream)), "moe_quant_mxfp8")
    return q, s


def moe_quant_mxfp8_plan(shp: MoeShape, x, plan: "Plan", xq_plan=None, xs_plan=None, xq=None, xs=None,
                         stream=None):
    """MXFP8 codes/scales written to plan rows ([T*k, H] / [T*k, H/32]); token order too if given."""
    S = shp.T * shp.k
    xq_plan = torch.empty(max(S, 1), shp.H, dtype=torch.uint8, device=x.device) if xq_plan is None else xq_plan
    xs_plan = torch.empty(max(S, 1), shp.H // 32, dtype=torch.uint8, device=x.device) if xs_plan is None else xs_plan
    _check(lib.moe_quant_mxfp8_plan(
        ctypes.byref(shp), _ptr(x, torch.bfloat16, shp.T * shp.H, "x"), _ptr(plan.row_of_slot, torch.int32, S),
        _ptr(xq_plan, torch.uint8, S * shp.H), _ptr(xs_plan, torch.uint8, S * shp.H // 32),
        _ptr(xq, torch.uint8, shp.T * shp.H), _ptr(xs, torch.uint8, shp.T * shp.H // 32), _stream(stream)),
        "moe_quant_mxfp8_plan")
    return xq_plan, xs_plan


SURVIVAL_THRESHOLD = 0.2


def moe_dead_from_survival(p_survive: torch.Tensor, threshold: float = SURVIVAL_THRESHOLD,
                           dead: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """u8 [T] dead-row mask: 1 where the fp32 survival estimate is below the threshold."""
    T = p_survive.numel()
    dead = torch.empty(T, dtype=torch.uint8, device=p_survive.device) if dead is None else dead
    _check(lib.moe_dead_from_survival(T, _ptr(p_survive, torch.float32, T, "p_survive"), float(threshold),
                                      _ptr(dead, torch.uint8, T, "dead"), _stream(stream)), "moe_dead_from_survival")
    return dead


def moe_pack_w13(shp: MoeShape, q: torch.Tensor, s: torch.Tensor, stream=None):
    nq, ns = moe_packed_w13_bytes(shp)
    qp = torch.empty(nq, dtype=torch.uint8, device=q.device)
    sp = torch.empty(ns, dtype=torch.uint8, device=q.device)
    _check(lib.moe_pack_w13(ctypes.byref(shp), _ptr(q, torch.uint8, shp.E * 2 * shp.I * shp.H // 2),
                            _ptr(s, torch.uint8, shp.E * 2 * shp.I * shp.H // 32), _ptr(qp), _ptr(sp),
                            _stream(stream)), "moe_pack_w13")
    return qp, sp


def moe_pack_w2(shp: MoeShape, q: torch.Tensor, s: torch.Tensor, stream=None):
    nq, ns = moe_packed_w2_bytes(shp)
    qp = torch.empty(nq, dtype=torch.uint8, device=q.device)
    sp = torch.empty(ns, dtype=torch.uint8, device=q.device)
    _check(lib.moe_pack_w2(ctypes.byref(shp), _ptr(q, torch.uint8, shp.E * shp.H * shp.I // 2),
                           _ptr(s, torch.uint8, shp.E * shp.H * shp.I // 32), _ptr(qp), _ptr(sp),
                           _stream(stream)), "moe_pack_w2")
    return qp, sp


class Plan:
    """Device tensors written by moe_route_topk."""

    def __init__(self, shp: MoeShape, device):
        T, k, E = shp.T, shp.k, shp.E
        self.topk_idx = torch.empty(T, k, dtype=torch.int32, device=device)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=device)
        self.expert_counts = torch.empty(E, dtype=torch.int32, device=device)
        self.expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=device)
        self.slot_of_row = torch.empty(max(T * k, 1), dtype=torch.int32, device=device)
        self.row_of_slot = torch.empty(max(T * k, 1), dtype=torch.int32, device=device)


def moe_route_topk(shp: MoeShape, x, w_router, bias, dead, ws, plan: Plan | None = None, stream=None,
                   anchor=None) -> Plan:
    """anchor (optional int32 [T]): -1 routes the row itself, a >= 0 reuses row a's experts."""
    plan = Plan(shp, x.device) if plan is None else plan
    T, H, E = shp.T, shp.H, shp.E
    _check(lib.moe_route_topk_anchored(
        ctypes.byref(shp), _ptr(x, torch.bfloat16, T * H, "x"), _ptr(w_router, torch.bfloat16, E * H, "w_router"),
        _ptr(bias, torch.float32, E, "bias"), _ptr(dead, torch.uint8, T, "dead"),
        _ptr(anchor, torch.int32, T, "anchor"),
        _ptr(plan.topk_idx), _ptr(plan.topk_w), _ptr(plan.expert_counts), _ptr(plan.expert_offsets),
        _ptr(plan.slot_of_row), _ptr(plan.row_of_slot), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_route_topk_anchored")
    return plan


def moe_route_topk_noalloc(shp: MoeShape, x, w_router, bias, dead, plan: Plan | None = None,
                           stream=None) -> Plan:
    """moe_route_topk without a workspace (scratch inside the library; see include/moe.h)."""
    plan = Plan(shp, x.device) if plan is None else plan
    T, H, E = shp.T, shp.H, shp.E
    _check(lib.moe_route_topk_noalloc(
        ctypes.byref(shp), _ptr(x, torch.bfloat16, T * H, "x"), _ptr(w_router, torch.bfloat16, E * H, "w_router"),
        _ptr(bias, torch.float32, E, "bias"), _ptr(dead, torch.uint8, T, "dead"),
        _ptr(plan.topk_idx), _ptr(plan.topk_w), _ptr(plan.expert_counts), _ptr(plan.expert_offsets),
        _ptr(plan.slot_of_row), _ptr(plan.row_of_slot), _stream(stream)), "moe_route_topk_noalloc")
    return plan


def moe_w13_swiglu_grouped(shp: MoeShape, xq, xs, w13p, w13sp, plan: Plan, ws, hq=None, hs=None, debug=None,
                           stream=None):
    """xq/xs in token order, or in plan order when shp.flags has MOE_FLAG_X_PLAN_ORDER."""
    S = shp.T * shp.k
    dev = xq.device
    rows = S if shp.flags & MOE_FLAG_X_PLAN_ORDER else shp.T
    hq = torch.empty(max(S, 1), shp.I, dtype=torch.uint8, device=dev) if hq is None else hq
    hs = torch.empty(max(S, 1), hs_pitch(shp.I), dtype=torch.uint8, device=dev) if hs is None else hs
    _check(lib.moe_w13_swiglu_grouped(
        ctypes.byref(shp), _ptr(xq, torch.uint8, rows * shp.H), _ptr(xs, torch.uint8, rows * shp.H // 32),
        _ptr(w13p, torch.uint8), _ptr(w13sp, torch.uint8), _ptr(plan.expert_offsets), _ptr(plan.slot_of_row),
        _ptr(hq, torch.uint8, S * shp.I), _ptr(hs, torch.uint8, S * hs_pitch(shp.I)),
        _ptr(debug, torch.float32, S * shp.I), _ptr(ws), ws.numel(), _stream(stream)), "moe_w13_swiglu_grouped")
    return hq, hs


def moe_w2_combine_grouped(shp: MoeShape, hq, hs, w2p, w2sp, plan: Plan, ws, out=None, stream=None, dead=None):
    out = torch.empty(shp.T, shp.H, dtype=torch.bfloat16, device=hq.device) if out is None else out
    _check(lib.moe_w2_combine_grouped(
        ctypes.byref(shp), _ptr(hq, torch.uint8), _ptr(hs, torch.uint8), _ptr(w2p, torch.uint8),
        _ptr(w2sp, torch.uint8), _ptr(plan.topk_w), _ptr(plan.expert_offsets), _ptr(plan.slot_of_row),
        _ptr(plan.row_of_slot), _ptr(dead, torch.uint8, shp.T, "dead"),
        _ptr(out, torch.bfloat16, shp.T * shp.H, "out"), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_w2_combine_grouped")
    return out


def moe_w2_grouped(shp: MoeShape, hq, hs, w2p, w2sp, plan: Plan, ws, y=None, stream=None):
    """Down-projection GEMM alone: fp32 rows y [T*k, H] in plan order, before the routing weight."""
    S = shp.T * shp.k
    y = torch.empty(max(S, 1), shp.H, dtype=torch.float32, device=hq.device) if y is None else y
    _check(lib.moe_w2_grouped(
        ctypes.byref(shp), _ptr(hq, torch.uint8), _ptr(hs, torch.uint8), _ptr(w2p, torch.uint8),
        _ptr(w2sp, torch.uint8), _ptr(plan.expert_offsets), _ptr(plan.slot_of_row),
        _ptr(y, torch.float32, S * shp.H, "y"), _ptr(ws), ws.numel(), _stream(stream)), "moe_w2_grouped")
    return y


def moe_combine(shp: MoeShape, y, plan: Plan, ws, dead=None, out=None, stream=None):
    """Fixed-order combine alone: out[t] = bf16(((w_0 y[r_0] + w_1 y[r_1]) + ...)), dead rows +0."""
    out = torch.empty(shp.T, shp.H, dtype=torch.bfloat16, device=y.device) if out is None else out
    _check(lib.moe_combine(
        ctypes.byref(shp), _ptr(y, torch.float32, shp.T * shp.k * shp.H, "y"),
        _ptr(plan.topk_w, torch.float32, shp.T * shp.k, "topk_w"),
        _ptr(plan.row_of_slot, torch.int32, shp.T * shp.k, "row_of_slot"), _ptr(dead, torch.uint8, shp.T, "dead"),
        _ptr(out, torch.bfloat16, shp.T * shp.H, "out"), _ptr(ws), ws.numel(), _stream(stream)), "moe_combine")
    return out


def moe_experts_grouped(shp: MoeShape, xq, xs, w13p, w13sp, w2p, w2sp, plan: Plan, ws, hq=None, hs=None, y=None,
                        debug=None, stream=None):
    """Both expert GEMMs (one launch for decode-sized batches): hq / hs and plan-order fp32 y."""
    S = shp.T * shp.k
    dev = xq.device
    rows = S if shp.flags & MOE_FLAG_X_PLAN_ORDER else shp.T
    hq = torch.empty(max(S, 1), shp.I, dtype=torch.uint8, device=dev) if hq is None else hq
    hs = torch.empty(max(S, 1), hs_pitch(shp.I), dtype=torch.uint8, device=dev) if hs is None else hs
    y = torch.empty(max(S, 1), shp.H, dtype=torch.float32, device=dev) if y is None else y
    _check(lib.moe_experts_grouped(
        ctypes.byref(shp), _ptr(xq, torch.uint8, rows * shp.H), _ptr(xs, torch.uint8, rows * shp.H // 32),
        _ptr(w13p, torch.uint8), _ptr(w13sp, torch.uint8), _ptr(w2p, torch.uint8), _ptr(w2sp, torch.uint8),
        _ptr(plan.expert_offsets), _ptr(plan.slot_of_row), _ptr(hq, torch.uint8, S * shp.I),
        _ptr(hs, torch.uint8, S * hs_pitch(shp.I)), _ptr(debug, torch.float32, S * shp.I),
        _ptr(y, torch.float32, S * shp.H, "y"), _ptr(ws), ws.numel(), _stream(stream)), "moe_experts_grouped")
    return hq, hs, y


class SharedExpert:
    """A shared expert's packed MXFP8 weights on the device (canonical E4M3 codes and UE8M0 scales
    in, see include/moe.h) and its per-T scratch."""

    def __init__(self, H: int, I: int, q13, s13, q2, s2, stream=None):
        self.H, self.I = H, I
        dev = q13.device
        shp = shape(1, H, 1, 1, I)
        sb = ctypes.c_size_t(0)
        n = lib.moe_packed_shared_w13_bytes(ctypes.byref(shp), ctypes.byref(sb))
        if n == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_packed_shared_w13_bytes")
        self.w13p = torch.empty(n, dtype=torch.uint8, device=dev)
        self.w13sp = torch.empty(sb.value, dtype=torch.uint8, device=dev)
        _check(lib.moe_pack_shared_w13(ctypes.byref(shp), _ptr(q13, torch.uint8, 2 * I * H), _ptr(s13, torch.uint8),
                                       _ptr(self.w13p), _ptr(self.w13sp), _stream(stream)), "moe_pack_shared_w13")
        n = lib.moe_packed_shared_w2_bytes(ctypes.byref(shp), ctypes.byref(sb))
        self.w2p = torch.empty(n, dtype=torch.uint8, device=dev)
        self.w2sp = torch.empty(sb.value, dtype=torch.uint8, device=dev)
        _check(lib.moe_pack_shared_w2(ctypes.byref(shp), _ptr(q2, torch.uint8, H * I), _ptr(s2, torch.uint8),
                                      _ptr(self.w2p), _ptr(self.w2sp), _stream(stream)), "moe_pack_shared_w2")
        self._ws = {}

    def descriptor(self, shp: MoeShape) -> MoeSharedExpert:
        if shp.T not in self._ws:
            n = lib.moe_shared_workspace_bytes(ctypes.byref(shp), self.I)
            if n == 0:
                raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_shared_workspace_bytes")
            self._ws[shp.T] = torch.empty(n, dtype=torch.uint8, device=self.w13p.device)
        ws = self._ws[shp.T]
        return MoeSharedExpert(self.I, self.w13p.data_ptr(), self.w13sp.data_ptr(), self.w2p.data_ptr(),
                               self.w2sp.data_ptr(), ws.data_ptr(), ws.numel())


def moe_forward(shp: MoeShape, x, w_router, bias, dead, w13p, w13sp, w2p, w2sp, ws, out=None,
                inter: dict | None = None, stream=None, anchor=None, shared: SharedExpert | None = None,
                side_stream=None):
    out = torch.empty(shp.T, shp.H, dtype=torch.bfloat16, device=x.device) if out is None else out
    im = None
    if inter:
        im = MoeIntermediates(*[ctypes.c_void_p(inter[n].data_ptr()) if inter.get(n) is not None else None
                                for n, _ in MoeIntermediates._fields_])
    if shared is not None:
        desc = shared.descriptor(shp)
        _check(lib.moe_forward_shared(
            ctypes.byref(shp), _ptr(x, torch.bfloat16, shp.T * shp.H, "x"),
            _ptr(w_router, torch.bfloat16, shp.E * shp.H, "w_router"), _ptr(bias, torch.float32, shp.E, "bias"),
            _ptr(dead, torch.uint8, shp.T, "dead"), _ptr(anchor, torch.int32, shp.T, "anchor"),
            _ptr(w13p, torch.uint8), _ptr(w13sp, torch.uint8), _ptr(w2p, torch.uint8), _ptr(w2sp, torch.uint8),
            ctypes.byref(desc), _ptr(out, torch.bfloat16, shp.T * shp.H, "out"),
            ctypes.byref(im) if im is not None else None, _ptr(ws), ws.numel(), _stream(stream),
            _stream(side_stream) if side_stream is not None else None), "moe_forward_shared")
    elif anchor is None:
        _check(lib.moe_forward(
            ctypes.byref(shp), _ptr(x, torch.bfloat16, shp.T * shp.H, "x"),
            _ptr(w_router, torch.bfloat16, shp.E * shp.H, "w_router"), _ptr(bias, torch.float32, shp.E, "bias"),
            _ptr(dead, torch.uint8, shp.T, "dead"), _ptr(w13p, torch.uint8), _ptr(w13sp, torch.uint8),
            _ptr(w2p, torch.uint8), _ptr(w2sp, torch.uint8), _ptr(out, torch.bfloat16, shp.T * shp.H, "out"),
            ctypes.byref(im) if im is not None else None, _ptr(ws), ws.numel(), _stream(stream)), "moe_forward")
    else:
        _check(lib.moe_forward_anchored(
            ctypes.byref(shp), _ptr(x, torch.bfloat16, shp.T * shp.H, "x"),
            _ptr(w_router, torch.bfloat16, shp.E * shp.H, "w_router"), _ptr(bias, torch.float32, shp.E, "bias"),
            _ptr(dead, torch.uint8, shp.T, "dead"), _ptr(anchor, torch.int32, shp.T, "anchor"),
            _ptr(w13p, torch.uint8), _ptr(w13sp, torch.uint8),
            _ptr(w2p, torch.uint8), _ptr(w2sp, torch.uint8), _ptr(out, torch.bfloat16, shp.T * shp.H, "out"),
            ctypes.byref(im) if im is not None else None, _ptr(ws), ws.numel(), _stream(stream)),
            "moe_forward_anchored")
    return out


def moe_probe_mma_rate(iters: int, ws, mode: int = 0, stream=None) -> tuple[int, int]:
    """Launch the block-scaled MMA rate probe (time it with events on `stream`); returns
    (CTAs, FLOPs of the launch). mode: see include/moe.h (0 = the tensor-peak denominator)."""
    ctas = _I32(0)
    flops = ctypes.c_int64(0)
    _check(lib.moe_probe_mma_rate(int(iters), int(mode), ctypes.byref(ctas), ctypes.byref(flops), _ptr(ws),
                                  ws.numel(), _stream(stream)), "moe_probe_mma_rate")
    return int(ctas.value), int(flops.value)


def moe_selftest_timeout(ws, limit_ns: int, stream=None) -> None:
    _check(lib.moe_selftest_timeout(_ptr(ws), int(limit_ns), _stream(stream)), "moe_selftest_timeout")


def moe_check_device_status(ws, stream=None) -> None:
    _check(lib.moe_check_device_status(_ptr(ws), _stream(stream)), "moe_check_device_status")


class MoeLayer:
    """One routed-expert layer with packed MXFP4 weights resident on the device."""

    def __init__(self, H, E, k, I, w_router, bias, w13p, w13sp, w2p, w2sp):
        self.H, self.E, self.k, self.I = H, E, k, I
        self.w_router, self.bias = w_router, bias
        self.w13p, self.w13sp, self.w2p, self.w2sp = w13p, w13sp, w2p, w2sp
        self._ws: dict[int, torch.Tensor] = {}

    @classmethod
    def from_fp32(cls, w_router, bias, w13, w2, k):
        """w13 fp32 [E, 2I, H], w2 fp32 [E, H, I] on the device -> quantise (MXFP4) and pack."""
        E, I2, H = w13.shape
        I = I2 // 2
        shp = shape(1, H, E, k, I)
        q13, s13 = moe_quant_mxfp4(w13)
        q2, s2 = moe_quant_mxfp4(w2)
        w13p, w13sp = moe_pack_w13(shp, q13, s13)
        w2p, w2sp = moe_pack_w2(shp, q2, s2)
        return cls(H, E, k, I, w_router, bias, w13p, w13sp, w2p, w2sp)

    def shape(self, T, flags=0) -> MoeShape:
        return shape(T, self.H, self.E, self.k, self.I, flags)

    def workspace(self, T) -> torch.Tensor:
        if T not in self._ws:
            self._ws[T] = alloc_workspace(self.shape(T), self.w_router.device)
        return self._ws[T]

    def forward(self, x, dead=None, out=None, inter=None, stream=None, anchor=None, shared=None, side_stream=None):
        T = x.shape[0]
        return moe_forward(self.shape(T), x, self.w_router, self.bias, dead, self.w13p, self.w13sp, self.w2p,
                           self.w2sp, self.workspace(T), out=out, inter=inter, stream=stream, anchor=anchor,
                           shared=shared, side_stream=side_stream)
