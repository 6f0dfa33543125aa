"""Python binding of the C ABI in ``include/moe.h`` (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA library.
Tensors are torch CUDA tensors (torch provides device memory and streams);
their data pointers and the current CUDA stream are passed through. If the
library has not been built, :func:`load` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_TIMEOUT = 5
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE_BOUNDS"}

EXPORTS = ["moe_version", "moe_status_string", "moe_workspace_size", "moe_check", "moe_route",
           "moe_permute", "moe_expert_ffn", "moe_combine", "moe_layer_forward", "moe_set_option",
           "moe_get_option", "moe_permute_static", "moe_route_ex", "moe_layer_forward_ex",
           "moe_layer_plan", "moe_selftest_wait_timeout", "moe_launch_count", "moe_selftest_route_tc",
           "moe_layer_forward_host", "moe_host_chunks"]

OPT_GEMM0_A = 0
GEMM0_A_PERMUTED = 0      # dispatch copies token rows to x_perm; GEMM0 loads dense tiles
GEMM0_A_TMA_GATHER = 1    # GEMM0 producer gathers token rows with TMA gather4
GEMM0_A_CP_GATHER = 2     # a GEMM0 producer warp gathers token rows with cp.async
OPT_COMBINE = 1
COMBINE_AUTO = 0          # fused when the last GEMM1 has K >= 4096
COMBINE_FUSED = 1         # GEMM1's epilogue: the last contribution sums the slots
COMBINE_SEPARATE = 2      # a streaming combine kernel after the GEMMs
OPT_GEMM_FUSION = 2
GEMM_FUSION_AUTO = 0      # by shape (the library's table)
GEMM_FUSION_ON = 1        # both routed GEMMs in one persistent launch
GEMM_FUSION_OFF = 2       # two launches
OPT_CTA_GROUP = 3
CTA_GROUP_AUTO = 0        # by rows per expert (the library's table)
CTA_GROUP_ONE = 1         # one CTA per 128 x 256 MMA tile
CTA_GROUP_PAIR = 2        # a 2-CTA cluster per 256 x 256 MMA tile (tcgen05 cta_group::2)
OPT_X_PERM_COPY = 4
X_PERM_COPY_AUTO = 0      # by the library's table
X_PERM_COPY_INLINE = 1    # GEMM0's copy warps fill x_perm while the GEMM runs
X_PERM_COPY_KERNEL = 2    # a copy kernel before GEMM0
OPT_ROUTER = 5
ROUTER_OPT_AUTO = 0       # by the library's table
ROUTER_OPT_FMA = 1        # the FMA routers (the canonical order itself)
ROUTER_OPT_TENSOR = 2     # the tensor-core router wherever it applies


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("F_shared", ctypes.c_int32)]


class StageEvents(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("before_route", "before_permute", "before_gemm0",
                                               "before_gemm1", "before_shared", "before_combine",
                                               "after_combine")]


class Gating(ctypes.Structure):
    _fields_ = [("renormalize", ctypes.c_int32), ("shared_gate", ctypes.c_void_p)]


class RoutingOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_idx", "topk_w", "counts", "offsets", "src_row",
                                               "inv_pos")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("router", "gemm0_a", "combine", "gemm_fusion", "tile_m",
                                              "tile_n", "tile_k", "stages", "cta_group",
                                              "cta_group_gemm1", "x_perm_copy")]


ROUTER_STREAM, ROUTER_SLICED, ROUTER_CLUSTER, ROUTER_BLOCK, ROUTER_TENSOR = 0, 1, 2, 3, 4


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run `python -m token_dispatch_grouped_moe_gb300.build`"
                           " (the MoE layer has no CPU fallback)")
    lib = ctypes.CDLL(path)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(Dims)
    lib.moe_version.restype = ctypes.c_int
    lib.moe_version.argtypes = []
    lib.moe_launch_count.restype = ctypes.c_uint64
    lib.moe_launch_count.argtypes = []
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [ctypes.c_int]
    lib.moe_workspace_size.restype = sz
    lib.moe_workspace_size.argtypes = [D]
    lib.moe_set_option.restype = ctypes.c_int
    lib.moe_set_option.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.moe_get_option.restype = ctypes.c_int
    lib.moe_get_option.argtypes = [ctypes.c_int]
    lib.moe_check.restype = ctypes.c_int
    lib.moe_check.argtypes = [P, P]
    lib.moe_route.restype = ctypes.c_int
    lib.moe_route.argtypes = [D, P, P, P, P, P, P]
    lib.moe_permute.restype = ctypes.c_int
    lib.moe_permute.argtypes = [D, P, P, P, P, P, P, P, P, sz, P]
    lib.moe_permute_static.restype = ctypes.c_int
    lib.moe_permute_static.argtypes = [D, P, P, P, P, P, P, P, P]
    lib.moe_expert_ffn.restype = ctypes.c_int
    lib.moe_expert_ffn.argtypes = [D, P, P, P, P, P, P, P, P, P, sz, P]
    lib.moe_combine.restype = ctypes.c_int
    lib.moe_combine.argtypes = [D, P, i32, P, P]
    lib.moe_route_ex.restype = ctypes.c_int
    lib.moe_route_ex.argtypes = [D, P, P, P, ctypes.POINTER(Gating), P, P, P]
    lib.moe_layer_forward_ex.restype = ctypes.c_int
    lib.moe_layer_forward_ex.argtypes = [D, P, P, P, ctypes.POINTER(Gating), P, P, P, P, P, P, P,
                                         ctypes.POINTER(RoutingOut), P, sz, ctypes.POINTER(StageEvents), P]
    lib.moe_selftest_wait_timeout.restype = ctypes.c_int
    lib.moe_selftest_wait_timeout.argtypes = [i32, P]
    lib.moe_selftest_route_tc.restype = ctypes.c_int
    lib.moe_selftest_route_tc.argtypes = [D, P, P, P, i32, i32, P, P, P, P, ctypes.POINTER(ctypes.c_int64),
                                          P, sz, P]
    lib.moe_layer_plan.restype = ctypes.c_int
    lib.moe_layer_plan.argtypes = [D, ctypes.POINTER(Plan)]
    lib.moe_layer_forward.restype = ctypes.c_int
    lib.moe_layer_forward.argtypes = [D, P, P, P, P, P, P, P, P, P, P, ctypes.POINTER(RoutingOut), P,
                                      sz, ctypes.POINTER(StageEvents), P]
    lib.moe_layer_forward_host.restype = ctypes.c_int
    lib.moe_layer_forward_host.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, P, i32, P, sz, P]
    lib.moe_host_chunks.restype = i32
    lib.moe_host_chunks.argtypes = [D]
    _lib = lib
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ok(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def set_gemm0_a(mode: int) -> None:
    """Choose how GEMM0 obtains its token rows (GEMM0_A_PERMUTED or GEMM0_A_TMA_GATHER)."""
    _ok(load().moe_set_option(OPT_GEMM0_A, int(mode)), "moe_set_option")


def get_gemm0_a() -> int:
    return int(load().moe_get_option(OPT_GEMM0_A))


def set_combine(mode: int) -> None:
    """Choose where the layer sums the expert rows (COMBINE_AUTO / _FUSED / _SEPARATE)."""
    _ok(load().moe_set_option(OPT_COMBINE, int(mode)), "moe_set_option")


def get_combine() -> int:
    return int(load().moe_get_option(OPT_COMBINE))


def set_gemm_fusion(mode: int) -> None:
    """Run the routed GEMMs as one launch or two (GEMM_FUSION_AUTO / _ON / _OFF)."""
    _ok(load().moe_set_option(OPT_GEMM_FUSION, int(mode)), "moe_set_option")


def get_gemm_fusion() -> int:
    return int(load().moe_get_option(OPT_GEMM_FUSION))


def set_cta_group(mode: int) -> None:
    """CTAs per MMA of the dense-A expert GEMMs (CTA_GROUP_AUTO / _ONE / _PAIR)."""
    _ok(load().moe_set_option(OPT_CTA_GROUP, int(mode)), "moe_set_option")


def get_cta_group() -> int:
    return int(load().moe_get_option(OPT_CTA_GROUP))


def set_x_perm_copy(mode: int) -> None:
    """Who fills x_perm for GEMM0 (X_PERM_COPY_AUTO / _INLINE / _KERNEL)."""
    _ok(load().moe_set_option(OPT_X_PERM_COPY, int(mode)), "moe_set_option")


def get_x_perm_copy() -> int:
    return int(load().moe_get_option(OPT_X_PERM_COPY))


def set_router(mode: int) -> None:
    """Which router the layer call runs (ROUTER_OPT_AUTO / _FMA / _TENSOR)."""
    _ok(load().moe_set_option(OPT_ROUTER, int(mode)), "moe_set_option")


def route_tc_selftest(dims: Dims, x, Wg, ws, bias=None, renormalize=True, force_exact=False,
                      want_fast=False, stream=None):
    """The tensor-core router alone (test hook moe_selftest_route_tc).
    Returns (topk_idx, topk_w, fast_logits or None, fast_bound or None,
    number of tokens recomputed in the canonical order)."""
    T, k, E = dims.T, dims.k, dims.E
    dev = x.device
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    fast = torch.empty(T, E, dtype=torch.float32, device=dev) if want_fast else None
    bound = torch.empty(T, dtype=torch.float32, device=dev) if want_fast else None
    n = ctypes.c_int64(0)
    _ok(load().moe_selftest_route_tc(ctypes.byref(dims), _p(x), _p(Wg), _p(bias), int(renormalize),
                                     int(force_exact), _p(idx), _p(w), _p(fast), _p(bound),
                                     ctypes.byref(n), _p(ws), ws.numel(), _stream(stream)),
        "moe_selftest_route_tc")
    return idx, w, fast, bound, int(n.value)


def launch_count() -> int:
    """Kernels this library has launched in this process so far."""
    return int(load().moe_launch_count())


def selftest_wait_timeout(limit_ms: int = 200, stream=None) -> int:
    """Status of the bounded-wait self-test (MOE_ERR_TIMEOUT is the expected one)."""
    return int(load().moe_selftest_wait_timeout(int(limit_ms), _stream(stream)))


def layer_plan(dims: Dims) -> Plan:
    """The configuration moe_layer_forward runs for this shape (host only)."""
    p = Plan()
    _ok(load().moe_layer_plan(ctypes.byref(dims), ctypes.byref(p)), "moe_layer_plan")
    return p


def make_dims(T, H, F, E, k, F_shared=0) -> Dims:
    return Dims(int(T), int(H), int(F), int(E), int(k), int(F_shared))


def workspace_size(dims: Dims) -> int:
    return int(load().moe_workspace_size(ctypes.byref(dims)))


def workspace(dims: Dims, device=None) -> torch.Tensor:
    """A zeroed workspace (uint8) for ``dims``; the zeroed head is the error word."""
    n = workspace_size(dims)
    if n == 0:
        raise MoeError(1, "workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def check(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return (and clear) the device error status in ``ws``."""
    return int(load().moe_check(_p(ws), _stream(stream)))


def _gating(renormalize=True, shared_gate=None):
    if renormalize and shared_gate is None:
        return None
    return Gating(1 if renormalize else 0, None if shared_gate is None else shared_gate.data_ptr())


def route(dims: Dims, x, Wg, bias=None, topk_idx=None, topk_w=None, stream=None, renormalize=True):
    T, k = dims.T, dims.k
    dev = x.device
    topk_idx = topk_idx if topk_idx is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty(T, k, dtype=torch.float32, device=dev)
    g = _gating(renormalize)
    _ok(load().moe_route_ex(ctypes.byref(dims), _p(x), _p(Wg), _p(bias),
                            ctypes.byref(g) if g is not None else None, _p(topk_idx), _p(topk_w),
                            _stream(stream)), "moe_route_ex")
    return topk_idx, topk_w


def permute(dims: Dims, topk_idx, ws, x=None, want_x_perm=False, stream=None):
    R, E = dims.T * dims.k, dims.E
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    src_row = torch.empty(R, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(R, dtype=torch.int32, device=dev)
    x_perm = torch.empty(R, dims.H, dtype=torch.bfloat16, device=dev) if want_x_perm else None
    _ok(load().moe_permute(ctypes.byref(dims), _p(topk_idx), _p(counts), _p(offsets), _p(src_row),
                           _p(inv_pos), _p(x), _p(x_perm), _p(ws), ws.numel(), _stream(stream)),
        "moe_permute")
    return counts, offsets, src_row, inv_pos, x_perm


def permute_static(dims: Dims, topk_idx, x=None, want_x_perm=False, stream=None):
    """Dispatch without a workspace (scratch is a fixed array inside the
    library; calls on one device must not overlap on the GPU)."""
    R, E = dims.T * dims.k, dims.E
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    src_row = torch.empty(R, dtype=torch.int32, device=dev)
    inv_pos = torch.empty(R, dtype=torch.int32, device=dev)
    x_perm = torch.empty(R, dims.H, dtype=torch.bfloat16, device=dev) if want_x_perm else None
    _ok(load().moe_permute_static(ctypes.byref(dims), _p(topk_idx), _p(counts), _p(offsets),
                                  _p(src_row), _p(inv_pos), _p(x), _p(x_perm), _stream(stream)),
        "moe_permute_static")
    return counts, offsets, src_row, inv_pos, x_perm


def expert_ffn(dims: Dims, x, src_row, offsets, W1, W3, W2, topk_w, ws, slot=None, stream=None):
    if slot is None:
        slot = torch.empty(dims.k, dims.T, dims.H, dtype=torch.float32, device=x.device)
    _ok(load().moe_expert_ffn(ctypes.byref(dims), _p(x), _p(src_row), _p(offsets), _p(W1), _p(W3),
                              _p(W2), _p(topk_w), _p(slot), _p(ws), ws.numel(), _stream(stream)),
        "moe_expert_ffn")
    return slot


def combine(dims: Dims, slot, n_slots=None, out=None, stream=None):
    n_slots = n_slots if n_slots is not None else slot.shape[0]
    if out is None:
        out = torch.empty(dims.T, dims.H, dtype=torch.bfloat16, device=slot.device)
    _ok(load().moe_combine(ctypes.byref(dims), _p(slot), int(n_slots), _p(out), _stream(stream)),
        "moe_combine")
    return out


@dataclass
class Routing:
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    src_row: torch.Tensor
    inv_pos: torch.Tensor


def routing_buffers(dims: Dims, device) -> Routing:
    R = dims.T * dims.k
    i32 = dict(dtype=torch.int32, device=device)
    return Routing(torch.empty(dims.T, dims.k, **i32),
                   torch.empty(dims.T, dims.k, dtype=torch.float32, device=device),
                   torch.empty(dims.E, **i32), torch.empty(dims.E + 1, **i32),
                   torch.empty(R, **i32), torch.empty(R, **i32))


def layer_forward(dims: Dims, x, Wg, W1, W3, W2, ws, bias=None, W1s=None, W3s=None, W2s=None,
                  out=None, routing: Routing | None = None, events: StageEvents | None = None,
                  stream=None, renormalize=True, shared_gate=None):
    if out is None:
        out = torch.empty(dims.T, dims.H, dtype=torch.bfloat16, device=x.device)
    r = None
    if routing is not None:
        r = RoutingOut(*(ctypes.c_void_p(getattr(routing, n).data_ptr()) for n in
                         ("topk_idx", "topk_w", "counts", "offsets", "src_row", "inv_pos")))
    g = _gating(renormalize, shared_gate)
    if g is None:
        _ok(load().moe_layer_forward(ctypes.byref(dims), _p(x), _p(Wg), _p(bias), _p(W1), _p(W3), _p(W2),
                                     _p(W1s), _p(W3s), _p(W2s), _p(out),
                                     ctypes.byref(r) if r is not None else None, _p(ws), ws.numel(),
                                     ctypes.byref(events) if events is not None else None,
                                     _stream(stream)), "moe_layer_forward")
    else:
        _ok(load().moe_layer_forward_ex(ctypes.byref(dims), _p(x), _p(Wg), _p(bias), ctypes.byref(g),
                                        _p(W1), _p(W3), _p(W2), _p(W1s), _p(W3s), _p(W2s), _p(out),
                                        ctypes.byref(r) if r is not None else None, _p(ws), ws.numel(),
                                        ctypes.byref(events) if events is not None else None,
                                        _stream(stream)), "moe_layer_forward_ex")
    return out


def layer_forward_host(dims: Dims, x_host, Wg, W1, W3, W2, ws, x_dev, out_dev, out_host=None, bias=None,
                       W1s=None, W3s=None, W2s=None, n_chunks=0, stream=None):
    """moe_layer_forward_host: x_host and out_host in (pinned) host memory,
    x_dev/out_dev device staging buffers of [T, H] bf16; the chunks' copies
    overlap the layer's kernels. Returns out_host (valid once the stream has
    been synchronized)."""
    if out_host is None:
        out_host = torch.empty(dims.T, dims.H, dtype=torch.bfloat16).pin_memory()
    _ok(load().moe_layer_forward_host(ctypes.byref(dims), _p(x_host), _p(Wg), _p(bias), _p(W1), _p(W3), _p(W2),
                                      _p(W1s), _p(W3s), _p(W2s), _p(out_host), _p(x_dev), _p(out_dev),
                                      int(n_chunks), _p(ws), ws.numel(), _stream(stream)),
        "moe_layer_forward_host")
    return out_host


def host_chunks(dims: Dims) -> int:
    return int(load().moe_host_chunks(ctypes.byref(dims)))


class MoELayer:
    """Weights and a workspace on one device; ``forward(x)`` runs the layer."""

    def __init__(self, Wg, W1, W3, W2, k, bias=None, W1s=None, W3s=None, W2s=None):
        self.Wg, self.W1, self.W3, self.W2, self.k, self.bias = Wg, W1, W3, W2, int(k), bias
        self.W1s, self.W3s, self.W2s = W1s, W3s, W2s
        self.H, self.E = Wg.shape
        self.F = W1.shape[2]
        self.Fs = 0 if W1s is None else W1s.shape[1]
        self._ws = None
        self._T = None

    def dims(self, T) -> Dims:
        return make_dims(T, self.H, self.F, self.E, self.k, self.Fs)

    def workspace(self, T):
        if self._ws is None or self._T != T:
            self._ws = workspace(self.dims(T), device=self.Wg.device)
            self._T = T
        return self._ws

    def forward(self, x, out=None, routing=None, events=None, stream=None):
        T = x.shape[0]
        return layer_forward(self.dims(T), x, self.Wg, self.W1, self.W3, self.W2, self.workspace(T),
                             self.bias, self.W1s, self.W3s, self.W2s, out=out, routing=routing,
                             events=events, stream=stream)
