"""Torch-facing wrappers of the C ABI (argument marshalling only).

Every function takes and returns CUDA tensors; outputs are allocated with
torch (device memory plumbing) and every step of the computation runs in the
library's kernels.  Tensors on any other device are rejected: there is no CPU
path.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import call, lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _cuda(*tensors: Optional[torch.Tensor]) -> None:
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("nvfp4 ops take CUDA tensors only (no CPU fallback)")
        if t is not None and not t.is_contiguous():
            raise ValueError("nvfp4 ops take contiguous tensors")


def _u8(*shape: int, device) -> torch.Tensor:
    return torch.empty(*shape, dtype=torch.uint8, device=device)


def sf_bytes(rows: int, K: int) -> int:
    return int(lib().nvfp4_sf_bytes(rows, K))


# --------------------------------------------------------------------------- (a) quantize

def quantize_act(x: torch.Tensor, gs: Optional[torch.Tensor] = None, sf_layout: str = "swizzled",
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """x (M, K) bf16 -> (q (M, K/2) uint8, sf uint8, gs (1,) fp32).

    ``gs=None`` computes the dynamic global scale amax/2688 on the device;
    a given ``gs`` (device fp32 scalar tensor) is used as a static scale.
    """
    _cuda(x, gs)
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    M, K = x.shape
    layout = _lib.SF_SWIZZLED if sf_layout == "swizzled" else _lib.SF_LINEAR
    q = _u8(M, K // 2, device=x.device)
    sf = _u8(sf_bytes(M, K) if layout == _lib.SF_SWIZZLED else M * (K // 16), device=x.device)
    dyn = gs is None
    gs_t = torch.empty(1, dtype=torch.float32, device=x.device) if dyn else gs
    ws_n = int(lib().nvfp4_quantize_workspace_bytes(M, K))
    ws = _u8(ws_n, device=x.device) if dyn else None
    call("nvfp4_quantize_act", x.data_ptr(), M, K, K, _lib.GS_DYNAMIC if dyn else _lib.GS_STATIC, gs_t.data_ptr(),
         q.data_ptr(), sf.data_ptr(), layout, _ptr(ws), ws_n if dyn else 0, _stream(stream))
    return q, sf, gs_t


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, stream=None) -> torch.Tensor:
    """x (M, K) bf16 -> x / rms(x) * gamma, bf16 (the unfused normalisation)."""
    _cuda(x, gamma)
    M, K = x.shape
    y = torch.empty_like(x)
    call("nvfp4_rmsnorm", x.data_ptr(), M, K, K, gamma.data_ptr(), eps, y.data_ptr(), _stream(stream))
    return y


def rmsnorm_quantize(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, gs: Optional[torch.Tensor] = None,
                     sf_layout: str = "swizzled", want_normed: bool = False, stream=None):
    """Fused RMSNorm -> NVFP4: returns (q, sf, gs, x_normed or None)."""
    _cuda(x, gamma, gs)
    M, K = x.shape
    layout = _lib.SF_SWIZZLED if sf_layout == "swizzled" else _lib.SF_LINEAR
    q = _u8(M, K // 2, device=x.device)
    sf = _u8(sf_bytes(M, K) if layout == _lib.SF_SWIZZLED else M * (K // 16), device=x.device)
    dyn = gs is None
    gs_t = torch.empty(1, dtype=torch.float32, device=x.device) if dyn else gs
    xn = torch.empty_like(x) if want_normed else None
    ws_n = int(lib().nvfp4_rmsnorm_quantize_workspace_bytes(M, K))
    ws = _u8(ws_n, device=x.device)
    call("nvfp4_rmsnorm_quantize", x.data_ptr(), M, K, K, gamma.data_ptr(), eps,
         _lib.GS_DYNAMIC if dyn else _lib.GS_STATIC, gs_t.data_ptr(), q.data_ptr(), sf.data_ptr(), layout,
         _ptr(xn), ws.data_ptr(), ws_n, _stream(stream))
    return q, sf, gs_t, xn


def prepare_weights(w: torch.Tensor, sf: torch.Tensor, N: int, K: int, interleave_w13: bool = False,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Checkpoint codes (G, N, K/2) + row-major scales (G, N, K/16) -> prepared (tile-major) codes
    + swizzled scales."""
    _cuda(w, sf)
    G = w.numel() // (N * K // 2)
    w_out = _u8(int(lib().nvfp4_prepared_weight_bytes(G, N, K)), device=w.device)
    sf_out = _u8(G * sf_bytes(N, K), device=w.device)
    call("nvfp4_prepare_weights", w.data_ptr(), sf.data_ptr(), G, N, K,
         _lib.PREP_W13_INTERLEAVE if interleave_w13 else _lib.PREP_PLAIN, w_out.data_ptr(), sf_out.data_ptr(),
         _stream(stream))
    return w_out, sf_out


# --------------------------------------------------------------------------- (e) dense linear

def linear(x: torch.Tensor, w: torch.Tensor, w_sf: torch.Tensor, ws2: torch.Tensor, N: int,
           gs: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """y (M, N) bf16 = (gs * ws2) * deq(quantize(x)) @ deq(W)^T; returns (y, gs)."""
    _cuda(x, w, w_sf, ws2, gs, workspace)
    M, K = x.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    dyn = gs is None
    gs_t = torch.empty(1, dtype=torch.float32, device=x.device) if dyn else gs
    ws_n = int(lib().nvfp4_linear_workspace_bytes(M, K))
    ws = workspace if workspace is not None else _u8(ws_n, device=x.device)
    call("nvfp4_linear", x.data_ptr(), M, K, N, w.data_ptr(), w_sf.data_ptr(), ws2.data_ptr(),
         _lib.GS_DYNAMIC if dyn else _lib.GS_STATIC, gs_t.data_ptr(), y.data_ptr(), ws.data_ptr(), ws.numel(),
         _stream(stream))
    return y, gs_t


def grouped_linear(x: torch.Tensor, w: torch.Tensor, w_sf: torch.Tensor, ws2: torch.Tensor, G: int, N: int,
                   gs: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """x (M, G*K) bf16, W (G, N, K/2) prepared -> y (M, G*N) bf16; group g uses x's K columns g."""
    _cuda(x, w, w_sf, ws2, gs, workspace)
    M, GK = x.shape
    K = GK // G
    y = torch.empty(M, G * N, dtype=torch.bfloat16, device=x.device)
    dyn = gs is None
    gs_t = torch.empty(1, dtype=torch.float32, device=x.device) if dyn else gs
    ws_n = int(lib().nvfp4_grouped_linear_workspace_bytes(M, G, K))
    ws = workspace if workspace is not None else _u8(ws_n, device=x.device)
    call("nvfp4_grouped_linear", x.data_ptr(), M, G, K, N, w.data_ptr(), w_sf.data_ptr(), ws2.data_ptr(),
         _lib.GS_DYNAMIC if dyn else _lib.GS_STATIC, gs_t.data_ptr(), y.data_ptr(), ws.data_ptr(), ws.numel(),
         _stream(stream))
    return y, gs_t


def gemm(xq: torch.Tensor, xsf: torch.Tensor, gs: torch.Tensor, K: int, w: torch.Tensor, w_sf: torch.Tensor,
         ws2: torch.Tensor, N: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """GEMM alone on quantised activations xq (M, K/2) + swizzled xsf."""
    _cuda(xq, xsf, gs, w, w_sf, ws2, out)
    M = xq.shape[0]
    y = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=xq.device)
    call("nvfp4_gemm", xq.data_ptr(), xsf.data_ptr(), gs.data_ptr(), M, K, N, w.data_ptr(), w_sf.data_ptr(),
         ws2.data_ptr(), y.data_ptr(), _stream(stream))
    return y


# --------------------------------------------------------------------------- router gate

def router_prepare(w: torch.Tensor, w_sf_linear: torch.Tensor, ws2: torch.Tensor, E: int, H: int,
                   stream=None) -> torch.Tensor:
    """NVFP4 gate weight (E, H/2) + row-major scales -> bf16 weight after the FP8-E4M3 round trip."""
    _cuda(w, w_sf_linear, ws2)
    wg = torch.empty(E, H, dtype=torch.bfloat16, device=w.device)
    n = int(lib().nvfp4_router_prepare_workspace_bytes(E, H))
    ws = _u8(n, device=w.device)
    call("nvfp4_router_prepare", w.data_ptr(), w_sf_linear.data_ptr(), ws2.data_ptr(), E, H, wg.data_ptr(),
         ws.data_ptr(), n, _stream(stream))
    return wg


def router(x: torch.Tensor, wg: torch.Tensor, topk: int, want_logits: bool = False, stream=None):
    """Dense router: (ids (T, topk) int32, weights (T, topk) fp32, logits (T, E) fp32 or None)."""
    _cuda(x, wg)
    T, H = x.shape
    E = wg.shape[0]
    ids = torch.empty(T, topk, dtype=torch.int32, device=x.device)
    w = torch.empty(T, topk, dtype=torch.float32, device=x.device)
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device) if want_logits else None
    n = int(lib().nvfp4_router_workspace_bytes(T, E))
    ws = _u8(max(n, 256), device=x.device)
    call("nvfp4_router", x.data_ptr(), T, H, wg.data_ptr(), E, topk, ids.data_ptr(), w.data_ptr(), _ptr(logits),
         ws.data_ptr(), ws.numel(), _stream(stream))
    return ids, w, logits


# --------------------------------------------------------------------------- (b) routing

def moe_route(ids: torch.Tensor, E: int, stream=None):
    """ids (T, k) int32 -> counts (E,), offsets (E+1,), sorted_idx (T*k,), inv_idx (T*k,)."""
    _cuda(ids)
    T, k = ids.shape
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_idx = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    inv_idx = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    call("nvfp4_moe_route", ids.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(), sorted_idx.data_ptr(),
         inv_idx.data_ptr(), _stream(stream))
    return counts, offsets, sorted_idx[: T * k], inv_idx[: T * k]


# --------------------------------------------------------------------------- MoE layer

@dataclass
class MoEWeights:
    """Prepared expert weights (see nvfp4_prepare_weights) and their ws2 scalars."""
    E: int
    H: int
    I: int
    w13: torch.Tensor       # (E, 2I, H/2) interleaved
    w13_sf: torch.Tensor
    w13_ws2: torch.Tensor   # (E,) fp32
    w2: torch.Tensor        # (E, H, I/2)
    w2_sf: torch.Tensor
    w2_ws2: torch.Tensor    # (E,)
    sh_w13: Optional[torch.Tensor] = None
    sh_w13_sf: Optional[torch.Tensor] = None
    sh_w2: Optional[torch.Tensor] = None
    sh_w2_sf: Optional[torch.Tensor] = None
    sh_ws2: Optional[torch.Tensor] = None  # (2,) = (w13 ws2, w2 ws2)

    @property
    def has_shared(self) -> bool:
        return self.sh_w13 is not None


def moe_workspace_layout(T: int, H: int, I: int, E: int, topk: int, has_shared: bool) -> _lib.MoeWsLayout:
    L = _lib.MoeWsLayout()
    call("nvfp4_moe_workspace_layout", T, H, I, E, topk, int(has_shared), _lib.ctypes.byref(L))
    return L


def moe_workspace(T: int, H: int, I: int, E: int, topk: int, has_shared: bool, device) -> torch.Tensor:
    n = int(lib().nvfp4_moe_workspace_bytes(T, H, I, E, topk, int(has_shared)))
    if n == 0:
        raise ValueError("unsupported MoE shape")
    return _u8(n, device=device)


def _wp(W: MoEWeights):
    return (W.w13.data_ptr(), W.w13_sf.data_ptr(), W.w13_ws2.data_ptr(), W.w2.data_ptr(), W.w2_sf.data_ptr(),
            W.w2_ws2.data_ptr(), _ptr(W.sh_w13), _ptr(W.sh_w13_sf), _ptr(W.sh_w2), _ptr(W.sh_w2_sf),
            _ptr(W.sh_ws2))


def moe_forward(x: torch.Tensor, ids: torch.Tensor, topk_w: torch.Tensor, W: MoEWeights, a2_gs: torch.Tensor,
                a1_gs: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Routed MoE + shared expert.  Returns (y (T, H) bf16, a1_gs)."""
    _cuda(x, ids, topk_w, a2_gs, a1_gs, workspace, out)
    T, H = x.shape
    k = ids.shape[1]
    dyn = a1_gs is None
    gs_t = torch.empty(1, dtype=torch.float32, device=x.device) if dyn else a1_gs
    ws = workspace if workspace is not None else moe_workspace(T, H, W.I, W.E, k, W.has_shared, x.device)
    y = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=x.device)
    call("nvfp4_moe_forward", x.data_ptr(), T, H, W.I, W.E, k, ids.data_ptr(), topk_w.data_ptr(), *_wp(W),
         _lib.GS_DYNAMIC if dyn else _lib.GS_STATIC, gs_t.data_ptr(), a2_gs.data_ptr(), y.data_ptr(),
         ws.data_ptr(), ws.numel(), _stream(stream))
    return y, gs_t


def moe_dispatch(x, ids, W: MoEWeights, a1_gs: torch.Tensor, dynamic: bool, workspace: torch.Tensor, stream=None):
    T, H = x.shape
    call("nvfp4_moe_dispatch", x.data_ptr(), T, H, W.I, W.E, ids.shape[1], ids.data_ptr(), int(W.has_shared),
         _lib.GS_DYNAMIC if dynamic else _lib.GS_STATIC, a1_gs.data_ptr(), workspace.data_ptr(), workspace.numel(),
         _stream(stream))


def moe_w13(T: int, topk: int, W: MoEWeights, a1_gs, a2_gs, workspace, h_debug=None, stream=None):
    call("nvfp4_moe_w13", T, W.H, W.I, W.E, topk, W.w13.data_ptr(), W.w13_sf.data_ptr(), W.w13_ws2.data_ptr(),
         _ptr(W.sh_w13), _ptr(W.sh_w13_sf), _ptr(W.sh_ws2), a1_gs.data_ptr(), a2_gs.data_ptr(), _ptr(h_debug),
         workspace.data_ptr(), workspace.numel(), _stream(stream))


def moe_w2(T: int, topk: int, topk_w, W: MoEWeights, a2_gs, workspace, stream=None):
    call("nvfp4_moe_w2", T, W.H, W.I, W.E, topk, topk_w.data_ptr(), W.w2.data_ptr(), W.w2_sf.data_ptr(),
         W.w2_ws2.data_ptr(), _ptr(W.sh_w2), _ptr(W.sh_w2_sf), _ptr(W.sh_ws2), a2_gs.data_ptr(),
         workspace.data_ptr(), workspace.numel(), _stream(stream))


def moe_finalize(T: int, topk: int, W: MoEWeights, y, workspace, stream=None):
    call("nvfp4_moe_finalize", T, W.H, W.I, W.E, topk, int(W.has_shared), y.data_ptr(), workspace.data_ptr(),
         workspace.numel(), _stream(stream))


# --------------------------------------------------------------------------- diagnostics

def device_error(stream=None) -> Tuple[int, int]:
    """(status, flags) of the device fault word; synchronises the stream and clears the flags."""
    flags = _lib.ctypes.c_int32(0)
    st = lib().nvfp4_get_device_error(_stream(stream), _lib.ctypes.byref(flags))
    return int(st), int(flags.value)


def debug_wait_timeout(timeout_us: int, stream=None) -> None:
    call("nvfp4_debug_wait_timeout", timeout_us, _stream(stream))
