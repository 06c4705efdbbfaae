"""Thin Python binding over the libmoedc C ABI.

Argument marshalling only: torch tensors supply device pointers and the
current CUDA stream; every step of layout / dispatch / combine runs in the
library's CUDA kernels.  There is no CPU fallback: if libmoedc.so is missing
or cannot load, every call raises.

Functions named moedc_* mirror the C entry points one to one (caller-owned
outputs, nothing allocated).  layout / dispatch / combine / layout_dispatch
are conveniences that allocate their outputs with torch first.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

OK = 0
ERR_ARG = 1
ERR_CAPACITY = 2
ERR_EXPERT_RANGE = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_UNIMPLEMENTED = 6

BF16 = 0
FP8_E4M3 = 1
SCALES_COL_MAJOR = 0x100    # OR into FP8_E4M3: scales stored [E, H/128, cap]
SCALES_PER_TOKEN = 0x200    # OR into FP8_E4M3: one scale per row, scales [E, cap]
TOKEN_SCALE_MAX_H = 32768   # MOEDC_TOKEN_SCALE_MAX_H

EXPORTED = ("moedc_api_version", "moedc_strerror", "moedc_layout_workspace_bytes",
            "moedc_layout", "moedc_dispatch", "moedc_combine", "moedc_layout_dispatch",
            "moedc_layout_static_scratch", "moedc_dequant_e4m3", "moedc_rank_layout",
            "moedc_rank_dispatch", "moedc_rank_combine", "moedc_combine_e4m3",
            "moedc_layout_dispatch_workspace_bytes", "moedc_test_set_wait_extra")

STATIC_SCRATCH_BYTES = 1 << 20   # MOEDC_STATIC_SCRATCH_BYTES

_lib = None


class MoedcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (status {code})")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmoedc.so (built in-tree by __graft_entry__.build()).  Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libmoedc.so not found at {p}: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.moedc_api_version.argtypes = []
    lib.moedc_api_version.restype = I
    lib.moedc_strerror.argtypes = [I]
    lib.moedc_strerror.restype = ctypes.c_char_p
    lib.moedc_layout_workspace_bytes.argtypes = [I, I, I, I]
    lib.moedc_layout_workspace_bytes.restype = Z
    lib.moedc_layout_dispatch_workspace_bytes.argtypes = [I, I, I, I]
    lib.moedc_layout_dispatch_workspace_bytes.restype = Z
    lib.moedc_layout.argtypes = [P, I, I, I, I, I, P, P, P, P, P, Z, P, P]
    lib.moedc_layout.restype = I
    lib.moedc_dispatch.argtypes = [P, I, I, P, P, P, I, I, I, I, P, P, P, P, P]
    lib.moedc_dispatch.restype = I
    lib.moedc_combine.argtypes = [P, I, I, I, P, P, P, I, I, P, P, P]
    lib.moedc_combine.restype = I
    lib.moedc_layout_dispatch.argtypes = [P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, Z,
                                          P, P]
    lib.moedc_layout_dispatch.restype = I
    lib.moedc_layout_static_scratch.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P]
    lib.moedc_layout_static_scratch.restype = I
    lib.moedc_dequant_e4m3.argtypes = [P, P, I, P, I, I, I, P, P]
    lib.moedc_dequant_e4m3.restype = I
    lib.moedc_rank_layout.argtypes = [P, I, I, I, P, P, P]
    lib.moedc_rank_layout.restype = I
    lib.moedc_rank_dispatch.argtypes = [P, I, I, P, P, I, I, I, P, P, P, P]
    lib.moedc_rank_dispatch.restype = I
    lib.moedc_rank_combine.argtypes = [P, I, I, I, P, I, P, P]
    lib.moedc_rank_combine.restype = I
    lib.moedc_combine_e4m3.argtypes = [P, P, I, I, I, I, P, P, P, I, I, P, P, P]
    lib.moedc_combine_e4m3.restype = I
    lib.moedc_test_set_wait_extra.argtypes = [ctypes.c_uint]
    lib.moedc_test_set_wait_extra.restype = None
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().moedc_strerror(int(code)).decode()
    except Exception:  # the library itself is missing
        return f"status {code}"


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(code: int, where: str) -> None:
    if code != OK:
        raise MoedcError(code, where)


# ------------------------------------------------------------ raw entry points


def moedc_layout_workspace_bytes(T: int, K: int, E: int, R: int) -> int:
    return int(load().moedc_layout_workspace_bytes(T, K, E, R))


def moedc_layout_dispatch_workspace_bytes(T: int, K: int, E: int, R: int) -> int:
    return int(load().moedc_layout_dispatch_workspace_bytes(T, K, E, R))


def moedc_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,
                 is_token_in_rank, slot, workspace, workspace_bytes, dev_status,
                 stream=None) -> int:
    return load().moedc_layout(_p(topk_idx), T, K, E, R, cap, _p(num_tokens_per_expert),
                               _p(num_tokens_per_rank), _p(is_token_in_rank), _p(slot),
                               _p(workspace), workspace_bytes, _p(dev_status), _stream(stream))


def moedc_layout_static_scratch(topk_idx, T, K, E, R, cap, num_tokens_per_expert,
                                num_tokens_per_rank, is_token_in_rank, slot, dev_status,
                                stream=None) -> int:
    """moedc_layout without a workspace: for callers that cannot allocate
    device memory, the library's own fixed-size device array serves as
    scratch.  Calls that overlap on the GPU race on that array."""
    return load().moedc_layout_static_scratch(
        _p(topk_idx), T, K, E, R, cap, _p(num_tokens_per_expert), _p(num_tokens_per_rank),
        _p(is_token_in_rank), _p(slot), _p(dev_status), _stream(stream))


def moedc_dispatch(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, out_dtype, recv,
                   scales, src_idx, dev_status, stream=None) -> int:
    return load().moedc_dispatch(_p(x), T, H, _p(topk_idx), _p(slot), _p(num_tokens_per_expert),
                                 K, E, cap, out_dtype, _p(recv), _p(scales), _p(src_idx),
                                 _p(dev_status), _stream(stream))


def moedc_combine(expert_out, E, cap, H, topk_idx, slot, topk_weights, T, K, y, dev_status,
                  stream=None) -> int:
    return load().moedc_combine(_p(expert_out), E, cap, H, _p(topk_idx), _p(slot),
                                _p(topk_weights), T, K, _p(y), _p(dev_status), _stream(stream))


def moedc_layout_dispatch(x, topk_idx, T, H, K, E, R, cap, out_dtype, num_tokens_per_expert,
                          num_tokens_per_rank, is_token_in_rank, slot, recv, scales, src_idx,
                          workspace, workspace_bytes, dev_status, stream=None) -> int:
    return load().moedc_layout_dispatch(
        _p(x), _p(topk_idx), T, H, K, E, R, cap, out_dtype, _p(num_tokens_per_expert),
        _p(num_tokens_per_rank), _p(is_token_in_rank), _p(slot), _p(recv), _p(scales),
        _p(src_idx), _p(workspace), workspace_bytes, _p(dev_status), _stream(stream))


def moedc_dequant_e4m3(recv, scales, scale_layout, num_tokens_per_expert, E, cap, H, out,
                       stream=None) -> int:
    return load().moedc_dequant_e4m3(_p(recv), _p(scales), scale_layout,
                                     _p(num_tokens_per_expert), E, cap, H, _p(out),
                                     _stream(stream))


def moedc_combine_e4m3(expert_out, expert_scales, scale_layout, E, cap, H, topk_idx, slot,
                       topk_weights, T, K, y, dev_status, stream=None) -> int:
    return load().moedc_combine_e4m3(_p(expert_out), _p(expert_scales), scale_layout, E, cap, H,
                                     _p(topk_idx), _p(slot), _p(topk_weights), T, K, _p(y),
                                     _p(dev_status), _stream(stream))


def moedc_rank_layout(is_token_in_rank, T, R, cap_rank, rank_slot, dev_status, stream=None) -> int:
    return load().moedc_rank_layout(_p(is_token_in_rank), T, R, cap_rank, _p(rank_slot),
                                    _p(dev_status), _stream(stream))


def moedc_rank_dispatch(x, T, H, rank_slot, num_tokens_per_rank, R, cap_rank, out_dtype,
                        recv_rank, scales_rank, rank_src_idx, stream=None) -> int:
    return load().moedc_rank_dispatch(_p(x), T, H, _p(rank_slot), _p(num_tokens_per_rank), R,
                                      cap_rank, out_dtype, _p(recv_rank), _p(scales_rank),
                                      _p(rank_src_idx), _stream(stream))


def moedc_rank_combine(rank_out, R, cap_rank, H, rank_slot, T, y, stream=None) -> int:
    return load().moedc_rank_combine(_p(rank_out), R, cap_rank, H, _p(rank_slot), T, _p(y),
                                     _stream(stream))


# ---------------------------------------------------------------- conveniences


@dataclass
class Layout:
    num_tokens_per_expert: torch.Tensor   # int32 [E]
    num_tokens_per_rank: torch.Tensor     # int32 [R]
    is_token_in_rank: torch.Tensor        # uint8 [T, R]
    slot: torch.Tensor                    # int32 [T, K]
    status: torch.Tensor                  # int32 [1] (device)


def _dev_i32(n, device):
    return torch.empty(n, dtype=torch.int32, device=device)


def _need(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def layout_workspace(T: int, K: int, E: int, R: int, device) -> torch.Tensor | None:
    n = moedc_layout_workspace_bytes(T, K, E, R)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None


def layout_dispatch_workspace(T: int, K: int, E: int, R: int, device) -> torch.Tensor | None:
    """Workspace that lets moedc_layout_dispatch run as one launch at any T
    (uninitialised memory is fine; do not share it between concurrent calls)."""
    n = moedc_layout_dispatch_workspace_bytes(T, K, E, R)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None


def layout(topk_idx: torch.Tensor, E: int, R: int, cap: int,
           workspace: torch.Tensor | None = None, status: torch.Tensor | None = None) -> Layout:
    _need(topk_idx, torch.int32, "topk_idx")
    T, K = topk_idx.shape
    dev = topk_idx.device
    out = Layout(_dev_i32(E, dev), _dev_i32(R, dev),
                 torch.empty((T, R), dtype=torch.uint8, device=dev), _dev_i32((T, K), dev),
                 status if status is not None else torch.zeros(1, dtype=torch.int32, device=dev))
    if workspace is None:
        workspace = layout_workspace(T, K, E, R, dev)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(moedc_layout(topk_idx, T, K, E, R, cap, out.num_tokens_per_expert,
                        out.num_tokens_per_rank, out.is_token_in_rank, out.slot, workspace, wsb,
                        out.status), "moedc_layout")
    return out


def alloc_recv(E: int, cap: int, H: int, out_dtype: int, device):
    """recv [E,cap,H] (bf16, or e4m3 as torch.float8_e4m3fn), scales [E,cap,H/128]
    ([E,H/128,cap] with SCALES_COL_MAJOR, [E,cap] with SCALES_PER_TOKEN; fp32,
    e4m3 only) and src_idx [E,cap]."""
    if out_dtype & ~(SCALES_COL_MAJOR | SCALES_PER_TOKEN) == FP8_E4M3:
        recv = torch.empty((E, cap, H), dtype=torch.float8_e4m3fn, device=device)
        shape = ((E, cap) if out_dtype & SCALES_PER_TOKEN
                 else (E, H // 128, cap) if out_dtype & SCALES_COL_MAJOR else (E, cap, H // 128))
        scales = torch.empty(shape, dtype=torch.float32, device=device)
    else:
        recv = torch.empty((E, cap, H), dtype=torch.bfloat16, device=device)
        scales = None
    return recv, scales, torch.empty((E, cap), dtype=torch.int32, device=device)


def dispatch(x: torch.Tensor, topk_idx: torch.Tensor, lay: Layout, E: int, cap: int,
             out_dtype: int, out=None):
    """Returns (recv, scales or None, src_idx)."""
    _need(x, torch.bfloat16, "x")
    _need(topk_idx, torch.int32, "topk_idx")
    T, H = x.shape
    K = topk_idx.shape[1]
    recv, scales, src_idx = out if out is not None else alloc_recv(E, cap, H, out_dtype, x.device)
    _check(moedc_dispatch(x, T, H, topk_idx, lay.slot, lay.num_tokens_per_expert, K, E, cap,
                          out_dtype, recv, scales, src_idx, lay.status), "moedc_dispatch")
    return recv, scales, src_idx


def combine(expert_out: torch.Tensor, topk_idx: torch.Tensor, slot: torch.Tensor,
            topk_weights: torch.Tensor, status: torch.Tensor | None = None,
            out: torch.Tensor | None = None) -> torch.Tensor:
    _need(expert_out, torch.bfloat16, "expert_out")
    _need(topk_weights, torch.float32, "topk_weights")
    E, cap, H = expert_out.shape
    T, K = topk_idx.shape
    y = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16,
                                                device=expert_out.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=expert_out.device)
    _check(moedc_combine(expert_out, E, cap, H, topk_idx, slot, topk_weights, T, K, y, status),
           "moedc_combine")
    return y


def layout_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, E: int, R: int, cap: int,
                    out_dtype: int, workspace: torch.Tensor | None = None):
    """Returns (Layout, recv, scales or None, src_idx)."""
    _need(x, torch.bfloat16, "x")
    _need(topk_idx, torch.int32, "topk_idx")
    T, H = x.shape
    K = topk_idx.shape[1]
    dev = x.device
    lay = Layout(_dev_i32(E, dev), _dev_i32(R, dev),
                 torch.empty((T, R), dtype=torch.uint8, device=dev), _dev_i32((T, K), dev),
                 torch.zeros(1, dtype=torch.int32, device=dev))
    recv, scales, src_idx = alloc_recv(E, cap, H, out_dtype, dev)
    if workspace is None:
        workspace = layout_dispatch_workspace(T, K, E, R, dev)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(moedc_layout_dispatch(x, topk_idx, T, H, K, E, R, cap, out_dtype,
                                 lay.num_tokens_per_expert, lay.num_tokens_per_rank,
                                 lay.is_token_in_rank, lay.slot, recv, scales, src_idx, workspace,
                                 wsb, lay.status), "moedc_layout_dispatch")
    return lay, recv, scales, src_idx


def dequant_e4m3(recv: torch.Tensor, scales: torch.Tensor, num_tokens_per_expert: torch.Tensor,
                 out: torch.Tensor | None = None, scale_layout: int = 0) -> torch.Tensor:
    """bf16 [E, cap, H] view of an e4m3 receive buffer (filled rows only)."""
    E, cap, H = recv.shape
    if out is None:
        out = torch.zeros((E, cap, H), dtype=torch.bfloat16, device=recv.device)
    _check(moedc_dequant_e4m3(recv, scales, scale_layout, num_tokens_per_expert, E, cap, H, out),
           "moedc_dequant_e4m3")
    return out


def combine_e4m3(expert_out: torch.Tensor, expert_scales: torch.Tensor, topk_idx: torch.Tensor,
                 slot: torch.Tensor, topk_weights: torch.Tensor, scale_layout: int = 0,
                 status: torch.Tensor | None = None) -> torch.Tensor:
    """Combine from e4m3 expert outputs [E, cap, H] with fp32 scales in the
    given scale_layout (0, SCALES_COL_MAJOR or SCALES_PER_TOKEN)."""
    _need(topk_weights, torch.float32, "topk_weights")
    E, cap, H = expert_out.shape
    T, K = topk_idx.shape
    y = torch.empty((T, H), dtype=torch.bfloat16, device=expert_out.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=expert_out.device)
    _check(moedc_combine_e4m3(expert_out, expert_scales, scale_layout, E, cap, H, topk_idx, slot,
                              topk_weights, T, K, y, status), "moedc_combine_e4m3")
    return y


def rank_layout(lay: Layout, cap_rank: int) -> torch.Tensor:
    """rank_slot [T, R] from a Layout (raises on argument errors)."""
    T, R = lay.is_token_in_rank.shape
    rank_slot = torch.empty((T, R), dtype=torch.int32, device=lay.slot.device)
    _check(moedc_rank_layout(lay.is_token_in_rank, T, R, cap_rank, rank_slot, lay.status),
           "moedc_rank_layout")
    return rank_slot


def rank_dispatch(x: torch.Tensor, rank_slot: torch.Tensor, lay: Layout, cap_rank: int,
                  out_dtype: int):
    """Returns (recv_rank [R, cap_rank, H], scales_rank or None, rank_src_idx [R, cap_rank])."""
    _need(x, torch.bfloat16, "x")
    T, H = x.shape
    R = rank_slot.shape[1]
    recv, scales, src = alloc_recv(R, cap_rank, H, out_dtype, x.device)
    _check(moedc_rank_dispatch(x, T, H, rank_slot, lay.num_tokens_per_rank, R, cap_rank,
                               out_dtype, recv, scales, src), "moedc_rank_dispatch")
    return recv, scales, src


def rank_combine(rank_out: torch.Tensor, rank_slot: torch.Tensor) -> torch.Tensor:
    _need(rank_out, torch.bfloat16, "rank_out")
    R, cap_rank, H = rank_out.shape
    T = rank_slot.shape[0]
    y = torch.empty((T, H), dtype=torch.bfloat16, device=rank_out.device)
    _check(moedc_rank_combine(rank_out, R, cap_rank, H, rank_slot, T, y), "moedc_rank_combine")
    return y
