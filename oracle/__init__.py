"""CPU oracle for MoE layout / dispatch / combine (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module.  The library itself never does: its product path is
the CUDA library alone.

The arithmetic lives in plain C (moedc_oracle.c, compiled without fused
multiply-add or fast-math); this file builds it with gcc and wraps it with
ctypes over numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moedc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoedc_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
ERR_CAPACITY = 2
ERR_EXPERT_RANGE = 3

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc; returns the library path."""
    with _lock:
        if not force and os.path.exists(_LIB_PATH) and \
                os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I = ctypes.c_int
    I64 = ctypes.c_int64
    lib.oracle_layout.argtypes = [P, I, I, I, I, I, P, P, P, P]
    lib.oracle_layout.restype = I
    lib.oracle_dispatch.argtypes = [P, I, I, P, P, I, I, I, I, P, P, P]
    lib.oracle_dispatch.restype = I
    lib.oracle_combine.argtypes = [P, I, I, I, P, P, P, I, I, P]
    lib.oracle_combine.restype = I
    lib.oracle_e4m3_encode_n.argtypes = [P, P, I64]
    lib.oracle_e4m3_decode_n.argtypes = [P, P, I64]
    lib.oracle_f32_to_bf16_n.argtypes = [P, P, I64]
    lib.oracle_dequant_e4m3.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_dequant_e4m3_token.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_dispatch_token_scale.argtypes = [P, I, I, P, P, I, I, I, P, P, P]
    lib.oracle_rank_layout.argtypes = [P, I, I, I, P]
    lib.oracle_rank_layout.restype = I
    lib.oracle_rank_dispatch.argtypes = [P, I, I, P, I, I, I, P, P, P]
    lib.oracle_rank_combine.argtypes = [P, I, I, I, P, I, P]
    lib.oracle_combine_e4m3.argtypes = [P, P, I, I, I, I, P, P, P, I, I, P]
    lib.oracle_combine_e4m3.restype = I
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_n(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_decode(c: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float32)
    _load().oracle_e4m3_decode_n(_ptr(c), _ptr(out), c.size)
    return out


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_f32_to_bf16_n(_ptr(v), _ptr(out), v.size)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def layout(topk_idx: np.ndarray, E: int, R: int, cap: int) -> dict:
    """Returns counts, rank counts, token-in-rank mask, slot map and status."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    out = dict(
        num_tokens_per_expert=np.empty(E, np.int32),
        num_tokens_per_rank=np.empty(R, np.int32),
        is_token_in_rank=np.empty((T, R), np.uint8),
        slot=np.empty((T, K), np.int32),
    )
    out["status"] = _load().oracle_layout(
        _ptr(topk_idx), T, K, E, R, cap, _ptr(out["num_tokens_per_expert"]),
        _ptr(out["num_tokens_per_rank"]), _ptr(out["is_token_in_rank"]), _ptr(out["slot"]))
    return out


def dispatch(x: np.ndarray, topk_idx: np.ndarray, slot: np.ndarray, E: int, cap: int,
             fp8: bool, recv: np.ndarray | None = None) -> dict:
    """x: uint16 bf16 bits [T, H].  Returns recv ([E,cap,H] uint16 or uint8),
    scales ([E,cap,H/128] float32, fp8 only), src_idx and status.
    Rows no entry reaches keep their initial contents (zeros unless `recv`
    is given)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T, H = x.shape
    K = topk_idx.shape[1] if topk_idx.ndim == 2 else 0
    if recv is None:
        recv = np.zeros((E, cap, H), np.uint8 if fp8 else np.uint16)
    scales = np.zeros((E, cap, H // 128), np.float32) if fp8 else np.zeros(1, np.float32)
    src_idx = np.empty((E, cap), np.int32)
    status = _load().oracle_dispatch(_ptr(x), T, H, _ptr(topk_idx), _ptr(slot), K, E, cap,
                                     1 if fp8 else 0, _ptr(recv), _ptr(scales), _ptr(src_idx))
    return dict(recv=recv, scales=scales if fp8 else None, src_idx=src_idx, status=status)


def dispatch_token_scale(x: np.ndarray, topk_idx: np.ndarray, slot: np.ndarray, E: int,
                         cap: int, recv: np.ndarray | None = None) -> dict:
    """e4m3 dispatch with one scale per token row.  Returns recv (uint8
    [E,cap,H]), scales (float32 [E,cap]), src_idx and status; untouched rows
    keep their initial contents (zeros unless `recv` is given)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    T, H = x.shape
    K = topk_idx.shape[1] if topk_idx.ndim == 2 else 0
    if recv is None:
        recv = np.zeros((E, cap, H), np.uint8)
    scales = np.zeros((E, cap), np.float32)
    src_idx = np.empty((E, cap), np.int32)
    status = _load().oracle_dispatch_token_scale(_ptr(x), T, H, _ptr(topk_idx), _ptr(slot), K,
                                                 E, cap, _ptr(recv), _ptr(scales),
                                                 _ptr(src_idx))
    return dict(recv=recv, scales=scales, src_idx=src_idx, status=status)


def combine(expert_out: np.ndarray, topk_idx: np.ndarray, slot: np.ndarray,
            topk_weights: np.ndarray) -> dict:
    """expert_out: uint16 bf16 bits [E, cap, H].  Returns y (uint16 [T, H]) and status."""
    expert_out = np.ascontiguousarray(expert_out, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    E, cap, H = expert_out.shape
    T, K = topk_idx.shape
    y = np.empty((T, H), np.uint16)
    status = _load().oracle_combine(_ptr(expert_out), E, cap, H, _ptr(topk_idx), _ptr(slot),
                                    _ptr(topk_weights), T, K, _ptr(y))
    return dict(y=y, status=status)


def dequant_e4m3(recv: np.ndarray, scales: np.ndarray, num_tokens_per_expert: np.ndarray,
                 out: np.ndarray | None = None) -> np.ndarray:
    """recv uint8 [E, cap, H], scales float32 [E, cap, H/128] -> bf16 bits
    [E, cap, H]; rows past each expert's count keep `out`'s contents (zeros
    by default)."""
    recv = np.ascontiguousarray(recv, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    cnt = np.ascontiguousarray(num_tokens_per_expert, dtype=np.int32)
    E, cap, H = recv.shape
    if out is None:
        out = np.zeros((E, cap, H), np.uint16)
    _load().oracle_dequant_e4m3(_ptr(recv), _ptr(scales), _ptr(cnt), E, cap, H, _ptr(out))
    return out


def dequant_e4m3_token(recv: np.ndarray, scales: np.ndarray, num_tokens_per_expert: np.ndarray,
                       out: np.ndarray | None = None) -> np.ndarray:
    """As dequant_e4m3 with one scale per row: scales float32 [E, cap]."""
    recv = np.ascontiguousarray(recv, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    cnt = np.ascontiguousarray(num_tokens_per_expert, dtype=np.int32)
    E, cap, H = recv.shape
    if out is None:
        out = np.zeros((E, cap, H), np.uint16)
    _load().oracle_dequant_e4m3_token(_ptr(recv), _ptr(scales), _ptr(cnt), E, cap, H, _ptr(out))
    return out


def rank_layout(is_token_in_rank: np.ndarray, cap_rank: int) -> dict:
    """rank_slot [T, R] (position of token t in rank r's buffer, -1 if absent) and status."""
    inr = np.ascontiguousarray(is_token_in_rank, dtype=np.uint8)
    T, R = inr.shape
    slot = np.empty((T, R), np.int32)
    status = _load().oracle_rank_layout(_ptr(inr), T, R, cap_rank, _ptr(slot))
    return dict(rank_slot=slot, status=status)


def rank_dispatch(x: np.ndarray, rank_slot: np.ndarray, cap_rank: int, fp8: bool) -> dict:
    """recv_rank [R, cap_rank, H] (bf16 bits or e4m3 codes), scales_rank
    [R, cap_rank, H/128] (e4m3 only), rank_src_idx [R, cap_rank]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    rank_slot = np.ascontiguousarray(rank_slot, dtype=np.int32)
    T, H = x.shape
    R = rank_slot.shape[1]
    recv = np.zeros((R, cap_rank, H), np.uint8 if fp8 else np.uint16)
    scales = np.zeros((R, cap_rank, H // 128), np.float32) if fp8 else np.zeros(1, np.float32)
    src = np.empty((R, cap_rank), np.int32)
    _load().oracle_rank_dispatch(_ptr(x), T, H, _ptr(rank_slot), R, cap_rank, 1 if fp8 else 0,
                                 _ptr(recv), _ptr(scales), _ptr(src))
    return dict(recv_rank=recv, scales_rank=scales if fp8 else None, rank_src_idx=src)


def rank_combine(rank_out: np.ndarray, rank_slot: np.ndarray) -> np.ndarray:
    """rank_out bf16 bits [R, cap_rank, H] -> y bf16 bits [T, H]."""
    rank_out = np.ascontiguousarray(rank_out, dtype=np.uint16)
    rank_slot = np.ascontiguousarray(rank_slot, dtype=np.int32)
    R, cap_rank, H = rank_out.shape
    T = rank_slot.shape[0]
    y = np.empty((T, H), np.uint16)
    _load().oracle_rank_combine(_ptr(rank_out), R, cap_rank, H, _ptr(rank_slot), T, _ptr(y))
    return y


def combine_e4m3(expert_out: np.ndarray, expert_scales: np.ndarray, topk_idx: np.ndarray,
                 slot: np.ndarray, topk_weights: np.ndarray, scale_cols: bool = False,
                 per_token: bool = False) -> dict:
    """expert_out: e4m3 codes uint8 [E, cap, H]; expert_scales float32 [E, cap, H/128]
    (or [E, H/128, cap] with scale_cols, or [E, cap] with per_token).  Returns
    y (bf16 bits [T, H]) and status."""
    expert_out = np.ascontiguousarray(expert_out, dtype=np.uint8)
    expert_scales = np.ascontiguousarray(expert_scales, dtype=np.float32)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    slot = np.ascontiguousarray(slot, dtype=np.int32)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    E, cap, H = expert_out.shape
    T, K = topk_idx.shape
    y = np.empty((T, H), np.uint16)
    status = _load().oracle_combine_e4m3(_ptr(expert_out), _ptr(expert_scales),
                                         2 if per_token else 1 if scale_cols else 0, E, cap,
                                         H, _ptr(topk_idx),
                                         _ptr(slot), _ptr(topk_weights), T, K, _ptr(y))
    return dict(y=y, status=status)
