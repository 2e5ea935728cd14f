"""CPU oracle for MoE dispatch / combine — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports it, and it shares no code with the product.

The arithmetic lives in ``ep_oracle.c`` (plain sequential C, built with
``gcc -O2 -ffp-contract=off``); this module only builds it, loads it and moves
numpy arrays in and out.  BF16 tensors are carried as ``uint16`` bit patterns,
E4M3 tensors as ``uint8`` codes.

What each function computes follows the DeepEP pages:
``layout`` — the dispatch layout (per-expert/per-rank counts, slots) that
"如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南" (section 技术解析) says is
computed once and reused; ``dispatch``/``quant_token`` — low_latency_dispatch
with the optional FP8 cast (section 核心API示例 and 核心优势 of the same page);
``combine`` — low_latency_combine's top-k weighted reduce to BF16 (same sections);
``rank_layout`` / ``rank_runs`` — the rank-deduplicated transport of the normal
kernels (DeepTech announcement of DeepEP, 010bt.com) and its per-(source rank,
destination rank) runs, which a receive that occupies no SM copies whole
(section 技术解析, 通信-计算重叠技术, of the first page).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB = os.path.join(_HERE, "libep_oracle.so")

LAYOUT_PADDED = 0
LAYOUT_PACKED = 1


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -ffp-contract=off (no fast-math) of one C file into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(
        ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
         "-Wall", "-shared", "-fPIC", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into libep_oracle.so next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


_lib = None


def _load():
    if _lib is None:
        use_library(build())
    return _lib


def use_library(path: str | None):
    """Bind this module to the oracle library at ``path`` (None: unbind, so the
    next call loads the built ep_oracle.c again).  The tests use it to run the
    pins against deliberately broken copies of the oracle."""
    global _lib
    if path is None:
        _lib = None
        return None
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I32, I64 = ctypes.c_int, ctypes.c_int64
    lib.orc_layout.restype = None
    lib.orc_layout.argtypes = [I32, I32, I32, I32, I32, I32, P,
                               P, P, P, P, P, P, P, P, I64, P]
    lib.orc_rank_layout.restype = None
    lib.orc_rank_layout.argtypes = [I32, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, I64]
    lib.orc_rank_runs.restype = ctypes.c_int64
    lib.orc_rank_runs.argtypes = [I32, I32, I32, I32, P, P, P, P, P, P]
    lib.orc_quant_block.argtypes = [P, P, P]
    lib.orc_quant_token.argtypes = [P, I32, P, P]
    lib.orc_dispatch.argtypes = [I64, I32, I32, I32, P, P, P, P]
    lib.orc_combine.argtypes = [I64, I32, I32, P, P, P, P]
    lib.orc_dequant_rows.argtypes = [I64, I32, I32, P, P, P, P]
    for name in ("orc_f32_to_bf16_n", "orc_bf16_to_f32_n",
                 "orc_f32_to_e4m3_n", "orc_e4m3_to_f32_n"):
        getattr(lib, name).argtypes = [P, P, I64]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
    lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
    _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats

def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint16)
    _load().orc_f32_to_bf16_n(_p(x), _p(y), x.size)
    return y


def bf16_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty(b.shape, np.float32)
    _load().orc_bf16_to_f32_n(_p(b), _p(y), b.size)
    return y


def f32_to_e4m3(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, np.uint8)
    _load().orc_f32_to_e4m3_n(_p(x), _p(y), x.size)
    return y


def e4m3_to_f32(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    y = np.empty(c.shape, np.float32)
    _load().orc_e4m3_to_f32_n(_p(c), _p(y), c.size)
    return y


# ---------------------------------------------------------------- layout

def recv_rows(R: int, Tmax: int, E: int, K: int, layout: int) -> int:
    """Rows of the receive buffer: E fixed buffers of R*Tmax rows (padded) or
    the worst case R*Tmax*K rows (packed)."""
    return E * R * Tmax if layout == LAYOUT_PADDED else R * Tmax * K


def layout(topk_idx: np.ndarray, num_experts: int, max_tokens_per_rank: int,
           layout: int = LAYOUT_PADDED) -> dict:
    """Dispatch layout of topk_idx [R, T, K] (int64).  Returns a dict of numpy
    arrays: cnt_er [E, R], off_er [E, R], tokens_per_expert [E], base [E],
    tokens_per_rank [R], is_token_in_rank [N, R] (uint8), slot [N, K],
    src_info [rows] (-1 where nothing lands), plus n_bad (ids outside
    [-1, E)), n_overflow (padded entries past an expert's R*Tmax rows), rows."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, K = idx.shape
    E = int(num_experts)
    assert E % R == 0 and T <= max_tokens_per_rank
    N = R * T
    rows = recv_rows(R, max_tokens_per_rank, E, K, layout)
    out = dict(
        cnt_er=np.zeros((E, R), np.int32), off_er=np.zeros((E, R), np.int32),
        tokens_per_expert=np.zeros(E, np.int32), base=np.zeros(E, np.int64),
        tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((N, R), np.uint8),
        slot=np.zeros((N, K), np.int32), src_info=np.full(rows, -1, np.int32))
    errors = np.zeros(2, np.int64)
    _load().orc_layout(
        R, T, max_tokens_per_rank, K, E, layout, _p(idx),
        _p(out["cnt_er"]), _p(out["off_er"]), _p(out["tokens_per_expert"]),
        _p(out["base"]), _p(out["tokens_per_rank"]), _p(out["is_token_in_rank"]),
        _p(out["slot"]), _p(out["src_info"]), rows, _p(errors))
    out["n_bad"] = int(errors[0])
    out["n_overflow"] = int(errors[1])
    out["rows"] = rows
    return out


def rank_recv_rows(R: int, Tmax: int, K: int, layout: int) -> int:
    """Rows of a rank-deduplicated receive buffer: R buffers of R*Tmax rows
    (padded) or the worst case R*Tmax*min(K, R) rows (packed)."""
    return R * R * Tmax if layout == LAYOUT_PADDED else R * Tmax * min(K, R)


def rank_layout(topk_idx: np.ndarray, topk_weights: np.ndarray | None, num_experts: int,
                max_tokens_per_rank: int, layout: int = LAYOUT_PACKED) -> dict:
    """Rank-deduplicated layout of topk_idx [R, T, K]: rank_slot [N, K] (row of
    the entry that carries the token to its rank, else -1), tokens_per_rank
    [R], rbase [R], src_info [rows] (-1 where nothing lands), recv_topk_idx
    [rows, K] (local expert ids or -1), recv_topk_weights [rows, K], rows."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, K = idx.shape
    E = int(num_experts)
    N = R * T
    rows = rank_recv_rows(R, max_tokens_per_rank, K, layout)
    w = None if topk_weights is None else np.ascontiguousarray(topk_weights, dtype=np.float32).reshape(N, K)
    out = dict(rank_slot=np.zeros((N, K), np.int32), tokens_per_rank=np.zeros(R, np.int32),
               rbase=np.zeros(R, np.int64), src_info=np.full(rows, -1, np.int32),
               recv_topk_idx=np.full((rows, K), -1, np.int32),
               recv_topk_weights=np.zeros((rows, K), np.float32))
    _load().orc_rank_layout(R, T, max_tokens_per_rank, K, E, layout, _p(idx),
                            None if w is None else _p(w), _p(out["rank_slot"]),
                            _p(out["tokens_per_rank"]), _p(out["rbase"]), _p(out["src_info"]),
                            _p(out["recv_topk_idx"]), _p(out["recv_topk_weights"]), rows)
    out["rows"] = rows
    return out


def rank_runs(topk_idx: np.ndarray, num_experts: int, rbase: np.ndarray) -> dict:
    """Runs of the rank-deduplicated transport (topk_idx [R, T, K], rbase [R]
    from rank_layout): send_slot [N, K] (row of the carrying entry in the send
    buffer ordered by source rank, destination rank, token; else -1),
    run_cnt [R, R] (tokens source r carries to rank d), send_off [R, R],
    recv_off [R, R] (first send / receive row of each run), send_rows."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    R, T, K = idx.shape
    rb = np.ascontiguousarray(rbase, dtype=np.int64)
    assert rb.shape == (R,)
    out = dict(send_slot=np.zeros((R * T, K), np.int32), run_cnt=np.zeros((R, R), np.int32),
               send_off=np.zeros((R, R), np.int64), recv_off=np.zeros((R, R), np.int64))
    out["send_rows"] = int(_load().orc_rank_runs(R, T, K, int(num_experts), _p(idx), _p(rb), _p(out["send_slot"]),
                                                _p(out["run_cnt"]), _p(out["send_off"]), _p(out["recv_off"])))
    return out


# ---------------------------------------------------------------- dispatch

def quant_token(x_bits: np.ndarray):
    """FP8 cast of one or more token rows x_bits [..., H] (bf16 bits):
    returns (q uint8 [..., H], scales float32 [..., H/128])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    H = x.shape[-1]
    assert H % 128 == 0
    rows = x.reshape(-1, H)
    q = np.empty(rows.shape, np.uint8)
    s = np.empty((rows.shape[0], H // 128), np.float32)
    lib = _load()
    for i in range(rows.shape[0]):
        lib.orc_quant_token(_p(rows[i]), H, _p(q[i]), _p(s[i]))
    return q.reshape(x.shape), s.reshape(x.shape[:-1] + (H // 128,))


def dispatch(x_bits: np.ndarray, slot: np.ndarray, rows: int, use_fp8: bool,
             recv: np.ndarray | None = None, scales: np.ndarray | None = None):
    """Scatter x_bits [N, H] (bf16 bits) into receive rows.  BF16: returns
    recv uint16 [rows, H].  FP8: returns (recv uint8 [rows, H], scales float32
    [rows, H/128]).  Rows nobody writes keep the given buffer's contents
    (zeros when no buffer is given)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    N, H = x.shape
    sl = np.ascontiguousarray(slot, dtype=np.int32)
    K = sl.shape[1]
    if use_fp8:
        recv = np.zeros((rows, H), np.uint8) if recv is None else recv
        scales = np.zeros((rows, H // 128), np.float32) if scales is None else scales
        _load().orc_dispatch(N, K, H, 1, _p(x), _p(sl), _p(recv), _p(scales))
        return recv, scales
    recv = np.zeros((rows, H), np.uint16) if recv is None else recv
    _load().orc_dispatch(N, K, H, 0, _p(x), _p(sl), _p(recv), None)
    return recv


# ---------------------------------------------------------------- identity expert

def dequant_rows(q: np.ndarray, scales: np.ndarray, slot: np.ndarray,
                 y: np.ndarray | None = None) -> np.ndarray:
    """BF16 rows (uint16 bits) of the FP8 rows the entries of slot [N, K]
    received: y[row] = bf16(e4m3(q[row]) * scale).  Other rows keep y's
    contents (zeros when y is not given)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.float32)
    sl = np.ascontiguousarray(slot, dtype=np.int32)
    rows, H = q.shape
    y = np.zeros((rows, H), np.uint16) if y is None else y
    _load().orc_dequant_rows(sl.shape[0], sl.shape[1], H, _p(q), _p(sc), _p(sl), _p(y))
    return y


# ---------------------------------------------------------------- combine

def combine(y_bits: np.ndarray, slot: np.ndarray, weights: np.ndarray | None) -> np.ndarray:
    """Weighted top-k reduce: y_bits [rows, H] (bf16 bits), slot [N, K],
    weights float32 [N, K] or None (all ones).  Returns uint16 [N, H]."""
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    sl = np.ascontiguousarray(slot, dtype=np.int32)
    N, K = sl.shape
    H = y.shape[1]
    assert sl.max(initial=-1) < y.shape[0]
    out = np.empty((N, H), np.uint16)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    _load().orc_combine(N, K, H, _p(y), _p(sl), None if w is None else _p(w), _p(out))
    return out
