"""Thin Python binding of libep.so: the C ABI of include/ep.h, one Python
function per C entry point with the same name, marshalling torch tensors to
device pointers.  Every step of the computation runs in libep.so's kernels;
this module only checks shapes / dtypes and passes pointers.

The library must have been built (``python -m combine_get_dispatch_02_gb300.build``
or ``__graft_entry__.build()``); loading fails loudly otherwise.  There is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libep.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_OOM = 3
EP_ERR_CUDA = 4
EP_ERR_BAD_EXPERT = 5
EP_ERR_CAPACITY = 6
EP_ERR_NO_LAYOUT = 7
EP_ERR_TIMEOUT = 8
EP_ERR_TIMEOUT_IN_FLIGHT = 9

EP_LAYOUT_PADDED = 0
EP_LAYOUT_PACKED = 1

EP_WIRE_DEVICE = 0
EP_WIRE_HOST = 1

# Every entry point include/ep.h declares (checked against the header and the
# library by the tests).
ENTRY_POINTS = (
    "ep_status_str", "ep_config_check", "ep_recv_rows", "ep_recv_bytes",
    "ep_create", "ep_destroy", "ep_handle_create", "ep_handle_destroy",
    "ep_handle_get_info", "ep_get_dispatch_layout", "ep_dispatch", "ep_combine",
    "ep_get_device_status", "ep_dispatch_noalloc", "ep_get_rank_layout", "ep_rank_recv_rows",
    "ep_dispatch_range", "ep_combine_range", "ep_expert_identity", "ep_round_trip",
    "ep_round_trip_auto_chunk", "ep_dispatch_send", "ep_dispatch_recv", "ep_combine_send", "ep_combine_recv",
    "ep_get_tuning", "ep_set_tuning", "ep_autotune", "ep_get_autotune_log", "ep_set_test_hooks",
    "ep_rank_send_rows", "ep_rank_dispatch_send", "ep_rank_dispatch_recv", "ep_rank_combine_send",
    "ep_rank_combine_recv", "ep_rank_runs",
)

TUNE_KNOBS = {0: "dispatch", 1: "combine_chunks", 2: "round_trip_chunk",
              3: "layout_form"}  # dispatch: 100 * kernel + CTAs/SM

EP_CHUNK_AUTO = -1


class EPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} (status {status})")


class ep_config(ctypes.Structure):
    _fields_ = [("num_ranks", ctypes.c_int32), ("max_tokens_per_rank", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("max_sms", ctypes.c_int32)]


class ep_tuning(ctypes.Structure):
    _fields_ = [("dispatch_ctas_per_sm", ctypes.c_int32), ("combine_chunks", ctypes.c_int32),
                ("round_trip_chunk", ctypes.c_int32), ("dispatch_kernel", ctypes.c_int32),
                ("layout_form", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


class ep_tune_record(ctypes.Structure):
    _fields_ = [("knob", ctypes.c_int32), ("value", ctypes.c_int32), ("median_us", ctypes.c_float)]


class ep_test_hooks(ctypes.Structure):
    _fields_ = [("move_withhold_item", ctypes.c_int64), ("move_wait_ns", ctypes.c_int64)]


class ep_handle_info(ctypes.Structure):
    _fields_ = [("tokens_per_rank", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("slot", ctypes.c_void_p),
                ("src_info", ctypes.c_void_p), ("cnt_er", ctypes.c_void_p),
                ("off_er", ctypes.c_void_p), ("base", ctypes.c_void_p),
                ("tokens_per_expert", ctypes.c_void_p), ("has_rank_ranges", ctypes.c_int32),
                ("rank_mode", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libep.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -m combine_get_dispatch_02_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        CFG = ctypes.POINTER(ep_config)
        sig = {
            "ep_status_str": (ctypes.c_char_p, [I32]),
            "ep_config_check": (I32, [CFG]),
            "ep_recv_rows": (I32, [CFG, ctypes.POINTER(I64)]),
            "ep_recv_bytes": (I32, [CFG, I32, ctypes.POINTER(ctypes.c_uint64),
                                    ctypes.POINTER(ctypes.c_uint64)]),
            "ep_create": (I32, [CFG, ctypes.POINTER(P)]),
            "ep_destroy": (I32, [P]),
            "ep_handle_create": (I32, [P, ctypes.POINTER(P)]),
            "ep_handle_destroy": (I32, [P]),
            "ep_handle_get_info": (I32, [P, ctypes.POINTER(ep_handle_info)]),
            "ep_get_dispatch_layout": (I32, [P, P, I32, P, P, P, P, P]),
            "ep_dispatch": (I32, [P, P, P, I32, I32, P, P, P, P, P]),
            "ep_combine": (I32, [P, P, P, P, P, P]),
            "ep_get_device_status": (I32, [P, P]),
            "ep_dispatch_noalloc": (I32, [CFG, P, P, I32, I32, P, P, P, P]),
            "ep_get_rank_layout": (I32, [P, P, P, I32, P, P, P, P, P]),
            "ep_rank_recv_rows": (I32, [CFG, ctypes.POINTER(I64)]),
            "ep_dispatch_range": (I32, [P, P, I32, P, I64, I64, P, P, P]),
            "ep_combine_range": (I32, [P, P, P, P, I64, I64, P, P]),
            "ep_expert_identity": (I32, [P, P, I32, P, P, P, I64, I64, P]),
            "ep_round_trip": (I32, [P, P, P, I32, P, I32, P, P, P, P, P, I32, P]),
            "ep_round_trip_auto_chunk": (I32, [P, I32, I32, ctypes.POINTER(I32)]),
            "ep_dispatch_send": (I32, [P, P, P, I32, I32, P, P, P, P]),
            "ep_dispatch_recv": (I32, [P, P, I32, P, P, P, P, P, I32, P]),
            "ep_combine_send": (I32, [P, P, P, P, I32, P]),
            "ep_combine_recv": (I32, [P, P, P, P, P, P]),
            "ep_get_tuning": (I32, [P, ctypes.POINTER(ep_tuning)]),
            "ep_set_tuning": (I32, [P, ctypes.POINTER(ep_tuning)]),
            "ep_autotune": (I32, [P, P, P, I32, P, I32, P, P, P, P, I32, ctypes.POINTER(ep_tuning), P]),
            "ep_get_autotune_log": (I32, [P, ctypes.POINTER(ep_tune_record), I32, ctypes.POINTER(I32)]),
            "ep_set_test_hooks": (I32, [P, ctypes.POINTER(ep_test_hooks)]),
            "ep_rank_send_rows": (I32, [CFG, ctypes.POINTER(I64)]),
            "ep_rank_dispatch_send": (I32, [P, P, P, P, I32, I32, P, P, P, P, P, P]),
            "ep_rank_dispatch_recv": (I32, [P, P, I32, P, P, P, P, P, I32, P, P]),
            "ep_rank_combine_send": (I32, [P, P, P, P, I32, P, P]),
            "ep_rank_combine_recv": (I32, [P, P, P, P, P]),
            "ep_rank_runs": (I32, [P, ctypes.POINTER(I32), ctypes.POINTER(I64), ctypes.POINTER(I64)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().ep_status_str(status).decode()


def _check(status: int, where: str) -> None:
    if status != EP_OK:
        raise EPError(status, where)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_config(num_ranks, max_tokens_per_rank, hidden, num_experts, topk,
                layout=EP_LAYOUT_PADDED, max_sms=0) -> ep_config:
    return ep_config(num_ranks, max_tokens_per_rank, hidden, num_experts, topk, layout, max_sms)


# ------------------------------------------------------------- entry points

def ep_config_check(cfg: ep_config) -> int:
    return lib().ep_config_check(ctypes.byref(cfg))


def ep_recv_rows(cfg: ep_config) -> int:
    rows = ctypes.c_int64()
    _check(lib().ep_recv_rows(ctypes.byref(cfg), ctypes.byref(rows)), "ep_recv_rows")
    return rows.value


def ep_recv_bytes(cfg: ep_config, use_fp8: bool) -> tuple[int, int]:
    pb, sb = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().ep_recv_bytes(ctypes.byref(cfg), int(use_fp8), ctypes.byref(pb), ctypes.byref(sb)),
           "ep_recv_bytes")
    return pb.value, sb.value


def ep_create(cfg: ep_config) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    _check(lib().ep_create(ctypes.byref(cfg), ctypes.byref(ctx)), "ep_create")
    return ctx


def ep_destroy(ctx) -> None:
    _check(lib().ep_destroy(ctx), "ep_destroy")


def ep_handle_create(ctx) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().ep_handle_create(ctx, ctypes.byref(h)), "ep_handle_create")
    return h


def ep_handle_destroy(h) -> None:
    _check(lib().ep_handle_destroy(h), "ep_handle_destroy")


def ep_handle_get_info(h) -> ep_handle_info:
    info = ep_handle_info()
    _check(lib().ep_handle_get_info(h, ctypes.byref(info)), "ep_handle_get_info")
    return info


def ep_get_dispatch_layout(ctx, topk_idx: torch.Tensor | None, tokens_per_rank: int,
                           num_tokens_per_rank: torch.Tensor | None,
                           num_tokens_per_expert: torch.Tensor | None,
                           is_token_in_rank: torch.Tensor | None, handle, stream=None) -> None:
    _check(lib().ep_get_dispatch_layout(
        ctx, _ptr(topk_idx, torch.int64, "topk_idx"), int(tokens_per_rank),
        _ptr(num_tokens_per_rank, torch.int32, "num_tokens_per_rank"),
        _ptr(num_tokens_per_expert, torch.int32, "num_tokens_per_expert"),
        _ptr(is_token_in_rank, None, "is_token_in_rank"), handle, _stream(stream)),
        "ep_get_dispatch_layout")


def ep_rank_recv_rows(cfg: ep_config) -> int:
    rows = ctypes.c_int64()
    _check(lib().ep_rank_recv_rows(ctypes.byref(cfg), ctypes.byref(rows)), "ep_rank_recv_rows")
    return rows.value


def ep_get_rank_layout(ctx, topk_idx: torch.Tensor | None, topk_weights: torch.Tensor | None,
                       tokens_per_rank: int, num_tokens_per_rank: torch.Tensor | None,
                       recv_topk_idx: torch.Tensor | None, recv_topk_weights: torch.Tensor | None,
                       handle, stream=None) -> None:
    _check(lib().ep_get_rank_layout(
        ctx, _ptr(topk_idx, torch.int64, "topk_idx"), _ptr(topk_weights, torch.float32, "topk_weights"),
        int(tokens_per_rank), _ptr(num_tokens_per_rank, torch.int32, "num_tokens_per_rank"),
        _ptr(recv_topk_idx, torch.int32, "recv_topk_idx"),
        _ptr(recv_topk_weights, torch.float32, "recv_topk_weights"), handle, _stream(stream)),
        "ep_get_rank_layout")


def ep_dispatch(ctx, x: torch.Tensor, topk_idx: torch.Tensor | None, tokens_per_rank: int,
                use_fp8: bool, handle, recv_x: torch.Tensor, recv_scales: torch.Tensor | None,
                recv_count: torch.Tensor | None, stream=None) -> None:
    _check(lib().ep_dispatch(
        ctx, _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"),
        int(tokens_per_rank), int(bool(use_fp8)), handle, _ptr(recv_x, None, "recv_x"),
        _ptr(recv_scales, torch.float32, "recv_scales"),
        _ptr(recv_count, torch.int32, "recv_count"), _stream(stream)), "ep_dispatch")


def ep_combine(ctx, y: torch.Tensor, topk_weights: torch.Tensor | None, handle,
               out: torch.Tensor, stream=None) -> None:
    _check(lib().ep_combine(
        ctx, _ptr(y, torch.bfloat16, "y"), _ptr(topk_weights, torch.float32, "topk_weights"),
        handle, _ptr(out, torch.bfloat16, "out"), _stream(stream)), "ep_combine")


def ep_dispatch_range(ctx, x: torch.Tensor, use_fp8: bool, handle, token_begin: int, token_end: int,
                      recv_x: torch.Tensor, recv_scales: torch.Tensor | None, stream=None) -> None:
    _check(lib().ep_dispatch_range(
        ctx, _ptr(x, torch.bfloat16, "x"), int(bool(use_fp8)), handle, int(token_begin), int(token_end),
        _ptr(recv_x, None, "recv_x"), _ptr(recv_scales, torch.float32, "recv_scales"),
        _stream(stream)), "ep_dispatch_range")


def ep_combine_range(ctx, y: torch.Tensor, topk_weights: torch.Tensor | None, handle,
                     token_begin: int, token_end: int, out: torch.Tensor, stream=None) -> None:
    _check(lib().ep_combine_range(
        ctx, _ptr(y, torch.bfloat16, "y"), _ptr(topk_weights, torch.float32, "topk_weights"),
        handle, int(token_begin), int(token_end), _ptr(out, torch.bfloat16, "out"),
        _stream(stream)), "ep_combine_range")


def ep_expert_identity(ctx, handle, use_fp8: bool, recv_x: torch.Tensor, recv_scales: torch.Tensor | None,
                       y: torch.Tensor, token_begin: int, token_end: int, stream=None) -> None:
    _check(lib().ep_expert_identity(
        ctx, handle, int(bool(use_fp8)), _ptr(recv_x, None, "recv_x"),
        _ptr(recv_scales, torch.float32, "recv_scales"), _ptr(y, torch.bfloat16, "y"),
        int(token_begin), int(token_end), _stream(stream)), "ep_expert_identity")


def ep_round_trip(ctx, x: torch.Tensor, topk_idx: torch.Tensor | None, tokens_per_rank: int,
                  topk_weights: torch.Tensor | None, use_fp8: bool, handle, recv_x: torch.Tensor,
                  recv_scales: torch.Tensor | None, y: torch.Tensor, out: torch.Tensor,
                  chunk_tokens: int = 0, stream=None) -> None:
    _check(lib().ep_round_trip(
        ctx, _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"), int(tokens_per_rank),
        _ptr(topk_weights, torch.float32, "topk_weights"), int(bool(use_fp8)), handle,
        _ptr(recv_x, None, "recv_x"), _ptr(recv_scales, torch.float32, "recv_scales"),
        _ptr(y, torch.bfloat16, "y"), _ptr(out, torch.bfloat16, "out"), int(chunk_tokens),
        _stream(stream)), "ep_round_trip")


def ep_round_trip_auto_chunk(ctx, use_fp8: bool, rank_layout: bool = False) -> int:
    n = ctypes.c_int32(0)
    _check(lib().ep_round_trip_auto_chunk(ctx, int(bool(use_fp8)), int(bool(rank_layout)), ctypes.byref(n)),
           "ep_round_trip_auto_chunk")
    return n.value


def ep_dispatch_send(ctx, x: torch.Tensor, topk_idx: torch.Tensor | None, tokens_per_rank: int, use_fp8: bool,
                     handle, send_x: torch.Tensor, send_scales: torch.Tensor | None, stream=None) -> None:
    _check(lib().ep_dispatch_send(
        ctx, _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"), int(tokens_per_rank),
        int(bool(use_fp8)), handle, _ptr(send_x, None, "send_x"), _ptr(send_scales, torch.float32, "send_scales"),
        _stream(stream)), "ep_dispatch_send")


def ep_dispatch_recv(ctx, handle, use_fp8: bool, send_x: torch.Tensor, send_scales: torch.Tensor | None,
                     recv_x: torch.Tensor, recv_scales: torch.Tensor | None, recv_count: torch.Tensor | None,
                     num_sms: int = 0, stream=None) -> None:
    _check(lib().ep_dispatch_recv(
        ctx, handle, int(bool(use_fp8)), _ptr(send_x, None, "send_x"),
        _ptr(send_scales, torch.float32, "send_scales"), _ptr(recv_x, None, "recv_x"),
        _ptr(recv_scales, torch.float32, "recv_scales"), _ptr(recv_count, torch.int32, "recv_count"),
        int(num_sms), _stream(stream)), "ep_dispatch_recv")


def ep_combine_send(ctx, handle, y: torch.Tensor, send_y: torch.Tensor, num_sms: int = 0, stream=None) -> None:
    _check(lib().ep_combine_send(ctx, handle, _ptr(y, torch.bfloat16, "y"), _ptr(send_y, torch.bfloat16, "send_y"),
                                 int(num_sms), _stream(stream)), "ep_combine_send")


def ep_combine_recv(ctx, handle, send_y: torch.Tensor, topk_weights: torch.Tensor | None, out: torch.Tensor,
                    stream=None) -> None:
    _check(lib().ep_combine_recv(ctx, handle, _ptr(send_y, torch.bfloat16, "send_y"),
                                 _ptr(topk_weights, torch.float32, "topk_weights"),
                                 _ptr(out, torch.bfloat16, "out"), _stream(stream)), "ep_combine_recv")


def ep_get_tuning(ctx) -> ep_tuning:
    t = ep_tuning()
    _check(lib().ep_get_tuning(ctx, ctypes.byref(t)), "ep_get_tuning")
    return t


def ep_set_tuning(ctx, tuning: ep_tuning) -> None:
    _check(lib().ep_set_tuning(ctx, ctypes.byref(tuning)), "ep_set_tuning")


def ep_autotune(ctx, x: torch.Tensor, topk_idx: torch.Tensor, tokens_per_rank: int,
                topk_weights: torch.Tensor | None, use_fp8: bool, recv_x: torch.Tensor,
                recv_scales: torch.Tensor | None, y: torch.Tensor, out: torch.Tensor, reps: int = 20,
                stream=None) -> ep_tuning:
    t = ep_tuning()
    _check(lib().ep_autotune(
        ctx, _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"), int(tokens_per_rank),
        _ptr(topk_weights, torch.float32, "topk_weights"), int(bool(use_fp8)), _ptr(recv_x, None, "recv_x"),
        _ptr(recv_scales, torch.float32, "recv_scales"), _ptr(y, torch.bfloat16, "y"),
        _ptr(out, torch.bfloat16, "out"), int(reps), ctypes.byref(t), _stream(stream)), "ep_autotune")
    return t


def ep_get_autotune_log(ctx) -> list[tuple[str, int, float]]:
    """(knob, value, median µs) of each candidate the last ep_autotune timed."""
    recs = (ep_tune_record * 24)()
    n = ctypes.c_int32(0)
    _check(lib().ep_get_autotune_log(ctx, recs, 24, ctypes.byref(n)), "ep_get_autotune_log")
    return [(TUNE_KNOBS.get(r.knob, str(r.knob)), r.value, r.median_us) for r in recs[:min(n.value, 24)]]


def ep_get_device_status(ctx, stream=None) -> int:
    return lib().ep_get_device_status(ctx, _stream(stream))


def ep_dispatch_noalloc(cfg: ep_config, x: torch.Tensor, topk_idx: torch.Tensor, tokens_per_rank: int,
                        use_fp8: bool, recv_x: torch.Tensor, recv_scales: torch.Tensor | None,
                        recv_count: torch.Tensor | None, stream=None) -> None:
    """Dispatch without any device allocation (intermediate state in the
    library's static device array); see include/ep.h for limits."""
    _check(lib().ep_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"),
        int(tokens_per_rank), int(bool(use_fp8)), _ptr(recv_x, None, "recv_x"),
        _ptr(recv_scales, torch.float32, "recv_scales"), _ptr(recv_count, torch.int32, "recv_count"),
        _stream(stream)), "ep_dispatch_noalloc")


def ep_set_test_hooks(ctx, move_withhold_item: int = -1, move_wait_ns: int = 0) -> None:
    """Test-only switches (see include/ep.h): the copy kernels' item whose
    load is never issued, and the bound of their waits."""
    h = ep_test_hooks(int(move_withhold_item), int(move_wait_ns))
    _check(lib().ep_set_test_hooks(ctx, ctypes.byref(h)), "ep_set_test_hooks")


def ep_rank_send_rows(cfg: ep_config) -> int:
    rows = ctypes.c_int64()
    _check(lib().ep_rank_send_rows(ctypes.byref(cfg), ctypes.byref(rows)), "ep_rank_send_rows")
    return rows.value


def _host_ptr(t: torch.Tensor | None, name: str = "h_stage"):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor")
    return ctypes.c_void_p(t.data_ptr())


def ep_rank_dispatch_send(ctx, x: torch.Tensor, topk_idx: torch.Tensor | None, topk_weights: torch.Tensor | None,
                          tokens_per_rank: int, use_fp8: bool, recv_topk_idx: torch.Tensor | None,
                          recv_topk_weights: torch.Tensor | None, handle, send_x: torch.Tensor,
                          send_scales: torch.Tensor | None, stream=None) -> None:
    _check(lib().ep_rank_dispatch_send(
        ctx, _ptr(x, torch.bfloat16, "x"), _ptr(topk_idx, torch.int64, "topk_idx"),
        _ptr(topk_weights, torch.float32, "topk_weights"), int(tokens_per_rank), int(bool(use_fp8)),
        _ptr(recv_topk_idx, torch.int32, "recv_topk_idx"), _ptr(recv_topk_weights, torch.float32, "recv_topk_weights"),
        handle, _ptr(send_x, None, "send_x"), _ptr(send_scales, torch.float32, "send_scales"), _stream(stream)),
        "ep_rank_dispatch_send")


def ep_rank_dispatch_recv(ctx, handle, use_fp8: bool, send_x: torch.Tensor, send_scales: torch.Tensor | None,
                          recv_x: torch.Tensor, recv_scales: torch.Tensor | None, recv_count: torch.Tensor | None,
                          wire: int = EP_WIRE_DEVICE, stage: torch.Tensor | None = None, stream=None) -> None:
    _check(lib().ep_rank_dispatch_recv(
        ctx, handle, int(bool(use_fp8)), _ptr(send_x, None, "send_x"), _ptr(send_scales, torch.float32, "send_scales"),
        _ptr(recv_x, None, "recv_x"), _ptr(recv_scales, torch.float32, "recv_scales"),
        _ptr(recv_count, torch.int32, "recv_count"), int(wire), _host_ptr(stage), _stream(stream)),
        "ep_rank_dispatch_recv")


def ep_rank_combine_send(ctx, handle, y: torch.Tensor, send_y: torch.Tensor, wire: int = EP_WIRE_DEVICE,
                         stage: torch.Tensor | None = None, stream=None) -> None:
    _check(lib().ep_rank_combine_send(ctx, handle, _ptr(y, torch.bfloat16, "y"),
                                      _ptr(send_y, torch.bfloat16, "send_y"), int(wire), _host_ptr(stage),
                                      _stream(stream)), "ep_rank_combine_send")


def ep_rank_combine_recv(ctx, handle, send_y: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _check(lib().ep_rank_combine_recv(ctx, handle, _ptr(send_y, torch.bfloat16, "send_y"),
                                      _ptr(out, torch.bfloat16, "out"), _stream(stream)), "ep_rank_combine_recv")


def ep_rank_runs(handle, num_ranks: int):
    """(run_cnt, send_off, recv_off), each an R x R list of lists indexed [r][d]."""
    n = num_ranks * num_ranks
    cnt, so, ro = (ctypes.c_int32 * n)(), (ctypes.c_int64 * n)(), (ctypes.c_int64 * n)()
    _check(lib().ep_rank_runs(handle, cnt, so, ro), "ep_rank_runs")
    mat = lambda a: [list(a[r * num_ranks:(r + 1) * num_ranks]) for r in range(num_ranks)]
    return mat(cnt), mat(so), mat(ro)
