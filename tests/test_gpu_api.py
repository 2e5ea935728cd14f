"""GPU checks of the C ABI's behaviour around the kernels: host-side errors
with a live context, CUDA-graph capture, repeatability, SM caps."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import bf16_to_bits, bits_to_bf16, make_buffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


def _inputs(w):
    d = wl.generate(w)
    return (bits_to_bf16(d["x_bits"]), torch.from_numpy(d["topk_idx"]).cuda(),
            torch.from_numpy(d["topk_weights"].reshape(w.num_tokens, w.topk)).cuda(), d)


def test_host_errors_with_a_live_context():
    w = wl.TINY
    buf = make_buffer(w)
    other = make_buffer(w)
    x, idx, wts, _ = _inputs(w)
    recv, _ = buf.alloc_recv(False)
    L = ep.lib()
    P = ctypes.c_void_p
    h = buf.new_handle()
    h_other = other.new_handle()
    st = P(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t, off=0: P(t.data_ptr() + off)
    T = w.tokens_per_rank
    # combine before any layout
    assert L.ep_combine(buf.ctx, ptr(recv), ptr(wts), h.raw, ptr(x), st) == ep.EP_ERR_NO_LAYOUT
    # reuse without a layout
    assert L.ep_dispatch(buf.ctx, ptr(x), None, T, 0, h.raw, ptr(recv), None, None, st) == ep.EP_ERR_NO_LAYOUT
    # a handle of another context
    assert L.ep_dispatch(buf.ctx, ptr(x), ptr(idx), T, 0, h_other.raw, ptr(recv), None, None, st) == \
        ep.EP_ERR_INVALID_ARG
    # misaligned rows, bad T, FP8 without scales
    assert L.ep_dispatch(buf.ctx, ptr(x, 2), ptr(idx), T, 0, h.raw, ptr(recv), None, None, st) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(buf.ctx, ptr(x), ptr(idx), w.max_tokens_per_rank + 1, 0, h.raw, ptr(recv), None, None,
                         st) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(buf.ctx, ptr(x), ptr(idx), T, 1, h.raw, ptr(recv), None, None, st) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(buf.ctx, ptr(x), ptr(idx), T, 2, h.raw, ptr(recv), None, None, st) == ep.EP_ERR_INVALID_ARG
    # nothing was enqueued by the rejected calls; a valid call still works
    torch.cuda.synchronize()
    assert L.ep_dispatch(buf.ctx, ptr(x), ptr(idx), T, 0, h.raw, ptr(recv), None, None, st) == ep.EP_OK
    assert buf.device_status() == ep.EP_OK
    # T = Tmax with a layout for a different T: reuse is refused
    assert L.ep_dispatch(buf.ctx, ptr(x), None, T - 1, 0, h.raw, ptr(recv), None, None, st) == ep.EP_ERR_NO_LAYOUT


def test_fp8_hidden_not_multiple_of_128_is_unsupported():
    w = wl.TINY.with_(hidden=200)
    buf = make_buffer(w)
    x, idx, _, _ = _inputs(w)
    recv = torch.empty(buf.rows, w.hidden, dtype=torch.uint8, device="cuda")
    sc = torch.empty(buf.rows, 2, dtype=torch.float32, device="cuda")
    h = buf.new_handle()
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch(buf.ctx, x, idx, w.tokens_per_rank, True, h.raw, recv, sc, None)
    assert e.value.status == ep.EP_ERR_UNSUPPORTED


@pytest.mark.parametrize("kernel", [0, 3])  # the rule's (row) kernel, the token kernel
def test_cuda_graph_replay_matches_eager(kernel):
    w = wl.LL
    buf = make_buffer(w)
    ep.ep_set_tuning(buf.ctx, ep.ep_tuning(0, 0, 0, kernel))
    x, idx, wts, _ = _inputs(w)
    h = buf.new_handle()
    recv, sc = buf.alloc_recv(True)
    cnt = torch.empty(w.num_experts, dtype=torch.int32, device="cuda")
    y = torch.randn(buf.rows // 64, w.hidden, device="cuda").to(torch.bfloat16).repeat(64, 1)
    out_eager = torch.empty(w.num_tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    out_graph = torch.empty_like(out_eager)

    def step(out, s):
        ep.ep_dispatch(buf.ctx, x, idx, w.tokens_per_rank, True, h.raw, recv, sc, cnt, s)
        ep.ep_combine(buf.ctx, y, wts, h.raw, out, s)

    recv.view(torch.uint8).zero_()
    step(out_eager, torch.cuda.current_stream())
    torch.cuda.synchronize()
    q_eager = recv.view(torch.uint8)[:: 61].clone()
    recv.view(torch.uint8).zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(out_graph, s)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(out_graph, s)
    out_graph.zero_()
    recv.view(torch.uint8).zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert buf.device_status() == ep.EP_OK
    assert torch.equal(out_graph.view(torch.int16), out_eager.view(torch.int16))
    assert torch.equal(recv.view(torch.uint8)[:: 61], q_eager)


def test_dispatch_and_combine_repeatable():
    w = wl.SKEW
    buf = make_buffer(w)
    x, idx, wts, _ = _inputs(w)
    ref = None
    for _ in range(5):
        (recv, sc), cnt, h = buf.low_latency_dispatch(x, idx, w.max_tokens_per_rank, w.num_experts, use_fp8=True)
        rows = h.tensors()["slot"].view(-1).long()
        y = torch.zeros(buf.rows, w.hidden, dtype=torch.bfloat16, device="cuda")
        y[rows] = (recv.view(torch.uint8)[rows].view(torch.float8_e4m3fn).float()
                   .view(len(rows), -1, 128) * sc[rows].unsqueeze(-1)).view(len(rows), -1).to(torch.bfloat16)
        out = buf.low_latency_combine(y, idx, wts, h, w.num_experts)
        cur = (recv.view(torch.uint8)[rows].clone(), sc[rows].clone(), out.clone())
        if ref is None:
            ref = cur
        assert all(torch.equal(a, b) for a, b in zip(cur, ref))


def test_combine_max_sms_same_result():
    w = wl.LL
    x, idx, wts, _ = _inputs(w)
    outs = []
    y = None
    for ms in (0, 5):
        buf = make_buffer(w, max_sms=ms)
        _, _, _, h = buf.get_dispatch_layout(idx)
        if y is None:
            y = torch.randn(4096, w.hidden, device="cuda").to(torch.bfloat16).repeat(buf.rows // 4096, 1)
        outs.append(buf.low_latency_combine(y, idx, wts, h, w.num_experts).clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
