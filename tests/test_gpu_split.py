"""GPU parity of the split (send / receive-hook) dispatch and combine against
the oracle and against the fused calls, bit for bit: the send buffer holds
the oracle's per-token cast, the receive buffers and counts equal
ep_dispatch's, the combine staging holds each entry's expert-output row and
the hook's reduce equals ep_combine.  The receive hooks run on a few SMs as
well as on all of them."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import ORACLE_LAYOUT, bf16_to_bits, bits_to_bf16, e4m3_to_bits, make_buffer, place_rows, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _inputs(w, masks=0.0):
    d = wl.generate(w)
    idx = d["topk_idx"]
    if masks:
        idx = wl.inject_masks(idx, masks, 13)
    return idx, d["x_bits"].reshape(w.num_tokens, w.hidden), \
        d["topk_weights"].reshape(w.num_tokens, w.topk).astype(np.float32)


CASES = {
    "tiny_fp8": (wl.TINY.with_(use_fp8=True, x_scale="loguniform"), 0.0),
    "tiny_bf16": (wl.TINY, 0.0),
    "ll_fp8": (wl.LL, 0.0),
    "skew_fp8_masked": (wl.SKEW.with_(tokens_per_rank=300), 0.1),
    "packed_ragged_fp8": (wl.LL.with_(tokens_per_rank=77, layout=wl.PACKED), 0.05),
    "h16384_bf16": (wl.TINY.with_(hidden=16384, tokens_per_rank=8, max_tokens_per_rank=8), 0.0),
}


@pytest.mark.parametrize("num_sms", [0, 4])
@pytest.mark.parametrize("name", list(CASES))
def test_split_dispatch_and_combine_parity(name, num_sms):
    w, masks = CASES[name]
    idx, x_bits, wts = _inputs(w, masks)
    N, K, H = w.num_tokens, w.topk, w.hidden
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    o = oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    slot = o["slot"]
    rows = valid_rows(slot)
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    g_of = np.nonzero(slot.reshape(-1) >= 0)[0] // K

    # send: the layout, then each token cast once into the send buffer
    h = buf.new_handle()
    if w.use_fp8:
        send_x = torch.empty(N, H, dtype=torch.float8_e4m3fn, device="cuda")
        send_sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
    else:
        send_x, send_sc = torch.empty(N, H, dtype=torch.bfloat16, device="cuda"), None
    ep.ep_dispatch_send(buf.ctx, x, idx_d, w.tokens_per_rank, w.use_fp8, h.raw, send_x, send_sc)
    recv, scales = buf.alloc_recv(w.use_fp8)
    cnt = torch.full((w.num_experts,), -1, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_recv(buf.ctx, h.raw, w.use_fp8, send_x, send_sc, recv, scales, cnt, num_sms)
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), slot)
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    if w.use_fp8:
        q, s = oracle.quant_token(x_bits)
        assert np.array_equal(e4m3_to_bits(send_x), q)
        assert np.array_equal(send_sc.cpu().numpy().view(np.uint32), s.view(np.uint32))
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[g_of])
        assert np.array_equal(scales[rows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(send_x), x_bits)
        assert np.array_equal(bf16_to_bits(recv[rows_d]), x_bits[g_of])

    # combine: expert outputs sent back to token order, then the weighted reduce
    ye = wl.expert_outputs(w)
    y = place_rows(buf.rows, H, slot, ye, np.arange(N))
    send_y = torch.full((N * K, H), -21931, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ep.ep_combine_send(buf.ctx, h.raw, y, send_y, num_sms)
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine_recv(buf.ctx, h.raw, send_y, wts_d, out)
    assert buf.device_status() == ep.EP_OK
    m = slot.reshape(-1) >= 0
    staged = bf16_to_bits(send_y)
    assert np.array_equal(staged[m], ye.reshape(N * K, H)[m])
    assert np.all(staged[~m] == np.uint16(0xAA55))  # masked entries' rows are not written
    # the oracle reduces over the received rows only, renumbered 0..M-1 in slot order
    slot_c = np.full(N * K, -1, np.int32)
    slot_c[m] = np.arange(int(m.sum()), dtype=np.int32)
    ref = oracle.combine(ye.reshape(N * K, H)[m], slot_c.reshape(N, K), wts)
    assert np.array_equal(bf16_to_bits(out), ref)


def test_split_bf16_sends_from_x_itself():
    w = wl.TINY
    idx, x_bits, _ = _inputs(w)
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    h = buf.new_handle()
    ep.ep_dispatch_send(buf.ctx, x, torch.from_numpy(idx).cuda(), w.tokens_per_rank, False, h.raw, x, None)
    recv, _ = buf.alloc_recv(False)
    ep.ep_dispatch_recv(buf.ctx, h.raw, False, x, None, recv, None, None, 2)
    assert buf.device_status() == ep.EP_OK
    slot = h.tensors()["slot"].cpu().numpy()
    rows_d = torch.from_numpy(valid_rows(slot).astype(np.int64)).cuda()
    g_of = np.nonzero(slot.reshape(-1) >= 0)[0] // w.topk
    assert np.array_equal(bf16_to_bits(recv[rows_d]), x_bits[g_of])


def test_split_rank_layout():
    """Rank-deduplicated layout: one row per (token, destination rank)."""
    w = wl.NORMAL.with_(tokens_per_rank=256, max_tokens_per_rank=256, use_fp8=True)
    idx, x_bits, _ = _inputs(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    _, _, _, h = buf.get_rank_layout(torch.from_numpy(idx).cuda())
    o = oracle.rank_layout(idx, None, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    slot = o["rank_slot"]
    send_x = torch.empty(N, H, dtype=torch.float8_e4m3fn, device="cuda")
    send_sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
    ep.ep_dispatch_send(buf.ctx, x, None, w.tokens_per_rank, True, h.raw, send_x, send_sc)
    recv, scales = buf.alloc_rank_recv(True)
    cnt = torch.empty(w.num_ranks, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, scales, cnt, 8)
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_rank"])
    rows = valid_rows(slot)
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    g_of = np.nonzero(slot.reshape(-1) >= 0)[0] // K
    q, s = oracle.quant_token(x_bits)
    assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[g_of])
    assert np.array_equal(scales[rows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    # combine of the rank rows (weights 1) through the staging buffer
    ye = wl.expert_outputs(w)
    y = place_rows(buf.rank_rows, H, slot, ye, np.arange(N))
    send_y = torch.empty(N * K, H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine_send(buf.ctx, h.raw, y, send_y, 0)
    ep.ep_combine_recv(buf.ctx, h.raw, send_y, None, out)
    fused = torch.empty_like(out)
    ep.ep_combine(buf.ctx, y, None, h.raw, fused)
    assert buf.device_status() == ep.EP_OK
    assert torch.equal(out.view(torch.int16), fused.view(torch.int16))


def test_buffer_recv_hooks_match_the_fused_calls():
    w = wl.LL
    idx, x_bits, wts = _inputs(w)
    buf = make_buffer(w)
    buf.num_hook_sms = 16
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    (q1, s1), c1, h1 = buf.low_latency_dispatch(x, idx_d, w.max_tokens_per_rank, w.num_experts)
    (q2, s2), c2, h2, hook = buf.low_latency_dispatch(x, idx_d, w.max_tokens_per_rank, w.num_experts,
                                                      return_recv_hook=True)
    hook()
    rows = torch.from_numpy(valid_rows(h1.tensors()["slot"].cpu().numpy()).astype(np.int64)).cuda()
    assert torch.equal(q1.view(torch.uint8)[rows], q2.view(torch.uint8)[rows])
    assert torch.equal(s1[rows].view(torch.int32), s2[rows].view(torch.int32))
    assert torch.equal(c1, c2)
    y = torch.randn(buf.rows, w.hidden, device="cuda").to(torch.bfloat16)
    o1 = buf.low_latency_combine(y, idx_d, wts_d, h1, w.num_experts)
    o2, hook = buf.low_latency_combine(y, idx_d, wts_d, h2, w.num_experts, return_recv_hook=True)
    hook()
    assert buf.device_status() == ep.EP_OK
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_split_graph_replay_matches_eager():
    w = wl.LL
    idx, x_bits, wts = _inputs(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    send_x = torch.empty(N, H, dtype=torch.float8_e4m3fn, device="cuda")
    send_sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
    recv, scales = buf.alloc_recv(True)
    y = torch.randn(buf.rows, H, device="cuda").to(torch.bfloat16)
    send_y = torch.empty(N * K, H, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    h = buf.new_handle()

    def step(s):
        ep.ep_dispatch_send(buf.ctx, x, idx_d, w.tokens_per_rank, True, h.raw, send_x, send_sc, s)
        ep.ep_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, scales, None, 32, s)
        ep.ep_combine_send(buf.ctx, h.raw, y, send_y, 32, s)
        ep.ep_combine_recv(buf.ctx, h.raw, send_y, wts_d, out, s)

    step(torch.cuda.current_stream())
    eager = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert buf.device_status() == ep.EP_OK


def test_split_host_errors():
    w = wl.TINY.with_(hidden=384)
    buf = make_buffer(w)
    N, H = w.num_tokens, w.hidden
    x = torch.zeros(N, H, dtype=torch.bfloat16, device="cuda")
    h = buf.new_handle()
    sx = torch.empty(N, H, dtype=torch.uint8, device="cuda")
    sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
    idx = torch.from_numpy(wl.generate(w, with_x=False)["topk_idx"]).cuda()
    with pytest.raises(ep.EPError) as e:  # FP8 needs H % 512 == 0 here
        ep.ep_dispatch_send(buf.ctx, x, idx, w.tokens_per_rank, True, h.raw, sx, sc)
    assert e.value.status == ep.EP_ERR_UNSUPPORTED
    recv, _ = buf.alloc_recv(False)
    with pytest.raises(ep.EPError) as e:  # no layout yet
        ep.ep_dispatch_recv(buf.ctx, h.raw, False, x, None, recv, None, None)
    assert e.value.status == ep.EP_ERR_NO_LAYOUT
    ep.ep_dispatch_send(buf.ctx, x, idx, w.tokens_per_rank, False, h.raw, x, None)
    with pytest.raises(ep.EPError) as e:  # misaligned staging
        ep.ep_combine_send(buf.ctx, h.raw, recv, recv.view(-1)[1:], 0)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert buf.device_status() == ep.EP_OK
