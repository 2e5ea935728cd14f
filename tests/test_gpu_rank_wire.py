"""GPU parity of the rank-deduplicated transport whose receive runs no kernel
(ep_rank_dispatch_send / _recv, ep_rank_combine_send / _recv) against the
oracle, bit for bit, over both wires: the send buffer holds each carried
token's row in (source rank, destination rank, token) order, the run table
equals oracle.rank_runs, the receive rows equal the rank layout's dispatch,
the combine's wire brings each received row back to its send row and the
reduce equals the oracle's rank combine.  Also: a reused layout, T = 0."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import ORACLE_LAYOUT, bf16_to_bits, bits_to_bf16, e4m3_to_bits, make_buffer, place_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


CASES = {
    "normal_bf16_packed": (wl.NORMAL.with_(tokens_per_rank=256, max_tokens_per_rank=256), 0.0),
    "normal_fp8_padded": (wl.NORMAL.with_(tokens_per_rank=512, max_tokens_per_rank=512, use_fp8=True,
                                          layout=wl.PADDED), 0.0),
    "tiny_bf16_padded_masked": (wl.TINY, 0.1),
    "skew_fp8_packed_ragged": (wl.SKEW.with_(tokens_per_rank=300, layout=wl.PACKED), 0.05),
    "ll_fp8_packed_ragged": (wl.LL.with_(tokens_per_rank=37, max_tokens_per_rank=40, layout=wl.PACKED), 0.0),
}

SENTINEL = 0x5A


def _send_buffers(buf, w):
    rows = ep.ep_rank_send_rows(buf.cfg)
    if w.use_fp8:
        return (torch.empty(rows, w.hidden, dtype=torch.float8_e4m3fn, device="cuda"),
                torch.empty(rows, w.hidden // 128, dtype=torch.float32, device="cuda"))
    return torch.empty(rows, w.hidden, dtype=torch.bfloat16, device="cuda"), None


def _stage(buf, w):
    rows = ep.ep_rank_send_rows(buf.cfg)
    row = (w.hidden + w.hidden // 32) if w.use_fp8 else 2 * w.hidden
    return torch.empty(rows * max(row, 2 * w.hidden), dtype=torch.uint8).pin_memory()


@pytest.mark.parametrize("wire", [ep.EP_WIRE_DEVICE, ep.EP_WIRE_HOST])
@pytest.mark.parametrize("name", list(CASES))
def test_rank_wire_parity(name, wire):
    w, masks = CASES[name]
    d = wl.generate(w)
    idx = wl.inject_masks(d["topk_idx"], masks, 31) if masks else d["topk_idx"]
    N, K, H, R = w.num_tokens, w.topk, w.hidden, w.num_ranks
    wts = d["topk_weights"].reshape(N, K)
    x_bits = d["x_bits"].reshape(N, H)
    o = oracle.rank_layout(idx, wts, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    runs = oracle.rank_runs(idx, w.num_experts, o["rbase"])

    buf = make_buffer(w)
    h = buf.new_handle()
    x = bits_to_bf16(x_bits)
    send_x, send_sc = _send_buffers(buf, w)
    ridx = torch.full((buf.rank_rows, K), -7, dtype=torch.int32, device="cuda")
    ep.ep_rank_dispatch_send(buf.ctx, x, torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda(),
                             w.tokens_per_rank, w.use_fp8, ridx, None, h.raw, send_x, send_sc)
    stage = _stage(buf, w) if wire == ep.EP_WIRE_HOST else None
    recv, sc = buf.alloc_rank_recv(w.use_fp8)
    recv.view(torch.uint8).fill_(SENTINEL)
    cnt = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ep.ep_rank_dispatch_recv(buf.ctx, h.raw, w.use_fp8, send_x, send_sc, recv, sc, cnt, wire, stage)
    assert buf.device_status() == ep.EP_OK

    # layout and runs
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["rank_slot"])
    cnt_r, so, ro = ep.ep_rank_runs(h.raw, R)
    assert np.array_equal(np.array(cnt_r), runs["run_cnt"])
    assert np.array_equal(np.array(so), runs["send_off"])
    assert np.array_equal(np.array(ro), runs["recv_off"])
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_rank"])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    assert np.array_equal(ridx.cpu().numpy()[rows], o["recv_topk_idx"][rows])

    # send buffer and receive rows, bit for bit
    ns = runs["send_rows"]
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    if w.use_fp8:
        q_s, s_s = oracle.dispatch(x_bits, runs["send_slot"], ns, True)
        assert np.array_equal(e4m3_to_bits(send_x[:ns]), q_s)
        assert np.array_equal(send_sc[:ns].cpu().numpy().view(np.uint32), s_s.view(np.uint32))
        q_r, s_r = oracle.dispatch(x_bits, o["rank_slot"], o["rows"], True)
        got = e4m3_to_bits(recv.view(torch.uint8))
        assert np.array_equal(got[rows], q_r[rows])
        assert np.array_equal(sc[rows_d].cpu().numpy().view(np.uint32), s_r[rows].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(send_x[:ns]), oracle.dispatch(x_bits, runs["send_slot"], ns, False))
        got = recv.view(torch.uint8).cpu().numpy().reshape(o["rows"], -1)
        ref = oracle.dispatch(x_bits, o["rank_slot"], o["rows"], False)
        assert np.array_equal(got[rows].view(np.uint16), ref[rows])
    untouched = np.setdiff1d(np.arange(o["rows"]), rows)
    assert np.all(got[untouched] == SENTINEL)  # rows that receive nothing are not written

    # combine: the wire back to send order, then the reduce
    rng = np.random.default_rng(11)
    tokens = np.arange(N)
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(buf.rank_rows, H, o["rank_slot"], ye, tokens)
    send_y = torch.full((ep.ep_rank_send_rows(buf.cfg), H), -21931, dtype=torch.int16,
                        device="cuda").view(torch.bfloat16)
    ep.ep_rank_combine_send(buf.ctx, h.raw, y, send_y, wire, stage)
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_rank_combine_recv(buf.ctx, h.raw, send_y, out)
    assert buf.device_status() == ep.EP_OK
    m = runs["send_slot"] >= 0
    ye2 = ye.reshape(N, K, H)
    sy = bf16_to_bits(send_y)
    assert np.array_equal(sy[runs["send_slot"][m]], ye2[m])
    assert np.all(sy[ns:] == np.uint16(0xAA55))
    ref = oracle.combine(ye.reshape(N * K, H), np.where(m, np.arange(N * K).reshape(N, K), -1).astype(np.int32), None)
    assert np.array_equal(bf16_to_bits(out), ref)
    del rng


def test_rank_wire_reused_layout_and_empty_batch():
    """A reused layout (d_topk_idx NULL) casts again and the wire calls wait
    for nothing; T = 0 moves nothing and gives zero counts."""
    w = wl.SKEW.with_(tokens_per_rank=64, max_tokens_per_rank=64, use_fp8=True)
    d = wl.generate(w)
    N, K, H, R = w.num_tokens, w.topk, w.hidden, w.num_ranks
    buf = make_buffer(w)
    h = buf.new_handle()
    x = bits_to_bf16(d["x_bits"])
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    send_x, send_sc = _send_buffers(buf, w)
    ep.ep_rank_dispatch_send(buf.ctx, x, idx, None, w.tokens_per_rank, True, None, None, h.raw, send_x, send_sc)
    recv, sc = buf.alloc_rank_recv(True)
    ep.ep_rank_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None)
    first = recv.view(torch.uint8).clone()
    # the same layout, other token values: a second send without topk_idx
    x2 = bits_to_bf16(wl.generate(w.with_(seed=w.seed + 1))["x_bits"])
    ep.ep_rank_dispatch_send(buf.ctx, x2, None, None, w.tokens_per_rank, True, None, None, h.raw, send_x, send_sc)
    ep.ep_rank_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None)
    assert buf.device_status() == ep.EP_OK
    o = oracle.rank_layout(d["topk_idx"], None, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    q2, _ = oracle.dispatch(bits_from(x2, N, H), o["rank_slot"], o["rows"], True)
    assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8))[rows], q2[rows])
    assert not torch.equal(first, recv.view(torch.uint8))
    # a reuse with another T has no layout
    with pytest.raises(ep.EPError) as e:
        ep.ep_rank_dispatch_send(buf.ctx, x2, None, None, w.tokens_per_rank - 1, True, None, None, h.raw,
                                 send_x, send_sc)
    assert e.value.status == ep.EP_ERR_NO_LAYOUT
    # empty batch
    h0 = buf.new_handle()
    ep.ep_rank_dispatch_send(buf.ctx, x, torch.empty(R, 0, K, dtype=torch.int64, device="cuda"), None, 0, True,
                             None, None, h0.raw, send_x, send_sc)
    cnt = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ep.ep_rank_dispatch_recv(buf.ctx, h0.raw, True, send_x, send_sc, recv, sc, cnt)
    assert buf.device_status() == ep.EP_OK
    assert int(cnt.abs().sum().item()) == 0
    cnt_r, _, _ = ep.ep_rank_runs(h0.raw, R)
    assert sum(map(sum, cnt_r)) == 0


def bits_from(t, N, H):
    return bf16_to_bits(t).reshape(N, H)


def test_rank_wire_rejects_pageable_stage_and_other_layouts():
    w = wl.TINY
    d = wl.generate(w)
    buf = make_buffer(w)
    h = buf.new_handle()
    x = bits_to_bf16(d["x_bits"])
    send_x, _ = _send_buffers(buf, w)
    recv, _ = buf.alloc_rank_recv(False)
    # no rank transport layout in the handle yet
    with pytest.raises(ep.EPError) as e:
        ep.ep_rank_dispatch_recv(buf.ctx, h.raw, False, send_x, None, recv, None, None)
    assert e.value.status == ep.EP_ERR_NO_LAYOUT
    ep.ep_rank_dispatch_send(buf.ctx, x, torch.from_numpy(d["topk_idx"]).cuda(), None, w.tokens_per_rank, False,
                             None, None, h.raw, send_x, None)
    pageable = torch.empty(1 << 20, dtype=torch.uint8)
    with pytest.raises(ep.EPError) as e:
        ep.ep_rank_dispatch_recv(buf.ctx, h.raw, False, send_x, None, recv, None, None, ep.EP_WIRE_HOST, pageable)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
    # a plain layout call on the handle replaces the transport's layout
    ep.ep_get_rank_layout(buf.ctx, torch.from_numpy(d["topk_idx"]).cuda(), None, w.tokens_per_rank, None, None,
                          None, h.raw)
    with pytest.raises(ep.EPError) as e:
        ep.ep_rank_dispatch_recv(buf.ctx, h.raw, False, send_x, None, recv, None, None)
    assert e.value.status == ep.EP_ERR_NO_LAYOUT
    assert buf.device_status() == ep.EP_OK


@pytest.mark.parametrize("wire", [ep.EP_WIRE_DEVICE, ep.EP_WIRE_HOST])
def test_buffer_rank_dispatch_and_combine_hooks(wire):
    """Buffer.rank_dispatch / rank_combine with return_recv_hook=True equal the
    oracle's rank dispatch and rank combine."""
    w = wl.SKEW.with_(tokens_per_rank=96, max_tokens_per_rank=96, use_fp8=True, layout=wl.PACKED)
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    wts = d["topk_weights"].reshape(N, K)
    buf = make_buffer(w)
    x = bits_to_bf16(d["x_bits"])
    (recv, sc), cnt, ridx, rw, h, hook = buf.rank_dispatch(
        x, torch.from_numpy(d["topk_idx"]).cuda(), torch.from_numpy(wts).cuda(), use_fp8=True, wire=wire,
        return_recv_hook=True)
    hook()
    assert buf.device_status() == ep.EP_OK
    o = oracle.rank_layout(d["topk_idx"], wts, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    q, s = oracle.dispatch(d["x_bits"].reshape(N, H), o["rank_slot"], o["rows"], True)
    rd = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rd]), q[rows])
    assert np.array_equal(sc[rd].cpu().numpy().view(np.uint32), s[rows].view(np.uint32))
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(rw.cpu().numpy()[rows].view(np.uint32), o["recv_topk_weights"][rows].view(np.uint32))
    tokens = np.arange(N)
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(buf.rank_rows, H, o["rank_slot"], ye, tokens)
    out, chook = buf.rank_combine(y, h, wire=wire, return_recv_hook=True)
    chook()
    assert buf.device_status() == ep.EP_OK
    m = o["rank_slot"] >= 0
    ref = oracle.combine(ye.reshape(N * K, H), np.where(m, np.arange(N * K).reshape(N, K), -1).astype(np.int32),
                         None)
    assert np.array_equal(bf16_to_bits(out), ref)


@pytest.mark.parametrize("wire", [ep.EP_WIRE_DEVICE, ep.EP_WIRE_HOST])
def test_rank_wire_calls_replay_from_a_cuda_graph(wire):
    """Once the run sizes are on the host (after the first wire call on a
    layout), the send on the cached layout, the receive and the combine's
    wire + reduce only enqueue: captured into a CUDA graph and replayed with
    new token values, they give the oracle's bits."""
    w = wl.SKEW.with_(tokens_per_rank=64, max_tokens_per_rank=64, use_fp8=True, layout=wl.PACKED)
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    buf = make_buffer(w)
    h = buf.new_handle()
    x = bits_to_bf16(d["x_bits"])
    send_x, send_sc = _send_buffers(buf, w)
    stage = _stage(buf, w) if wire == ep.EP_WIRE_HOST else None
    recv, sc = buf.alloc_rank_recv(True)
    send_y = torch.empty(ep.ep_rank_send_rows(buf.cfg), H, dtype=torch.bfloat16, device="cuda")
    o = oracle.rank_layout(d["topk_idx"], None, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    tokens = np.arange(N)
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(buf.rank_rows, H, o["rank_slot"], ye, tokens)
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_rank_dispatch_send(buf.ctx, x, torch.from_numpy(d["topk_idx"]).cuda(), None, w.tokens_per_rank, True,
                             None, None, h.raw, send_x, send_sc)
    ep.ep_rank_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None, wire, stage)  # runs -> host
    assert buf.device_status() == ep.EP_OK

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ep.ep_rank_dispatch_send(buf.ctx, x, None, None, w.tokens_per_rank, True, None, None, h.raw, send_x,
                                 send_sc, s)
        ep.ep_rank_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None, wire, stage, s)
        ep.ep_rank_combine_send(buf.ctx, h.raw, y, send_y, wire, stage, s)
        ep.ep_rank_combine_recv(buf.ctx, h.raw, send_y, out, s)
    x2_bits = wl.generate(w.with_(seed=w.seed + 7))["x_bits"]
    x.copy_(bits_to_bf16(x2_bits))
    recv.view(torch.uint8).zero_()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert buf.device_status() == ep.EP_OK
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    q, s_ = oracle.dispatch(x2_bits.reshape(N, H), o["rank_slot"], o["rows"], True)
    rd = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rd]), q[rows])
    assert np.array_equal(sc[rd].cpu().numpy().view(np.uint32), s_[rows].view(np.uint32))
    m = o["rank_slot"] >= 0
    ref = oracle.combine(ye.reshape(N * K, H), np.where(m, np.arange(N * K).reshape(N, K), -1).astype(np.int32),
                         None)
    assert np.array_equal(bf16_to_bits(out), ref)


def _random_case(i):
    """Seeded random shape of the rank transport: 1-8 ranks including 3 and 5,
    1-5 experts per rank, top-1 to top-10 (K not dividing 32 too), T in
    [0, Tmax], masked entries and repeats, padded or packed, BF16 or FP8."""
    rng = np.random.default_rng(7700 + i)
    R = int(rng.choice([1, 2, 3, 4, 5, 8]))
    L = int(rng.choice([1, 2, 3, 5]))
    E = R * L
    Tmax = int(rng.integers(1, 80))
    T = 0 if i % 7 == 3 else int(rng.integers(1, Tmax + 1))
    K = int(rng.integers(1, 11))
    fp8 = i % 2 == 0
    H = 128 * int(rng.integers(1, 9)) if fp8 else 8 * int(rng.integers(1, 129))
    packed = bool(rng.integers(0, 2))
    idx = rng.integers(-1, E, size=(R, T, K)).astype(np.int64)
    return rng, idx, E, Tmax, H, fp8, packed


@pytest.mark.parametrize("wire", [ep.EP_WIRE_DEVICE, ep.EP_WIRE_HOST])
@pytest.mark.parametrize("i", range(10))
def test_rank_wire_random_shapes(i, wire):
    rng, idx, E, Tmax, H, fp8, packed = _random_case(i)
    R, T, K = idx.shape
    N = R * T
    from combine_get_dispatch_02_gb300 import Buffer
    buf = Buffer(R, Tmax, H, E, K, low_latency_mode=not packed)
    xb = torch.from_numpy(rng.standard_normal((N, H)).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    o = oracle.rank_layout(idx, None, E, Tmax, 1 if packed else 0)
    runs = oracle.rank_runs(idx, E, o["rbase"])
    h = buf.new_handle()
    rows_s = ep.ep_rank_send_rows(buf.cfg)
    if fp8:
        send_x = torch.empty(rows_s, H, dtype=torch.float8_e4m3fn, device="cuda")
        send_sc = torch.empty(rows_s, H // 128, dtype=torch.float32, device="cuda")
    else:
        send_x, send_sc = torch.empty(rows_s, H, dtype=torch.bfloat16, device="cuda"), None
    stage = torch.empty(rows_s * (2 * H + H // 32), dtype=torch.uint8).pin_memory() \
        if wire == ep.EP_WIRE_HOST else None
    x = bits_to_bf16(xb) if N > 0 else torch.empty(0, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_rank_dispatch_send(buf.ctx, x, torch.from_numpy(idx).cuda(), None, T, fp8, None, None, h.raw,
                             send_x, send_sc)
    recv, sc = buf.alloc_rank_recv(fp8)
    recv.view(torch.uint8).fill_(SENTINEL)
    cnt = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    ep.ep_rank_dispatch_recv(buf.ctx, h.raw, fp8, send_x, send_sc, recv, sc, cnt, wire, stage)
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_rank"])
    cnt_r, so, ro = ep.ep_rank_runs(h.raw, R)
    assert np.array_equal(np.array(cnt_r), runs["run_cnt"])
    assert np.array_equal(np.array(so), runs["send_off"])
    assert np.array_equal(np.array(ro), runs["recv_off"])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    got = recv.view(torch.uint8).cpu().numpy().reshape(o["rows"], -1)
    if fp8:
        q, s_ = oracle.dispatch(xb.reshape(N, H), o["rank_slot"], o["rows"], True)
        assert np.array_equal(got[rows], q[rows])
        rd = torch.from_numpy(rows.astype(np.int64)).cuda()
        assert np.array_equal(sc[rd].cpu().numpy().view(np.uint32), s_[rows].view(np.uint32))
    else:
        ref = oracle.dispatch(xb.reshape(N, H), o["rank_slot"], o["rows"], False)
        assert np.array_equal(got[rows].view(np.uint16), ref[rows])
    assert np.all(np.delete(got, rows, axis=0) == SENTINEL)
    # combine back over the same wire
    ye = rng.standard_normal((N, K, H)).astype(np.float32)
    ye = torch.from_numpy(ye).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = place_rows(buf.rank_rows, H, o["rank_slot"], ye, np.arange(N))
    send_y = torch.empty(rows_s, H, dtype=torch.bfloat16, device="cuda")
    out = torch.full((N, H), 7, dtype=torch.bfloat16, device="cuda")
    ep.ep_rank_combine_send(buf.ctx, h.raw, y, send_y, wire, stage)
    ep.ep_rank_combine_recv(buf.ctx, h.raw, send_y, out)
    assert buf.device_status() == ep.EP_OK
    m = o["rank_slot"] >= 0
    ref = oracle.combine(ye.reshape(N * K, H), np.where(m, np.arange(N * K).reshape(N, K), -1).astype(np.int32),
                         None) if N > 0 else np.zeros((0, H), np.uint16)
    assert np.array_equal(bf16_to_bits(out), ref)
