"""GPU parity of the round trip: token-range dispatch / combine, the identity
expert (FP8 rows back to BF16) and ep_round_trip over token chunks, against
the oracle's dispatch -> dequant_rows -> combine on the same seeded inputs.

Everything is compared bit for bit: the identity expert's rows (one fp32
multiply, one bf16 rounding on both sides) and the combined tokens for every
chunk size.  The oracle works on the received rows only (the receive-row ids
renumbered 0..M-1): dispatch, the identity expert and combine treat every row
on its own, so the renumbering changes no value."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import ORACLE_LAYOUT, bf16_to_bits, bits_to_bf16, make_buffer, valid_rows

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


def _compact(slot: np.ndarray):
    """(slot with the received rows renumbered 0..M-1 in slot order, the
    original row ids in that order)."""
    flat = slot.reshape(-1)
    m = flat >= 0
    rows = flat[m]
    sc = np.full(flat.shape, -1, np.int32)
    sc[m] = np.arange(rows.size, dtype=np.int32)
    return sc.reshape(slot.shape), rows


def _oracle_round_trip(x_bits, slot, weights, use_fp8):
    """(out [N, H] bits, y [M, H] bits of the received rows in slot order)."""
    sc, rows = _compact(slot)
    if use_fp8:
        q, s = oracle.dispatch(x_bits, sc, rows.size, True)
        y = oracle.dequant_rows(q, s, sc)
    else:
        y = oracle.dispatch(x_bits, sc, rows.size, False)
    return oracle.combine(y, sc, weights), y


def _inputs(w, masks=0.0):
    d = wl.generate(w)
    idx = d["topk_idx"]
    if masks:
        idx = wl.inject_masks(idx, masks, 11)
    x_bits = d["x_bits"].reshape(w.num_tokens, w.hidden)
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk).astype(np.float32)
    return idx, x_bits, wts


def _sentinel_y(buf):
    return torch.full((buf.rows, buf.hidden), -21931, dtype=torch.int16, device="cuda").view(torch.bfloat16)


# ------------------------------------------------------------------ identity expert

IDENTITY_CASES = {
    "tiny_fp8": wl.TINY.with_(use_fp8=True, x_scale="loguniform"),
    "ll_fp8": wl.LL,
    "skew_packed_fp8": wl.SKEW.with_(layout=wl.PACKED),
    "h384_fp8": wl.TINY.with_(hidden=384, use_fp8=True, x_scale="loguniform"),  # item tail
    "tiny_bf16": wl.TINY,
    "h200_bf16": wl.TINY.with_(hidden=200),                                     # 8-channel tail
}


@pytest.mark.parametrize("name", list(IDENTITY_CASES))
def test_identity_expert_parity(name):
    w = IDENTITY_CASES[name]
    idx, x_bits, _ = _inputs(w, masks=0.05)
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    recv, scales = buf.alloc_recv(w.use_fp8)
    _, _, h = buf.low_latency_dispatch(x, torch.from_numpy(idx).cuda(), w.max_tokens_per_rank,
                                       w.num_experts, use_fp8=w.use_fp8, out=(recv, scales))
    y = _sentinel_y(buf)
    ep.ep_expert_identity(buf.ctx, h.raw, w.use_fp8, recv, scales, y, 0, w.num_tokens)
    assert buf.device_status() == ep.EP_OK
    slot = h.tensors()["slot"].cpu().numpy()
    o = oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    assert np.array_equal(slot, o["slot"])
    _, y_ref = _oracle_round_trip(x_bits, slot, None, w.use_fp8)
    rows = valid_rows(slot)
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert np.array_equal(bf16_to_bits(y[rows_d]), y_ref)
    mask = torch.ones(buf.rows, dtype=torch.bool, device="cuda")
    mask[rows_d] = False
    assert bool((y.view(torch.int16)[mask] == -21931).all().item())


def test_identity_expert_token_range_touches_only_its_rows():
    w = IDENTITY_CASES["tiny_fp8"]
    idx, x_bits, _ = _inputs(w)
    buf = make_buffer(w)
    recv, scales = buf.alloc_recv(True)
    _, _, h = buf.low_latency_dispatch(bits_to_bf16(x_bits), torch.from_numpy(idx).cuda(),
                                       w.max_tokens_per_rank, w.num_experts, use_fp8=True,
                                       out=(recv, scales))
    y = _sentinel_y(buf)
    g0, g1 = 37, 90
    ep.ep_expert_identity(buf.ctx, h.raw, True, recv, scales, y, g0, g1)
    slot = h.tensors()["slot"].cpu().numpy()
    inside = valid_rows(slot[g0:g1])
    outside = np.setdiff1d(valid_rows(slot), inside)
    written = (y.view(torch.int16) != -21931).any(dim=1).cpu().numpy()
    assert written[inside].all() and not written[outside].any()


# ------------------------------------------------------------------ ranges

def test_ranges_compose_to_the_full_calls():
    w = wl.LL.with_(tokens_per_rank=77)
    idx, x_bits, wts = _inputs(w, masks=0.05)
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    r_full, s_full = buf.alloc_recv(True)
    _, _, h = buf.low_latency_dispatch(x, idx_d, w.max_tokens_per_rank, w.num_experts, use_fp8=True,
                                       out=(r_full, s_full))
    r_part, s_part = buf.alloc_recv(True)
    N = w.num_tokens
    cuts = [0, 1, 500, 501, 1999, N]
    for a, b in zip(cuts[:-1], cuts[1:]):
        ep.ep_dispatch_range(buf.ctx, x, True, h.raw, a, b, r_part, s_part)
    rows = torch.from_numpy(valid_rows(h.tensors()["slot"].cpu().numpy()).astype(np.int64)).cuda()
    assert torch.equal(r_full.view(torch.uint8)[rows], r_part.view(torch.uint8)[rows])
    assert torch.equal(s_full[rows].view(torch.int32), s_part[rows].view(torch.int32))
    y = torch.empty(buf.rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    ep.ep_expert_identity(buf.ctx, h.raw, True, r_full, s_full, y, 0, N)
    full = buf.low_latency_combine(y, None, wts_d, h, w.num_experts)
    part = torch.empty_like(full)
    for a, b in zip(cuts[:-1], cuts[1:]):
        ep.ep_combine_range(buf.ctx, y, wts_d, h.raw, a, b, part)
    assert buf.device_status() == ep.EP_OK
    assert torch.equal(full.view(torch.int16), part.view(torch.int16))


def test_range_host_errors():
    w = wl.TINY
    buf = make_buffer(w)
    x = torch.zeros(w.num_tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    recv, _ = buf.alloc_recv(False)
    h = buf.new_handle()
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch_range(buf.ctx, x, False, h.raw, 0, 4, recv, None)
    assert e.value.status == ep.EP_ERR_NO_LAYOUT
    _, _, _, h = buf.get_dispatch_layout(torch.from_numpy(wl.generate(w, with_x=False)["topk_idx"]).cuda(), h)
    N = w.num_tokens
    for a, b in [(-1, 3), (5, 4), (0, N + 1)]:
        with pytest.raises(ep.EPError) as e:
            ep.ep_dispatch_range(buf.ctx, x, False, h.raw, a, b, recv, None)
        assert e.value.status == ep.EP_ERR_INVALID_ARG
        with pytest.raises(ep.EPError) as e:
            ep.ep_combine_range(buf.ctx, recv, None, h.raw, a, b, x)
        assert e.value.status == ep.EP_ERR_INVALID_ARG
    # FP8 identity needs scales; an empty range is a no-op
    y = torch.empty(buf.rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError):
        ep.ep_expert_identity(buf.ctx, h.raw, True, recv, None, y, 0, N)
    ep.ep_expert_identity(buf.ctx, h.raw, True, recv, None, y, 3, 3)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ round trip

ROUND_TRIP_CASES = {
    "tiny_fp8": (wl.TINY.with_(use_fp8=True, x_scale="loguniform"), 0.0),
    "ll_fp8": (wl.LL, 0.0),
    "ll_bf16_in_place": (wl.LL.with_(use_fp8=False), 0.0),
    "skew_fp8_masked": (wl.SKEW.with_(tokens_per_rank=300), 0.1),
    "packed_ragged_fp8": (wl.LL.with_(tokens_per_rank=77, layout=wl.PACKED), 0.05),
}


@pytest.mark.parametrize("name", list(ROUND_TRIP_CASES))
def test_round_trip_parity_every_chunk_size(name):
    w, masks = ROUND_TRIP_CASES[name]
    idx, x_bits, wts = _inputs(w, masks)
    N = w.num_tokens
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    o = oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    out_ref, _ = _oracle_round_trip(x_bits, o["slot"], wts, w.use_fp8)
    recv = buf.alloc_recv(w.use_fp8)
    y = recv[0] if not w.use_fp8 else torch.empty(buf.rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    h = None
    for chunk in [0, 1, 7, 512, N - 1, N, ep.EP_CHUNK_AUTO]:
        out, h = buf.round_trip(x, idx_d if h is None else None, wts_d, use_fp8=w.use_fp8,
                                chunk_tokens=chunk, handle=h, recv=recv, y=y)
        assert buf.device_status() == ep.EP_OK
        assert np.array_equal(bf16_to_bits(out), out_ref), f"chunk_tokens={chunk}"


def test_round_trip_rank_layout():
    """Round trip on a rank-deduplicated layout: one row per (token, rank),
    the rank rows summed with weight 1 (the expert side would weight them)."""
    w = wl.NORMAL.with_(tokens_per_rank=256, max_tokens_per_rank=256, use_fp8=True)
    idx, x_bits, _ = _inputs(w)
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    _, _, _, h = buf.get_rank_layout(torch.from_numpy(idx).cuda())
    o = oracle.rank_layout(idx, None, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["rank_slot"])
    out_ref, _ = _oracle_round_trip(x_bits, o["rank_slot"], None, True)
    recv, scales = buf.alloc_rank_recv(True)
    y = torch.empty(buf.rank_rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(w.num_tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    for chunk in [0, 100]:
        ep.ep_round_trip(buf.ctx, x, None, w.tokens_per_rank, None, True, h.raw, recv, scales, y, out, chunk)
        assert buf.device_status() == ep.EP_OK
        assert np.array_equal(bf16_to_bits(out), out_ref)


def test_round_trip_graph_replay_matches_eager():
    w = wl.LL
    idx, x_bits, wts = _inputs(w)
    buf = make_buffer(w)
    x = bits_to_bf16(x_bits)
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    recv = buf.alloc_recv(True)
    y = torch.empty(buf.rows, w.hidden, dtype=torch.bfloat16, device="cuda")
    h = buf.new_handle()
    eager, _ = buf.round_trip(x, idx_d, wts_d, chunk_tokens=512, handle=h, recv=recv, y=y)
    eager = eager.clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ep.ep_round_trip(buf.ctx, x, idx_d, w.tokens_per_rank, wts_d, True, h.raw, recv[0], recv[1],
                             y, out, 512, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert buf.device_status() == ep.EP_OK


def test_auto_chunk_fills_most_of_l2():
    w = wl.LL
    buf = make_buffer(w)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    H, K = w.hidden, w.topk
    for fp8, row in ((True, H + H // 32 + 2 * H), (False, 2 * H)):
        c = ep.ep_round_trip_auto_chunk(buf.ctx, fp8)
        assert c % 64 == 0 and c >= 64
        assert c * K * row <= 0.7 * l2 < (c + 64) * K * row
    r = min(K, w.num_ranks)
    assert ep.ep_round_trip_auto_chunk(buf.ctx, True, True) == \
        max(64, int(l2 * 7 // 10 // (r * (H + H // 32 + 2 * H)) // 64 * 64))
    h = buf.new_handle()  # kept alive across the call
    with pytest.raises(ep.EPError) as e:
        ep.ep_round_trip(buf.ctx, torch.empty(1, dtype=torch.bfloat16, device="cuda"), None, 0, None, True,
                         h.raw, None, None, None, None, -2)
    assert e.value.status == ep.EP_ERR_INVALID_ARG
