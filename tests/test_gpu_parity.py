"""GPU parity: libep.so (through the C ABI binding) against the CPU oracle on
the same seeded inputs.

Layouts, counts, slots, BF16 rows, FP8 codes and scales are compared bit for
bit; the combine is compared bit for bit too (both sides run the same fp32
fused multiply-add chain in ascending k and round once to bf16).  At the full
sizes of the ``normal`` workload the oracle computes sampled tokens and the
rest is checked by properties that hold at any size (BF16 rows are bit copies
of their token; untouched rows keep their sentinel)."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import (ORACLE_LAYOUT, bf16_to_bits, bits_to_bf16, e4m3_to_bits, make_buffer,
                     place_rows, valid_rows)

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


def _orc_layout(w, idx):
    return oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])


def _check_layout(w, idx, buf=None, expect_status=ep.EP_OK):
    buf = buf or make_buffer(w)
    o = _orc_layout(w, idx)
    ntr, nte, itr, h = buf.get_dispatch_layout(torch.from_numpy(idx).cuda())
    assert buf.device_status() == expect_status
    t = h.tensors()
    assert h.info().has_rank_ranges == 1
    assert np.array_equal(t["slot"].cpu().numpy(), o["slot"])
    rows = valid_rows(o["slot"])
    assert np.array_equal(t["src_info"].cpu().numpy()[rows], o["src_info"][rows])
    assert np.array_equal(t["cnt_er"].cpu().numpy(), o["cnt_er"])
    assert np.array_equal(t["off_er"].cpu().numpy(), o["off_er"])
    assert np.array_equal(t["base"].cpu().numpy(), o["base"])
    assert np.array_equal(t["tokens_per_expert"].cpu().numpy(), o["tokens_per_expert"])
    assert np.array_equal(nte.cpu().numpy(), o["tokens_per_expert"])
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(itr.cpu().numpy().astype(np.uint8), o["is_token_in_rank"])
    return o, h, buf


# ------------------------------------------------------------------ layout

LAYOUT_CASES = {
    "tiny": wl.TINY,
    "ll": wl.LL,
    "normal": wl.NORMAL,
    "skew": wl.SKEW,
    "skew_packed": wl.SKEW.with_(layout=wl.PACKED),
    "ll_ragged": wl.LL.with_(tokens_per_rank=77),
    "tiny_r1_e1_k1": wl.TINY.with_(num_ranks=1, num_experts=1, topk=1, tokens_per_rank=300,
                                   max_tokens_per_rank=300),
    "tiny_l1": wl.TINY.with_(num_experts=4, topk=2),
    "tiny_k32": wl.TINY.with_(num_experts=64, topk=32),
    "r16_e1024": wl.TINY.with_(num_ranks=16, num_experts=1024, topk=8, tokens_per_rank=40,
                               max_tokens_per_rank=64),
    # the most ranks the limits allow (E % R == 0 and E*R <= 16384): one expert per rank
    "r128_e128": wl.TINY.with_(num_ranks=128, num_experts=128, topk=8, tokens_per_rank=16,
                               max_tokens_per_rank=16),
    "empty": wl.TINY.with_(tokens_per_rank=0),
    # 1M entries (the grid form; the cluster form at this size, which keeps
    # no shared-memory copy of the entries, runs in test_gpu_layout_forms)
    "unstaged_packed": wl.LL.with_(tokens_per_rank=4096, max_tokens_per_rank=4096, layout=wl.PACKED),
    # 128K+ entries: the grid form (one cooperative kernel over all SMs)
    "grid_ll_padded": wl.LL.with_(tokens_per_rank=2048, max_tokens_per_rank=2048),
    "grid_skew_packed": wl.SKEW.with_(tokens_per_rank=6000, max_tokens_per_rank=6000, layout=wl.PACKED),
    "grid_ragged_e1024": wl.TINY.with_(num_ranks=8, num_experts=1024, topk=8, tokens_per_rank=8193,
                                       max_tokens_per_rank=8200),
}


@pytest.mark.parametrize("name", list(LAYOUT_CASES))
def test_layout_parity(name):
    w = LAYOUT_CASES[name]
    idx = wl.generate(w, with_x=False)["topk_idx"]
    _check_layout(w, idx)


@pytest.mark.parametrize("name", ["tiny", "skew", "grid_ll_padded"])
def test_layout_masked_entries(name):
    w = LAYOUT_CASES[name]
    idx = wl.inject_masks(wl.generate(w, with_x=False)["topk_idx"], 0.1, 5)
    _check_layout(w, idx)


@pytest.mark.parametrize("name", ["tiny", "grid_ll_padded"])
def test_layout_bad_expert_ids_flagged_and_skipped(name):
    w = LAYOUT_CASES[name]
    idx = wl.generate(w, with_x=False)["topk_idx"].copy()
    idx.reshape(-1)[[3, 50, 400, idx.size - 1]] = [w.num_experts, -7, 10 ** 9, -2]
    o, _, buf = _check_layout(w, idx, expect_status=ep.EP_ERR_BAD_EXPERT)
    assert o["n_bad"] == 4
    assert buf.device_status() == ep.EP_OK  # the status word was cleared


@pytest.mark.parametrize("T", [8, 65536])  # the cluster form, and the grid form (524288 entries)
def test_layout_capacity_overflow_flagged(T):
    # repeated experts in a row can offer an expert more than R*Tmax entries
    w = wl.TINY.with_(num_ranks=2, num_experts=4, topk=4, tokens_per_rank=T, max_tokens_per_rank=T)
    idx = np.zeros((2, T, 4), np.int64)
    idx[:, :, 3] = 3
    o, _, _ = _check_layout(w, idx, expect_status=ep.EP_ERR_CAPACITY)
    assert o["n_overflow"] == 2 * T * 3 - 2 * T


def test_layout_deterministic():
    w = wl.SKEW
    idx = torch.from_numpy(wl.generate(w, with_x=False)["topk_idx"]).cuda()
    buf = make_buffer(w)
    ref = None
    for _ in range(10):
        _, _, _, h = buf.get_dispatch_layout(idx)
        t = h.tensors()
        cur = (t["slot"].clone(), t["cnt_er"].clone())
        if ref is None:
            ref = cur
        assert torch.equal(cur[0], ref[0]) and torch.equal(cur[1], ref[1])


# ------------------------------------------------------------------ dispatch

def _sentinel_recv(buf, use_fp8):
    recv, scales = buf.alloc_recv(use_fp8)
    recv.view(torch.uint8).fill_(0xA5)
    if scales is not None:
        scales.fill_(-3.0)
    return recv, scales


def _untouched(recv, written_rows, byte=0xA5):
    mask = torch.ones(recv.shape[0], dtype=torch.bool, device="cuda")
    mask[torch.from_numpy(written_rows.astype(np.int64)).cuda()] = False
    rest = recv.view(torch.uint8)[mask]
    return bool((rest == byte).all().item())


DISPATCH_CASES = {
    "tiny_bf16": wl.TINY,
    "tiny_fp8": wl.TINY.with_(use_fp8=True, x_scale="loguniform"),
    "ll_fp8": wl.LL,
    "ll_bf16": wl.LL.with_(use_fp8=False),
    "skew_fp8": wl.SKEW,
    "ll_ragged_fp8": wl.LL.with_(tokens_per_rank=77),
    "h384_fp8": wl.TINY.with_(hidden=384, use_fp8=True, x_scale="loguniform"),  # chunk tail
    "h200_bf16": wl.TINY.with_(hidden=200),                                     # half-segment tail
    "k32_fp8": wl.TINY.with_(num_experts=64, topk=32, use_fp8=True),
    "h16384_bf16": wl.TINY.with_(hidden=16384),                                 # warp-item kernel (above 15872)
    # the largest rows of the row kernel: a ring of 2 buffers (BF16, 31 KB rows) and of 6 (FP8)
    "h15872_bf16": wl.TINY.with_(hidden=15872, tokens_per_rank=24, max_tokens_per_rank=24),
    "h15872_fp8": wl.TINY.with_(hidden=15872, tokens_per_rank=24, max_tokens_per_rank=24, use_fp8=True),
    "h12288_bf16": wl.TINY.with_(hidden=12288, tokens_per_rank=24, max_tokens_per_rank=24),
    "h32768_fp8": wl.TINY.with_(hidden=32768, use_fp8=True, tokens_per_rank=8,
                                max_tokens_per_rank=8),                          # warp-item kernel
    "packed_fp8": wl.SKEW.with_(layout=wl.PACKED),
    # the largest hidden size (the warp-item kernel)
    "h65536_bf16": wl.TINY.with_(hidden=65536, tokens_per_rank=2, max_tokens_per_rank=2),
    "h65536_fp8": wl.TINY.with_(hidden=65536, tokens_per_rank=2, max_tokens_per_rank=2, use_fp8=True),
    # from 64K receive rows the built-in rule takes the token kernel (one CTA per token)
    "token_rule_bf16": wl.TINY.with_(num_ranks=8, tokens_per_rank=2048, max_tokens_per_rank=2048, topk=4,
                                     layout=wl.PACKED),
    "token_rule_fp8": wl.TINY.with_(num_ranks=8, tokens_per_rank=2000, max_tokens_per_rank=2048, hidden=2048,
                                    num_experts=64, topk=6, use_fp8=True, x_scale="loguniform"),
    "token_rule_fp8_k2": wl.TINY.with_(num_ranks=8, tokens_per_rank=4096, max_tokens_per_rank=4096, hidden=2560,
                                       num_experts=64, topk=2, use_fp8=True, layout=wl.PACKED),
}


@pytest.mark.parametrize("name", list(DISPATCH_CASES))
@pytest.mark.parametrize("reuse", [False, True])
def test_dispatch_parity(name, reuse):
    _check_dispatch(DISPATCH_CASES[name], reuse)


# the token kernel forced by the tuning on every shape it runs (and on two it
# does not: H = 200 and 65536 fall back to the rule's kernel); H = 400 and 384
# leave 7 / 8 threads of the CTA's last warp without channels
TOKEN_CASES = ["tiny_bf16", "tiny_fp8", "ll_fp8", "ll_bf16", "skew_fp8", "ll_ragged_fp8", "h384_fp8", "h200_bf16",
               "k32_fp8", "h16384_bf16", "h15872_fp8", "packed_fp8", "h65536_fp8", "h400_bf16"]


@pytest.mark.parametrize("name", TOKEN_CASES)
def test_token_kernel_parity(name):
    w = DISPATCH_CASES.get(name) or {"h400_bf16": wl.TINY.with_(hidden=400)}[name]
    _check_dispatch(w, False, kernel=3)
    _check_dispatch(w, True, kernel=3)


@pytest.mark.parametrize("name", ["ll_fp8", "ll_bf16", "ll_ragged_fp8"])
def test_token_kernel_sm_budget(name):
    # on an SM budget the token kernel runs a persistent grid that loops over the tokens
    _check_dispatch(DISPATCH_CASES[name], False, kernel=3, max_sms=5)


def _check_dispatch(w, reuse, kernel=None, max_sms=0):
    d = wl.generate(w)
    idx, xb = d["topk_idx"], d["x_bits"]
    o = _orc_layout(w, idx)
    buf = make_buffer(w, max_sms=max_sms)
    if kernel is not None:
        ep.ep_set_tuning(buf.ctx, ep.ep_tuning(0, 0, 0, kernel))
    x = bits_to_bf16(xb)
    idx_d = torch.from_numpy(idx).cuda()
    recv, scales = _sentinel_recv(buf, w.use_fp8)
    if reuse:
        _, _, _, h = buf.get_dispatch_layout(idx_d)
        _, cnt, _ = buf.low_latency_dispatch(x, None, w.max_tokens_per_rank, w.num_experts,
                                             use_fp8=w.use_fp8, handle=h, out=(recv, scales))
    else:
        _, cnt, h = buf.low_latency_dispatch(x, idx_d, w.max_tokens_per_rank, w.num_experts,
                                             use_fp8=w.use_fp8, out=(recv, scales))
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    # per-(expert, rank) ranges come with the explicit layout call only
    assert h.info().has_rank_ranges == (1 if reuse else 0)
    slot = o["slot"]
    rows = valid_rows(slot)
    g_of = np.nonzero(slot.reshape(-1) >= 0)[0] // w.topk
    x2 = xb.reshape(w.num_tokens, w.hidden)
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    if w.use_fp8:
        q, s = oracle.quant_token(x2)
        got_q = e4m3_to_bits(recv.view(torch.uint8)[rows_d])
        got_s = scales[rows_d].cpu().numpy()
        assert np.array_equal(got_q, q[g_of])
        assert np.array_equal(got_s.view(np.uint32), s[g_of].view(np.uint32))
        smask = torch.ones(scales.shape[0], dtype=torch.bool, device="cuda")
        smask[rows_d] = False
        assert bool((scales[smask] == -3.0).all().item())
    else:
        got = bf16_to_bits(recv[rows_d])
        assert np.array_equal(got, x2[g_of])
    assert _untouched(recv, rows)


def test_dispatch_normal_full_size():
    """Prefill / training size (R=8 x 4096 tokens, H=7168, packed): every BF16
    row is a bit copy of its token and nothing else is written; FP8 rows of a
    seeded sample of tokens match the oracle; the layout matches in full."""
    w = wl.NORMAL
    d = wl.generate(w)
    idx, xb = d["topk_idx"], d["x_bits"]
    o = _orc_layout(w, idx)
    buf = make_buffer(w)
    x = bits_to_bf16(xb).view(w.num_tokens, w.hidden)
    idx_d = torch.from_numpy(idx).cuda()
    slot_d = torch.from_numpy(o["slot"].astype(np.int64)).cuda().view(-1)
    valid = slot_d >= 0
    g_d = torch.arange(w.num_entries, device="cuda")[valid] // w.topk
    rows_d = slot_d[valid]

    recv, _ = _sentinel_recv(buf, False)
    _, cnt, h = buf.low_latency_dispatch(x, idx_d, w.max_tokens_per_rank, w.num_experts,
                                         use_fp8=False, out=(recv, None))
    assert buf.device_status() == ep.EP_OK
    assert torch.equal(h.tensors()["slot"].view(-1).long(), slot_d)
    assert torch.equal(recv[rows_d].view(torch.int16), x[g_d].view(torch.int16))
    total = int(o["tokens_per_expert"].sum())
    assert bool((recv.view(torch.uint8)[total:] == 0xA5).all().item())
    del recv

    recv8, sc = _sentinel_recv(buf, True)
    buf.low_latency_dispatch(x, None, w.max_tokens_per_rank, w.num_experts, use_fp8=True,
                             handle=h, out=(recv8, sc))
    assert buf.device_status() == ep.EP_OK
    rng = np.random.default_rng(77)
    tokens = np.sort(rng.choice(w.num_tokens, 256, replace=False))
    q, s = oracle.quant_token(xb.reshape(w.num_tokens, w.hidden)[tokens])
    for j, g in enumerate(tokens):
        for k in range(w.topk):
            r = int(o["slot"][g, k])
            assert np.array_equal(e4m3_to_bits(recv8.view(torch.uint8)[r]), q[j])
            assert np.array_equal(sc[r].cpu().numpy().view(np.uint32), s[j].view(np.uint32))


def test_dispatch_max_sms_same_bytes():
    w = wl.LL
    d = wl.generate(w)
    x = bits_to_bf16(d["x_bits"])
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    outs = []
    for ms in (0, 3):
        buf = make_buffer(w, max_sms=ms)
        recv, sc = _sentinel_recv(buf, True)
        buf.low_latency_dispatch(x, idx, w.max_tokens_per_rank, w.num_experts, use_fp8=True, out=(recv, sc))
        torch.cuda.synchronize()
        outs.append((recv.view(torch.uint8)[:: 97].clone(), sc.clone()))
        del recv, sc
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# ------------------------------------------------------------------ combine

COMBINE_CASES = {
    "tiny": (wl.TINY, True),
    "tiny_unweighted": (wl.TINY, False),
    "ll": (wl.LL, True),
    "skew": (wl.SKEW, True),
    "ll_ragged": (wl.LL.with_(tokens_per_rank=77), True),
    "k32": (wl.TINY.with_(num_experts=64, topk=32), True),
    "k1": (wl.TINY.with_(topk=1), True),
    "h200": (wl.TINY.with_(hidden=200), True),
    "h32768_k2": (wl.TINY.with_(hidden=32768, topk=2, tokens_per_rank=8, max_tokens_per_rank=8), True),
    "k3": (wl.TINY.with_(topk=3), True),
    "skew_packed": (wl.SKEW.with_(layout=wl.PACKED), True),
    "h65536": (wl.TINY.with_(hidden=65536, tokens_per_rank=2, max_tokens_per_rank=2), True),
    "r128_e128": (wl.TINY.with_(num_ranks=128, num_experts=128, topk=8, tokens_per_rank=16,
                                max_tokens_per_rank=16), True),
}


@pytest.mark.parametrize("name", list(COMBINE_CASES))
@pytest.mark.parametrize("masked", [False, True])
def test_combine_parity(name, masked):
    w, weighted = COMBINE_CASES[name]
    d = wl.generate(w, with_x=False)
    idx = d["topk_idx"]
    if masked:
        idx = wl.inject_masks(idx, 0.15, 9)
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk)
    o = _orc_layout(w, idx)
    buf = make_buffer(w)
    _, _, _, h = buf.get_dispatch_layout(torch.from_numpy(idx).cuda())
    tokens = np.arange(w.num_tokens)
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(o["rows"], w.hidden, o["slot"], ye, tokens)
    wd = torch.from_numpy(wts).cuda() if weighted else None
    out = buf.low_latency_combine(y, None, wd, h, w.num_experts)
    assert buf.device_status() == ep.EP_OK
    # oracle on the compact rows: entry (g, k) -> row g*K + k of ye
    sl = np.where(o["slot"] >= 0, np.arange(w.num_entries).reshape(w.num_tokens, w.topk), -1)
    ref = oracle.combine(ye.reshape(-1, w.hidden), sl.astype(np.int32), wts if weighted else None)
    assert np.array_equal(bf16_to_bits(out), ref)


def test_combine_normal_sampled():
    w = wl.NORMAL
    d = wl.generate(w, with_x=False)
    idx = d["topk_idx"]
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk)
    o = _orc_layout(w, idx)
    buf = make_buffer(w)
    _, _, _, h = buf.get_dispatch_layout(torch.from_numpy(idx).cuda())
    rng = np.random.default_rng(78)
    tokens = np.sort(rng.choice(w.num_tokens, 384, replace=False))
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(o["rows"], w.hidden, o["slot"], ye, tokens)
    out = buf.low_latency_combine(y, None, torch.from_numpy(wts).cuda(), h, w.num_experts)
    assert buf.device_status() == ep.EP_OK
    sl = np.arange(len(tokens) * w.topk, dtype=np.int32).reshape(len(tokens), w.topk)
    ref = oracle.combine(ye.reshape(-1, w.hidden), sl, wts[tokens])
    assert np.array_equal(bf16_to_bits(out[torch.from_numpy(tokens).cuda()]), ref)


# ------------------------------------------------------------------ end to end

def test_round_trip_fp8_ll():
    """combine(identity(dispatch(x))) with weights summing to one returns x
    within the FP8 bound (identity expert = dequantise, round to bf16)."""
    w = wl.LL
    d = wl.generate(w)
    buf = make_buffer(w)
    x = bits_to_bf16(d["x_bits"])
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    (recv, sc), _, h = buf.low_latency_dispatch(x, idx, w.max_tokens_per_rank, w.num_experts, use_fp8=True)
    rows = h.tensors()["slot"].view(-1).long()
    rows = rows[rows >= 0]
    y = torch.zeros(recv.shape, dtype=torch.bfloat16, device="cuda")
    deq = recv.view(torch.uint8)[rows].view(torch.float8_e4m3fn).float().view(len(rows), -1, 128) \
        * sc[rows].unsqueeze(-1)
    y[rows] = deq.view(len(rows), -1).to(torch.bfloat16)
    wts = torch.from_numpy(d["topk_weights"].reshape(w.num_tokens, w.topk)).cuda()
    out = buf.low_latency_combine(y, idx, wts, h, w.num_experts).double()
    assert buf.device_status() == ep.EP_OK
    xf = x.view(w.num_tokens, w.hidden).double()
    scale = torch.from_numpy(oracle.quant_token(d["x_bits"].reshape(w.num_tokens, w.hidden))[1]).cuda()
    scale = scale.double().repeat_interleave(128, dim=1)
    bound = (2.0 ** -4 * xf.abs() + 2.0 ** -10 * scale) * (1 + 2.0 ** -8) \
        + 2.0 ** -8 * xf.abs() * (1 + 2.0 ** -4) + 2.0 ** -8 * out.abs() + w.topk * 2.0 ** -22 * xf.abs()
    assert bool(((out - xf).abs() <= bound).all().item())


def test_backward_pair_normal():
    """Training backward in the packed layout: grad of combine is a BF16
    dispatch of the output gradient with the cached handle; grad of dispatch
    is an unweighted combine of the received-row gradients."""
    w = wl.NORMAL
    d = wl.generate(w, with_x=False)
    idx = d["topk_idx"]
    o = _orc_layout(w, idx)
    buf = make_buffer(w)
    _, _, _, h = buf.get_dispatch_layout(torch.from_numpy(idx).cuda())
    rng = np.random.default_rng(79)
    gout = rng.standard_normal((w.num_tokens, w.hidden), dtype=np.float32)
    gout_b = bits_to_bf16(wl._bf16_bits(gout))
    recv, _ = _sentinel_recv(buf, False)
    buf.low_latency_dispatch(gout_b, None, w.max_tokens_per_rank, w.num_experts, use_fp8=False,
                             handle=h, out=(recv, None))
    slot_d = torch.from_numpy(o["slot"].astype(np.int64)).cuda().view(-1)
    g_d = torch.arange(w.num_entries, device="cuda") // w.topk
    ok = slot_d >= 0
    assert torch.equal(recv[slot_d[ok]].view(torch.int16), gout_b[g_d[ok]].view(torch.int16))
    tokens = np.sort(rng.choice(w.num_tokens, 256, replace=False))
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(o["rows"], w.hidden, o["slot"], ye, tokens)
    gx = buf.low_latency_combine(y, None, None, h, w.num_experts)
    assert buf.device_status() == ep.EP_OK
    sl = np.arange(len(tokens) * w.topk, dtype=np.int32).reshape(len(tokens), w.topk)
    ref = oracle.combine(ye.reshape(-1, w.hidden), sl, None)
    assert np.array_equal(bf16_to_bits(gx[torch.from_numpy(tokens).cuda()]), ref)


def test_empty_batch():
    w = wl.TINY.with_(tokens_per_rank=0)
    buf = make_buffer(w)
    x = torch.empty(w.num_ranks, 0, w.hidden, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.num_ranks, 0, w.topk, dtype=torch.int64, device="cuda")
    recv, cnt, h = buf.low_latency_dispatch(x, idx, w.max_tokens_per_rank, w.num_experts, use_fp8=False)
    out = buf.low_latency_combine(recv, idx, None, h, w.num_experts)
    assert buf.device_status() == ep.EP_OK
    assert out.shape == (0, w.hidden)
    assert int(cnt.sum().item()) == 0


def test_fresh_dispatch_layout_unstaged():
    """The layout computed inside ep_dispatch (no per-rank ranges) at a size
    whose entries do not fit in shared memory."""
    w = LAYOUT_CASES["unstaged_packed"]
    d = wl.generate(w, with_x=False)
    o = _orc_layout(w, d["topk_idx"])
    buf = make_buffer(w)
    x = torch.zeros(w.num_tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    _, cnt, h = buf.low_latency_dispatch(x, torch.from_numpy(d["topk_idx"]).cuda(), w.max_tokens_per_rank,
                                         w.num_experts, use_fp8=True)
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["slot"])
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
