"""Both forms of the layout kernel, forced through the layout_form tuning knob
(1: one thread-block cluster, 2: the cooperative grid kernel over all SMs),
give the oracle's layout bit for bit at every size: expert and
rank-deduplicated layouts, padded and packed, masked entries, invalid ids
(EP_ERR_BAD_EXPERT) and padded overflow (EP_ERR_CAPACITY); the fused
layout + dispatch on the grid form too."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import ORACLE_LAYOUT, e4m3_to_bits, make_buffer, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


CASES = {
    "tiny": wl.TINY,
    "ll": wl.LL,
    "ll_ragged_packed": wl.LL.with_(tokens_per_rank=77, layout=wl.PACKED),
    "normal": wl.NORMAL,
    "skew": wl.SKEW,
    "r128_e128": wl.TINY.with_(num_ranks=128, num_experts=128, topk=8, tokens_per_rank=16, max_tokens_per_rank=16),
    "e1024_ragged": wl.TINY.with_(num_ranks=8, num_experts=1024, topk=8, tokens_per_rank=2049,
                                  max_tokens_per_rank=2050),
    "one_token": wl.TINY.with_(tokens_per_rank=1, max_tokens_per_rank=4),
    # 1M entries: too many for the cluster form's shared-memory copy of the
    # entries, so its second pass re-reads topk_idx
    "unstaged_1m_packed": wl.LL.with_(tokens_per_rank=4096, max_tokens_per_rank=4096, layout=wl.PACKED),
}


def _buf(w, form):
    buf = make_buffer(w)
    t = ep.ep_get_tuning(buf.ctx)
    t.layout_form = form
    ep.ep_set_tuning(buf.ctx, t)
    return buf


def _check(w, idx, form, expect=ep.EP_OK):
    buf = _buf(w, form)
    o = oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    ntr, nte, itr, h = buf.get_dispatch_layout(torch.from_numpy(idx).cuda())
    assert buf.device_status() == expect
    t = h.tensors()
    assert np.array_equal(t["slot"].cpu().numpy(), o["slot"])
    rows = valid_rows(o["slot"])
    assert np.array_equal(t["src_info"].cpu().numpy()[rows], o["src_info"][rows])
    for k in ("cnt_er", "off_er", "base", "tokens_per_expert"):
        assert np.array_equal(t[k].cpu().numpy(), o[k]), k
    assert np.array_equal(nte.cpu().numpy(), o["tokens_per_expert"])
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(itr.cpu().numpy().astype(np.uint8), o["is_token_in_rank"])
    return o, buf, h


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("name", list(CASES))
def test_layout_forms_match_the_oracle(name, form):
    w = CASES[name]
    _check(w, wl.generate(w, with_x=False)["topk_idx"], form)


@pytest.mark.parametrize("form", [1, 2])
def test_layout_forms_masked_bad_ids_and_overflow(form):
    w = wl.SKEW
    idx = wl.inject_masks(wl.generate(w, with_x=False)["topk_idx"], 0.1, 8)
    _check(w, idx, form)
    bad = idx.copy()
    bad.reshape(-1)[[0, 77, 5000, bad.size - 1]] = [w.num_experts, -5, 1 << 40, -2]
    o, _, _ = _check(w, bad, form, expect=ep.EP_ERR_BAD_EXPERT)
    assert o["n_bad"] == 4
    T = 700
    wo = wl.TINY.with_(num_ranks=2, num_experts=4, topk=4, tokens_per_rank=T, max_tokens_per_rank=T)
    over = np.zeros((2, T, 4), np.int64)
    over[:, :, 3] = 3
    o, _, _ = _check(wo, over, form, expect=ep.EP_ERR_CAPACITY)
    assert o["n_overflow"] == 2 * T * 3 - 2 * T


@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("name", ["tiny", "normal", "skew_packed_masked"])
def test_rank_layout_forms_match_the_oracle(name, form):
    w = {"tiny": wl.TINY, "normal": wl.NORMAL, "skew_packed_masked": wl.SKEW.with_(layout=wl.PACKED)}[name]
    d = wl.generate(w, with_x=False)
    idx = wl.inject_masks(d["topk_idx"], 0.1, 3) if "masked" in name else d["topk_idx"]
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk)
    buf = _buf(w, form)
    ntr, ridx, rw, h = buf.get_rank_layout(torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda())
    assert buf.device_status() == ep.EP_OK
    o = oracle.rank_layout(idx, wts, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["rank_slot"])
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    assert np.array_equal(ridx.cpu().numpy()[rows], o["recv_topk_idx"][rows])
    assert np.array_equal(rw.cpu().numpy()[rows].view(np.uint32), o["recv_topk_weights"][rows].view(np.uint32))


def test_fused_dispatch_on_the_grid_form():
    w = wl.LL
    d = wl.generate(w)
    N, H = w.num_tokens, w.hidden
    buf = _buf(w, 2)
    from helpers import bits_to_bf16
    (q, sc), cnt, h = buf.low_latency_dispatch(bits_to_bf16(d["x_bits"]), torch.from_numpy(d["topk_idx"]).cuda(),
                                               w.max_tokens_per_rank, w.num_experts, use_fp8=True)
    assert buf.device_status() == ep.EP_OK
    o = oracle.layout(d["topk_idx"], w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["slot"])
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    rng = np.random.default_rng(3)
    rows = valid_rows(o["slot"])
    pick = np.sort(rng.choice(len(rows), 4096, replace=False))
    g_of = (np.nonzero(o["slot"].reshape(-1) >= 0)[0] // w.topk)[pick]
    qo, so = oracle.quant_token(d["x_bits"].reshape(N, H)[g_of])
    rd = torch.from_numpy(rows[pick].astype(np.int64)).cuda()
    assert np.array_equal(e4m3_to_bits(q.view(torch.uint8)[rd]), qo)
    assert np.array_equal(sc[rd].cpu().numpy().view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("max_sms", [7, 40])
def test_grid_form_under_an_sm_cap(max_sms):
    """The grid form on a few CTAs (ep_config.max_sms), each CTA taking
    thousands of tokens: layout and fused FP8 dispatch still equal the oracle."""
    w = wl.NORMAL.with_(use_fp8=True, hidden=512)
    d = wl.generate(w)
    buf = make_buffer(w, max_sms=max_sms)
    t = ep.ep_get_tuning(buf.ctx)
    t.layout_form = 2
    ep.ep_set_tuning(buf.ctx, t)
    from helpers import bits_to_bf16
    (q, sc), cnt, h = buf.low_latency_dispatch(bits_to_bf16(d["x_bits"]), torch.from_numpy(d["topk_idx"]).cuda(),
                                               w.max_tokens_per_rank, w.num_experts, use_fp8=True)
    assert buf.device_status() == ep.EP_OK
    o = oracle.layout(d["topk_idx"], w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["slot"])
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    rows = valid_rows(o["slot"])
    qo, so = oracle.dispatch(d["x_bits"].reshape(w.num_tokens, w.hidden), o["slot"], o["rows"], True)
    rd = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert np.array_equal(e4m3_to_bits(q.view(torch.uint8)[rd]), qo[rows])
    assert np.array_equal(sc[rd].cpu().numpy().view(np.uint32), so[rows].view(np.uint32))
    ntr, nte, itr, h2 = buf.get_dispatch_layout(torch.from_numpy(d["topk_idx"]).cuda())
    assert buf.device_status() == ep.EP_OK
    t2 = h2.tensors()
    for k in ("cnt_er", "off_er", "base", "tokens_per_expert"):
        assert np.array_equal(t2[k].cpu().numpy(), o[k]), k
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(itr.cpu().numpy().astype(np.uint8), o["is_token_in_rank"])


def test_grid_form_repeated_launches_with_changing_sizes():
    """The grid form's barrier counter is back at zero after every launch:
    many launches on one handle, with token counts that change the number of
    CTAs, each give the oracle's layout."""
    w0 = wl.NORMAL.with_(hidden=512)
    buf = _buf(w0, 2)
    h = buf.new_handle()
    rng = np.random.default_rng(12)
    for it in range(24):
        T = int(rng.choice([1, 7, 100, 999, 2048, 4096]))
        w = w0.with_(tokens_per_rank=T, seed=w0.seed + it)
        idx = wl.generate(w, with_x=False)["topk_idx"]
        ntr, nte, itr, _ = buf.get_dispatch_layout(torch.from_numpy(idx).cuda(), handle=h)
        if it % 3 == 0 or it == 23:
            assert buf.device_status() == ep.EP_OK
            o = oracle.layout(idx, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
            t = h.tensors()
            assert np.array_equal(t["slot"].cpu().numpy(), o["slot"]), (it, T)
            assert np.array_equal(t["off_er"].cpu().numpy(), o["off_er"]), (it, T)
            assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"]), (it, T)
    assert buf.device_status() == ep.EP_OK
