"""GPU parity of the rank-deduplicated (normal-mode) transport against the
oracle: layout (rows per rank, local top-k of each received row), dispatch
into rank rows (BF16 bit copy, FP8 cast) and the per-token sum over its rank
rows, all bit for bit."""
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
    "normal": wl.NORMAL,
    "normal_fp8_padded": wl.NORMAL.with_(tokens_per_rank=512, max_tokens_per_rank=512, use_fp8=True,
                                         layout=wl.PADDED),
    "tiny_padded": wl.TINY,
    "skew_packed": wl.SKEW.with_(layout=wl.PACKED),
    "ll_ragged": wl.LL.with_(tokens_per_rank=77, layout=wl.PACKED),
}


def _rank_layout(w, idx, wts):
    buf = make_buffer(w)
    ntr, ridx, rw, h = buf.get_rank_layout(torch.from_numpy(idx).cuda(), torch.from_numpy(wts).cuda())
    assert buf.device_status() == ep.EP_OK
    o = oracle.rank_layout(idx, wts, w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    return buf, h, ntr, ridx, rw, o


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("masked", [False, True])
def test_rank_layout_parity(name, masked):
    w = CASES[name]
    d = wl.generate(w, with_x=False)
    idx = wl.inject_masks(d["topk_idx"], 0.1, 21) if masked else d["topk_idx"]
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk)
    buf, h, ntr, ridx, rw, o = _rank_layout(w, idx, wts)
    info = h.info()
    assert info.rank_mode == 1
    t = h.tensors()
    R = w.num_ranks
    assert np.array_equal(t["slot"].cpu().numpy(), o["rank_slot"])
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(t["tokens_per_expert"].cpu().numpy()[:R], o["tokens_per_rank"])
    assert np.array_equal(t["base"].cpu().numpy()[:R], o["rbase"])
    rows = o["rank_slot"][o["rank_slot"] >= 0]
    assert np.array_equal(t["src_info"].cpu().numpy()[rows], o["src_info"][rows])
    assert np.array_equal(ridx.cpu().numpy()[rows], o["recv_topk_idx"][rows])
    assert np.array_equal(rw.cpu().numpy()[rows].view(np.uint32), o["recv_topk_weights"][rows].view(np.uint32))


@pytest.mark.parametrize("name", list(CASES))
def test_rank_dispatch_and_combine_parity(name):
    w = CASES[name]
    d = wl.generate(w)
    idx, xb = d["topk_idx"], d["x_bits"]
    wts = d["topk_weights"].reshape(w.num_tokens, w.topk)
    buf, h, ntr, ridx, rw, o = _rank_layout(w, idx, wts)
    x = bits_to_bf16(xb)
    recv, sc = buf.alloc_rank_recv(w.use_fp8)
    _, cnt, _ = buf.low_latency_dispatch(x, None, w.max_tokens_per_rank, w.num_experts, use_fp8=w.use_fp8,
                                         handle=h, out=(recv, sc))
    assert buf.device_status() == ep.EP_OK
    assert np.array_equal(cnt.cpu().numpy()[:w.num_ranks], o["tokens_per_rank"])
    slot = o["rank_slot"]
    rows = slot[slot >= 0]
    g_of = np.nonzero(slot.reshape(-1) >= 0)[0] // w.topk
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    x2 = xb.reshape(w.num_tokens, w.hidden)
    if w.use_fp8:
        rng = np.random.default_rng(5)
        pick = rng.choice(len(rows), min(len(rows), 2048), replace=False)
        q, s = oracle.quant_token(x2[g_of[pick]])
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d[pick]]), q)
        assert np.array_equal(sc[rows_d[pick]].cpu().numpy().view(np.uint32), s.view(np.uint32))
    else:
        assert torch.equal(recv[rows_d].view(torch.int16),
                           x.view(-1, w.hidden)[torch.from_numpy(g_of).cuda()].view(torch.int16))
    # combine: sum of each token's rank rows (expert outputs drawn per (token, k))
    rng = np.random.default_rng(6)
    tokens = np.sort(rng.choice(w.num_tokens, min(w.num_tokens, 512), replace=False))
    ye = wl.expert_outputs(w, tokens)
    y = place_rows(buf.rank_rows, w.hidden, slot, ye, tokens)
    out = buf.low_latency_combine(y, None, None, h, w.num_experts)
    assert buf.device_status() == ep.EP_OK
    sl = np.where(slot[tokens] >= 0, np.arange(len(tokens) * w.topk).reshape(len(tokens), w.topk), -1)
    ref = oracle.combine(ye.reshape(-1, w.hidden), sl.astype(np.int32), None)
    assert np.array_equal(bf16_to_bits(out[torch.from_numpy(tokens).cuda()]), ref)


def test_rank_mode_sends_fewer_rows():
    """Group-limited gating (top-4 of 8 groups, one group per rank) sends each
    token to at most 4 ranks instead of 8 expert rows."""
    w = wl.NORMAL
    d = wl.generate(w, with_x=False)
    _, h, ntr, _, _, o = _rank_layout(w, d["topk_idx"], d["topk_weights"].reshape(w.num_tokens, w.topk))
    per_token = (h.tensors()["slot"] >= 0).sum(dim=1)
    assert int(per_token.max().item()) <= 4
    assert 3 * w.num_tokens < int(ntr.sum().item()) <= 4 * w.num_tokens
