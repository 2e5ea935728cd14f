"""GPU parity over seeded random shapes: rank counts and experts per rank that
are not powers of two (3, 5, 6 ranks; 3 or 5 experts per rank), hidden sizes
that are any multiple of 8 (BF16) or of 128 (FP8) up to 2048 (so the row and
warp-item dispatch kernels run at odd sizes, and the token kernel, forced on
the cached layout, too), T anywhere in
[0, Tmax], top-k up to 12 (also above E, with repeated experts), masked
entries, both layouts and padded overflow.  Each case runs the fresh dispatch
(layout inside), the explicit layout and the combine through the C ABI and
compares all of it with the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import Buffer
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from helpers import bf16_to_bits, bits_to_bf16, e4m3_to_bits, place_rows, valid_rows

pytestmark = pytest.mark.gpu

CASES = 32


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _case(i):
    """Sizes and topk_idx of case i.  Every eighth case (from 3) has no
    tokens; every eighth (from 6) sends ~70% of its entries to one expert of
    a padded layout, so that expert's buffer overflows."""
    rng = np.random.default_rng(4200 + i)
    R = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 16]))
    L = int(rng.choice([1, 2, 3, 5, 8]))
    E = R * L
    Tmax = int(rng.integers(1, 97))
    T = Tmax if i % 5 == 0 else int(rng.integers(0, Tmax + 1))
    K = int(rng.integers(1, 13))
    fp8 = i % 2 == 1
    H = 128 * int(rng.integers(1, 17)) if fp8 else 8 * int(rng.integers(1, 257))
    if i % 4 == 0:  # BF16 rows of a multiple of 512 channels go to the row kernel
        H = 512 * int(rng.integers(1, 5))
    packed = bool(rng.integers(0, 2))
    weighted = i % 3 != 0
    hot = i % 8 == 6
    if i % 8 == 3:
        T = 0
    if hot:
        T, K, packed = Tmax, max(K, 3), False
    idx = rng.integers(-1, E, size=(R, T, K)).astype(np.int64)  # -1 masks, repeats
    if hot:
        idx = np.where(rng.random(idx.shape) < 0.7, int(rng.integers(0, E)), idx)
    return rng, idx, E, Tmax, H, fp8, packed, weighted


@pytest.mark.parametrize("i", range(CASES))
def test_random_shape_parity(i):
    rng, idx, E, Tmax, H, fp8, packed, weighted = _case(i)
    R, T, K = idx.shape
    N = R * T
    o = oracle.layout(idx, E, Tmax, 1 if packed else 0)
    want_status = ep.EP_ERR_CAPACITY if o["n_overflow"] > 0 else ep.EP_OK
    scale = np.exp(rng.uniform(np.log(1e-2), np.log(1e2), size=(N, 1)))
    xb = _bf16_bits(rng.standard_normal((N, H)) * scale)
    buf = Buffer(R, Tmax, H, E, K, low_latency_mode=not packed)

    # fresh dispatch: layout and rows in one call
    x = bits_to_bf16(xb.reshape(R, T, H))
    idx_d = torch.from_numpy(idx).cuda()
    recv, scales = buf.alloc_recv(fp8)
    recv.view(torch.uint8).fill_(0xA5)
    if fp8:
        scales.fill_(-3.0)
    _, cnt, h = buf.low_latency_dispatch(x, idx_d, Tmax, E, use_fp8=fp8, out=(recv, scales))
    assert buf.device_status() == want_status
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    assert np.array_equal(h.tensors()["slot"].cpu().numpy(), o["slot"])
    rows = valid_rows(o["slot"])
    g_of = np.nonzero(o["slot"].reshape(-1) >= 0)[0] // K
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    if fp8:
        q, s = oracle.quant_token(xb)
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[g_of])
        assert np.array_equal(scales[rows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(recv[rows_d]), xb[g_of])
    rest = torch.ones(recv.shape[0], dtype=torch.bool, device="cuda")
    rest[rows_d] = False
    assert bool((recv.view(torch.uint8)[rest] == 0xA5).all().item())

    # the same rows from the token kernel on the cached layout (where H suits it:
    # a multiple of 16, FP8 of 128; the rule's kernel elsewhere)
    ep.ep_set_tuning(buf.ctx, ep.ep_tuning(0, 0, 0, 3))
    recv.view(torch.uint8).fill_(0xA5)
    if fp8:
        scales.fill_(-3.0)
    buf.low_latency_dispatch(x, None, Tmax, E, use_fp8=fp8, handle=h, out=(recv, scales))
    assert buf.device_status() == ep.EP_OK  # (a capacity overflow is the layout's to report)
    if fp8:
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[g_of])
        assert np.array_equal(scales[rows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(recv[rows_d]), xb[g_of])
    assert bool((recv.view(torch.uint8)[rest] == 0xA5).all().item())
    ep.ep_set_tuning(buf.ctx, ep.ep_tuning())

    # explicit layout: every array of it
    ntr, nte, itr, h2 = buf.get_dispatch_layout(idx_d)
    assert buf.device_status() == want_status
    t = h2.tensors()
    assert np.array_equal(t["slot"].cpu().numpy(), o["slot"])
    assert np.array_equal(t["src_info"].cpu().numpy()[rows], o["src_info"][rows])
    assert np.array_equal(t["cnt_er"].cpu().numpy(), o["cnt_er"])
    assert np.array_equal(t["off_er"].cpu().numpy(), o["off_er"])
    assert np.array_equal(t["base"].cpu().numpy(), o["base"])
    assert np.array_equal(nte.cpu().numpy(), o["tokens_per_expert"])
    assert np.array_equal(ntr.cpu().numpy(), o["tokens_per_rank"])
    assert np.array_equal(itr.cpu().numpy().astype(np.uint8), o["is_token_in_rank"])

    # combine of seeded expert outputs in the receive layout
    wts = rng.random((N, K)).astype(np.float32)
    ye = _bf16_bits(rng.standard_normal((N, K, H)))
    if N > 0:
        y = place_rows(o["rows"], H, o["slot"], ye, np.arange(N))
    else:
        y = torch.zeros(o["rows"], H, dtype=torch.bfloat16, device="cuda")
    wd = torch.from_numpy(wts).cuda() if weighted else None
    out = buf.low_latency_combine(y, None, wd, h2, E)
    assert buf.device_status() == ep.EP_OK
    assert tuple(out.shape) == (N, H)
    sl = np.where(o["slot"] >= 0, np.arange(N * K).reshape(N, K), -1).astype(np.int32)
    ref = oracle.combine(ye.reshape(-1, H), sl, wts if weighted else None)
    assert np.array_equal(bf16_to_bits(out), ref)


def _compact(slot: np.ndarray):
    """slot with the received rows renumbered 0..M-1 in slot order."""
    flat = slot.reshape(-1)
    m = flat >= 0
    sc = np.full(flat.shape, -1, np.int32)
    sc[m] = np.arange(int(m.sum()), dtype=np.int32)
    return sc.reshape(slot.shape)


EXTRA = 16


@pytest.mark.parametrize("i", range(EXTRA))
def test_random_shape_rank_round_trip_split(i):
    """The other calls at the same kind of shapes: the rank-deduplicated
    layout with its dispatch and combine, the chunked round trip
    (dispatch -> identity expert -> combine) and the split send / receive-hook
    dispatch and combine."""
    rng, idx, E, Tmax, H, fp8, packed, weighted = _case(CASES + i)
    R, T, K = idx.shape
    N = R * T
    lay = 1 if packed else 0
    o = oracle.layout(idx, E, Tmax, lay)
    want_status = ep.EP_ERR_CAPACITY if o["n_overflow"] > 0 else ep.EP_OK
    scale = np.exp(rng.uniform(np.log(1e-2), np.log(1e2), size=(N, 1)))
    xb = _bf16_bits(rng.standard_normal((N, H)) * scale)
    wts = rng.random((N, K)).astype(np.float32)
    ye = _bf16_bits(rng.standard_normal((N, K, H)))
    hook_sms = int(rng.choice([0, 3]))
    buf = Buffer(R, Tmax, H, E, K, low_latency_mode=not packed, num_hook_sms=hook_sms)
    x = bits_to_bf16(xb.reshape(R, T, H))
    idx_d = torch.from_numpy(idx).cuda()
    wts_d = torch.from_numpy(wts).cuda()
    wd = wts_d if weighted else None
    wref = wts if weighted else None
    tokens = np.arange(N)

    # rank-deduplicated layout, its dispatch and its (unweighted) combine
    ro = oracle.rank_layout(idx, wts, E, Tmax, lay)
    ntr, ridx, rw, hr = buf.get_rank_layout(idx_d, wts_d)
    assert buf.device_status() == ep.EP_OK
    rslot = ro["rank_slot"]
    rrows = rslot[rslot >= 0]
    assert np.array_equal(hr.tensors()["slot"].cpu().numpy(), rslot)
    assert np.array_equal(ntr.cpu().numpy(), ro["tokens_per_rank"])
    assert np.array_equal(hr.tensors()["src_info"].cpu().numpy()[rrows], ro["src_info"][rrows])
    assert np.array_equal(ridx.cpu().numpy()[rrows], ro["recv_topk_idx"][rrows])
    assert np.array_equal(rw.cpu().numpy()[rrows].view(np.uint32), ro["recv_topk_weights"][rrows].view(np.uint32))
    recv, sc = buf.alloc_rank_recv(fp8)
    buf.low_latency_dispatch(x, None, Tmax, E, use_fp8=fp8, handle=hr, out=(recv, sc))
    assert buf.device_status() == ep.EP_OK
    g_of = np.nonzero(rslot.reshape(-1) >= 0)[0] // K
    rrows_d = torch.from_numpy(rrows.astype(np.int64)).cuda()
    if fp8:
        q, s = oracle.quant_token(xb)
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rrows_d]), q[g_of])
        assert np.array_equal(sc[rrows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(recv[rrows_d]), xb[g_of])
    if N > 0:
        yr = place_rows(buf.rank_rows, H, rslot, ye, tokens)
        out = buf.low_latency_combine(yr, None, None, hr, E)
        assert buf.device_status() == ep.EP_OK
        sl = np.where(rslot >= 0, np.arange(N * K).reshape(N, K), -1).astype(np.int32)
        assert np.array_equal(bf16_to_bits(out), oracle.combine(ye.reshape(-1, H), sl, None))
    del recv, sc

    # round trip over chunks (identity expert), against the oracle's
    # dispatch -> dequant_rows -> combine on the received rows
    chunk = int(rng.choice([0, -1, int(rng.integers(1, max(N, 1) + 1))]))
    out, h = buf.round_trip(x, idx_d, wd, use_fp8=fp8, chunk_tokens=chunk)
    assert buf.device_status() == want_status
    assert tuple(out.shape) == (N, H)
    csl = _compact(o["slot"])
    m = int((csl >= 0).sum())
    if fp8:
        q, s = oracle.dispatch(xb, csl, m, True)
        y = oracle.dequant_rows(q, s, csl)
    else:
        y = oracle.dispatch(xb, csl, m, False)
    assert np.array_equal(bf16_to_bits(out), oracle.combine(y, csl, wref))

    # split dispatch and combine (FP8 rows of a multiple of 512 channels)
    if fp8 and H % 512 != 0:
        return
    (res, cnt, hs, hook) = buf.low_latency_dispatch(x, idx_d, Tmax, E, use_fp8=fp8, return_recv_hook=True)
    hook()
    assert buf.device_status() == want_status
    assert np.array_equal(cnt.cpu().numpy(), o["tokens_per_expert"])
    rows = valid_rows(o["slot"])
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    g_of = np.nonzero(o["slot"].reshape(-1) >= 0)[0] // K
    if fp8:
        recv, sc = res
        q, s = oracle.quant_token(xb)
        assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[g_of])
        assert np.array_equal(sc[rows_d].cpu().numpy().view(np.uint32), s[g_of].view(np.uint32))
    else:
        assert np.array_equal(bf16_to_bits(res[rows_d]), xb[g_of])
    if N > 0:
        ys = place_rows(o["rows"], H, o["slot"], ye, tokens)
        out, hook = buf.low_latency_combine(ys, None, wd, hs, E, return_recv_hook=True)
        hook()
        assert buf.device_status() == ep.EP_OK
        sl = np.where(o["slot"] >= 0, np.arange(N * K).reshape(N, K), -1).astype(np.int32)
        assert np.array_equal(bf16_to_bits(out), oracle.combine(ye.reshape(-1, H), sl, wref))
