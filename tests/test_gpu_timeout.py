"""The row mover's bounded waits run out on the GPU without a fault: a
test-only switch (ep_set_test_hooks) makes the copy kernel never issue one
row's load, so its barrier phase never completes and the wait gives up after
1 ms.  ep_get_device_status must then report EP_ERR_TIMEOUT (not the
in-flight form: no load was outstanding for that row, and the others were
waited for), and the same context must work afterwards, bit for bit against
the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import ORACLE_LAYOUT, bf16_to_bits, bits_to_bf16, e4m3_to_bits, make_buffer, place_rows, valid_rows

pytestmark = pytest.mark.gpu

WAIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    oracle.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("withhold", [0, 5, 127])
def test_dispatch_hook_wait_runs_out_then_recovers(withhold):
    w = wl.TINY.with_(use_fp8=True, x_scale="loguniform")
    d = wl.generate(w)
    N, H = w.num_tokens, w.hidden
    buf = make_buffer(w)
    h = buf.new_handle()
    x = bits_to_bf16(d["x_bits"])
    send_x = torch.empty(N, H, dtype=torch.float8_e4m3fn, device="cuda")
    send_sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
    ep.ep_dispatch_send(buf.ctx, x, torch.from_numpy(d["topk_idx"]).cuda(), w.tokens_per_rank, True, h.raw,
                        send_x, send_sc)
    recv, sc = buf.alloc_recv(True)
    assert buf.device_status() == ep.EP_OK

    ep.ep_set_test_hooks(buf.ctx, move_withhold_item=withhold, move_wait_ns=WAIT_NS)
    ep.ep_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None, 4)
    assert buf.device_status() == ep.EP_ERR_TIMEOUT
    assert buf.device_status() == ep.EP_OK  # read and cleared

    ep.ep_set_test_hooks(buf.ctx)  # back to the defaults
    ep.ep_dispatch_recv(buf.ctx, h.raw, True, send_x, send_sc, recv, sc, None, 4)
    assert buf.device_status() == ep.EP_OK
    o = oracle.layout(d["topk_idx"], w.num_experts, w.max_tokens_per_rank, ORACLE_LAYOUT[w.layout])
    rows = valid_rows(o["slot"])
    q, s = oracle.dispatch(d["x_bits"].reshape(N, H), o["slot"], o["rows"], True)
    rows_d = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert np.array_equal(e4m3_to_bits(recv.view(torch.uint8)[rows_d]), q[rows])
    assert np.array_equal(sc[rows_d].cpu().numpy().view(np.uint32), s[rows].view(np.uint32))


def test_combine_send_wait_runs_out_then_recovers():
    w = wl.TINY
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    buf = make_buffer(w)
    h = buf.new_handle()
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    ep.ep_get_dispatch_layout(buf.ctx, idx, w.tokens_per_rank, None, None, None, h.raw)
    slot = h.tensors()["slot"].cpu().numpy()
    ye = wl.expert_outputs(w)
    y = place_rows(buf.rows, H, slot, ye, np.arange(N))
    send_y = torch.empty(N * K, H, dtype=torch.bfloat16, device="cuda")
    ep.ep_set_test_hooks(buf.ctx, move_withhold_item=N * K - 1, move_wait_ns=WAIT_NS)
    ep.ep_combine_send(buf.ctx, h.raw, y, send_y, 2)
    assert buf.device_status() == ep.EP_ERR_TIMEOUT
    ep.ep_set_test_hooks(buf.ctx)
    ep.ep_combine_send(buf.ctx, h.raw, y, send_y, 2)
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    wts = torch.from_numpy(d["topk_weights"].reshape(N, K)).cuda()
    ep.ep_combine_recv(buf.ctx, h.raw, send_y, wts, out)
    assert buf.device_status() == ep.EP_OK
    m = slot.reshape(-1) >= 0
    slot_c = np.full(N * K, -1, np.int32)
    slot_c[m] = np.arange(int(m.sum()), dtype=np.int32)
    ref = oracle.combine(ye.reshape(N * K, H)[m], slot_c.reshape(N, K), d["topk_weights"].reshape(N, K))
    assert np.array_equal(bf16_to_bits(out), ref)


def test_test_hooks_reject_out_of_range():
    w = wl.TINY
    buf = make_buffer(w)
    for bad in ((-2, 0), (0, -1), (0, 10_000_000_001)):
        with pytest.raises(ep.EPError) as e:
            ep.ep_set_test_hooks(buf.ctx, *bad)
        assert e.value.status == ep.EP_ERR_INVALID_ARG
