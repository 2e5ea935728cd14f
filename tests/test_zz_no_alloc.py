"""ep_dispatch_noalloc, the dispatch for callers that cannot allocate device
memory (inside a capture that must not allocate, under a runtime that owns all
device memory, in a plugin limited to the buffers it is handed): it keeps its
intermediate state in the library's static device array instead of buffers
from cudaMalloc.  Its receive rows, FP8 scales and per-expert counts must be
bit-identical to ep_dispatch's, on two calls in a row with different inputs
(the second call reuses the array the first one left behind).

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl
from helpers import bits_to_bf16, make_buffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    epbuild.build()
    torch.cuda.set_device(0)


def _regular(w, x, idx):
    buf = make_buffer(w)
    recv, sc, cnt, h = None, None, None, None
    out, cnt, h = buf.low_latency_dispatch(x, idx, w.max_tokens_per_rank, w.num_experts, use_fp8=w.use_fp8)
    recv, sc = out if w.use_fp8 else (out, None)
    assert buf.device_status() == ep.EP_OK
    slot = h.tensors()["slot"].view(-1).long()
    return recv, sc, cnt, slot[slot >= 0].clone()


def _noalloc(w, x, idx):
    cfg = ep.make_config(w.num_ranks, w.max_tokens_per_rank, w.hidden, w.num_experts, w.topk,
                         ep.EP_LAYOUT_PADDED if w.layout == wl.PADDED else ep.EP_LAYOUT_PACKED)
    rows = ep.ep_recv_rows(cfg)
    if w.use_fp8:
        recv = torch.empty(rows, w.hidden, dtype=torch.float8_e4m3fn, device="cuda")
        sc = torch.empty(rows, w.hidden // 128, dtype=torch.float32, device="cuda")
    else:
        recv, sc = torch.empty(rows, w.hidden, dtype=torch.bfloat16, device="cuda"), None
    cnt = torch.empty(w.num_experts, dtype=torch.int32, device="cuda")
    ep.ep_dispatch_noalloc(cfg, x, idx, w.tokens_per_rank, w.use_fp8, recv, sc, cnt)
    torch.cuda.synchronize()
    return recv, sc, cnt


def test_noalloc_dispatch_matches_dispatch_on_two_calls():
    cases = [wl.LL, wl.SKEW.with_(layout=wl.PACKED, use_fp8=False)]
    for w in cases:
        d = wl.generate(w)
        x = bits_to_bf16(d["x_bits"])
        idx = torch.from_numpy(wl.inject_masks(d["topk_idx"], 0.05, 3)).cuda()
        ref_recv, ref_sc, ref_cnt, rows = _regular(w, x, idx)
        got_recv, got_sc, got_cnt = _noalloc(w, x, idx)
        assert torch.equal(got_cnt, ref_cnt)
        assert torch.equal(got_recv.view(torch.uint8)[rows], ref_recv.view(torch.uint8)[rows])
        if w.use_fp8:
            assert torch.equal(got_sc[rows], ref_sc[rows])


def test_noalloc_rejects_sizes_beyond_its_limit():
    w = wl.NORMAL  # 262144 entries > 65536
    cfg = ep.make_config(w.num_ranks, w.max_tokens_per_rank, w.hidden, w.num_experts, w.topk,
                         ep.EP_LAYOUT_PACKED)
    x = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(1, dtype=torch.int64, device="cuda")
    recv = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.EPError) as e:
        ep.ep_dispatch_noalloc(cfg, x, idx, w.tokens_per_rank, False, recv, None, None)
    assert e.value.status == ep.EP_ERR_UNSUPPORTED
