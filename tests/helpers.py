"""Test helpers: moving bf16 / e4m3 bit patterns between numpy and torch,
and running the GPU path on a workload through the binding."""
from __future__ import annotations

import numpy as np
import torch

from combine_get_dispatch_02_gb300 import ep
from combine_get_dispatch_02_gb300 import workloads as wl

ORACLE_LAYOUT = {wl.PADDED: 0, wl.PACKED: 1}


def bits_to_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def e4m3_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def make_buffer(w: wl.Workload, max_sms: int = 0):
    from combine_get_dispatch_02_gb300 import Buffer
    return Buffer(w.num_ranks, w.max_tokens_per_rank, w.hidden, w.num_experts, w.topk,
                  low_latency_mode=(w.layout == wl.PADDED), max_sms=max_sms)


def valid_rows(slot: np.ndarray) -> np.ndarray:
    s = slot.reshape(-1)
    return s[s >= 0]


def place_rows(rows: int, H: int, slot: np.ndarray, y_entry: np.ndarray, tokens: np.ndarray,
               fill_bits: int = 0xFFFF) -> torch.Tensor:
    """Receive-layout bf16 tensor on the GPU: row slot[g, k] holds y_entry[i, k]
    for the i-th token g of ``tokens``; every other row holds ``fill_bits``
    (a NaN by default, so reading a row that received nothing shows up)."""
    y = torch.full((rows, H), fill_bits - 65536 if fill_bits >= 32768 else fill_bits,
                   dtype=torch.int16, device="cuda").view(torch.bfloat16)
    sl = slot[tokens]                      # [n, K]
    m = sl >= 0
    dst = torch.from_numpy(sl[m].astype(np.int64)).cuda()
    src = bits_to_bf16(y_entry[m])         # [cnt, H]
    y.index_copy_(0, dst, src)
    return y
