"""Pins for the CPU oracle: checks against things other than the oracle itself.

* number formats: torch's bf16 / float8_e4m3fn casts and decodes (library
  routines), the values the OCP E4M3FN definition fixes, and every rounding
  midpoint between adjacent codes;
* layout: hand-derived golden case, brute force on tiny routings with numpy's
  stable argsort and bincount, invariants on larger ones;
* FP8 cast: hand-derived golden blocks, the closed-form error bound, power-of-
  two scaling invariance, torch's cast on the same products;
* combine: hand-derived golden cases (fused multiply-add, ascending k, masks),
  exact rational arithmetic with one binary32 rounding per step;
* round trip: combine(identity(dispatch(x))) with weights summing to one.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from combine_get_dispatch_02_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_to_bf16_float(b):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _torch_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ formats

def test_e4m3_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_definition_values(orc):
    # values fixed by the OCP E4M3FN definition
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x77: 240.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for c, v in fixed.items():
        assert orc.e4m3_to_f32(np.array([c], np.uint8))[0] == v
        assert orc.f32_to_e4m3(np.array([v], np.float32))[0] == c
    neg0 = orc.f32_to_e4m3(np.array([-0.0], np.float32))[0]
    assert neg0 == 0x80


def test_e4m3_every_midpoint_ties_to_even(orc):
    vals = orc.e4m3_to_f32(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in binary32
        below = np.nextafter(mid, np.float32(-np.inf))
        above = np.nextafter(mid, np.float32(np.inf))
        got = orc.f32_to_e4m3(np.array([lo, below, mid, above, -mid], np.float32))
        even = c if c % 2 == 0 else c + 1
        assert list(got) == [c, c, even, c + 1, 0x80 | even], hex(c)


def test_e4m3_saturates(orc):
    big = np.array([448.0, 449.0, 463.99, 464.0, 465.0, 1e6, np.inf, -1e30, -np.inf], np.float32)
    got = orc.f32_to_e4m3(big)
    assert list(got) == [0x7E] * 7 + [0xFE] * 2


def test_e4m3_encode_matches_torch(orc):
    rng = np.random.default_rng(7)
    mag = np.exp(rng.uniform(np.log(1e-4), np.log(448.0), 200_000)).astype(np.float32)
    x = np.where(rng.random(mag.size) < 0.5, -mag, mag).astype(np.float32)
    x[:5] = [0.0, 2.0 ** -10, 2.0 ** -9, 3 * 2.0 ** -10, 447.9]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.f32_to_e4m3(x), ref)


def test_bf16_matches_torch(orc):
    rng = np.random.default_rng(8)
    bits = rng.integers(0, 2 ** 32, 400_000, dtype=np.uint64).astype(np.uint32)
    # halfway cases (low half exactly 0x8000) with odd and even upper halves
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, np.array([3.4028235e38, -3.4028235e38, 1e-45, -0.0, 0.0], np.float32)])
    assert np.array_equal(orc.f32_to_bf16(x), _torch_bf16_bits(x))
    b = rng.integers(0, 2 ** 16, 10_000, dtype=np.uint16)
    ours = orc.bf16_to_f32(b)
    ref = _bits_to_bf16_float(b)
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin].view(np.uint32), ref[fin].view(np.uint32))


# ------------------------------------------------------------------ layout

def _read_golden(name):
    out, cases, cur = {}, [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "y": []}
                cases.append(cur)
            elif cur is not None:
                if key == "y":
                    cur["y"].append([float(Fraction(v)) for v in vals])
                else:
                    cur[key] = vals
            else:
                out.setdefault(key, []).append(vals)
    return out, cases


def test_layout_golden(orc):
    g, _ = _read_golden("layout_small.txt")
    iv = lambda k: np.array([int(v) for v in g[k][0]])
    R, T, Tmax, K, E = (int(g[k][0][0]) for k in ("R", "T", "Tmax", "K", "E"))
    idx = iv("topk_idx").reshape(R, T, K)
    for lay, pfx in ((orc.LAYOUT_PADDED, "padded"), (orc.LAYOUT_PACKED, "packed")):
        o = orc.layout(idx, E, Tmax, lay)
        assert o["n_bad"] == 0
        assert np.array_equal(o["cnt_er"].ravel(), iv("cnt_er"))
        assert np.array_equal(o["off_er"].ravel(), iv("off_er"))
        assert np.array_equal(o["tokens_per_expert"], iv("tokens_per_expert"))
        assert np.array_equal(o["tokens_per_rank"], iv("tokens_per_rank"))
        assert np.array_equal(o["is_token_in_rank"].ravel(), iv("is_token_in_rank"))
        assert np.array_equal(o["base"], iv(pfx + "_base"))
        assert np.array_equal(o["slot"].ravel(), iv(pfx + "_slot"))
    o = orc.layout(idx, E, Tmax, orc.LAYOUT_PACKED)
    assert np.array_equal(o["src_info"][:7], iv("packed_src_info"))


def _brute_layout(idx, E, Tmax, packed):
    """Layout by enumeration: numpy stable argsort of the flattened expert
    ids gives each expert's rows in (token, k) order; bincount gives counts."""
    R, T, K = idx.shape
    L = E // R
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E)
    base = np.concatenate([[0], np.cumsum(counts)[:-1]]) if packed else np.arange(E) * R * Tmax
    cap = flat.size if packed else R * Tmax
    slot = np.full(flat.size, -1, np.int64)
    order = np.argsort(np.where(valid, flat, E), kind="stable")
    pos_in_expert = {}
    overflow = 0
    for j in order:
        if not valid[j]:
            continue
        e = flat[j]
        p = pos_in_expert.get(e, 0)
        pos_in_expert[e] = p + 1
        if p >= cap:
            overflow += 1
        else:
            slot[j] = base[e] + p
    src = np.arange(flat.size).reshape(R * T, K)
    cnt_er = np.zeros((E, R), int)
    in_rank = np.zeros((R * T, R), int)
    for g in range(R * T):
        for k in range(K):
            e = flat[g * K + k]
            if 0 <= e < E:
                cnt_er[e, g // T] += 1
                in_rank[g, e // L] = 1
    return dict(counts=np.minimum(counts, cap), base=base, slot=slot.reshape(R * T, K),
                src=src, cnt_er=cnt_er, in_rank=in_rank, overflow=overflow,
                n_bad=int(((flat < -1) | (flat >= E)).sum()))


@pytest.mark.parametrize("seed", range(60))
def test_layout_brute_force(orc, seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 4))
    L = int(rng.integers(1, 3))
    E = R * L
    Tmax = int(rng.integers(1, 5))
    T = int(rng.integers(1, Tmax + 1))
    K = int(rng.integers(1, 4))
    idx = rng.integers(-1, E, size=(R, T, K))  # duplicates and -1 allowed
    if seed % 5 == 0:  # invalid ids are counted and skipped
        idx.reshape(-1)[rng.integers(0, idx.size)] = E + int(rng.integers(0, 3))
    for packed in (False, True):
        lay = orc.LAYOUT_PACKED if packed else orc.LAYOUT_PADDED
        o = orc.layout(idx, E, Tmax, lay)
        b = _brute_layout(idx, E, Tmax, packed)
        assert o["n_bad"] == b["n_bad"]
        assert o["n_overflow"] == b["overflow"]
        assert np.array_equal(o["tokens_per_expert"], b["counts"])
        assert np.array_equal(o["base"], b["base"])
        assert np.array_equal(o["slot"], b["slot"])
        assert np.array_equal(o["cnt_er"], b["cnt_er"])
        assert np.array_equal(o["is_token_in_rank"], b["in_rank"])
        assert np.array_equal(o["tokens_per_rank"], b["in_rank"].sum(0))
        v = b["slot"] >= 0
        assert np.array_equal(o["src_info"][b["slot"][v]], b["src"][v])


def test_rank_layout_golden(orc):
    g, _ = _read_golden("layout_small.txt")
    iv = lambda k: np.array([int(v) for v in g[k][0]])
    R, T, Tmax, K, E = (int(g[k][0][0]) for k in ("R", "T", "Tmax", "K", "E"))
    idx = iv("topk_idx").reshape(R, T, K)
    for lay, pfx in ((orc.LAYOUT_PACKED, "rank_packed"), (orc.LAYOUT_PADDED, "rank_padded")):
        o = orc.rank_layout(idx, None, E, Tmax, lay)
        assert np.array_equal(o["tokens_per_rank"], iv("rank_tokens_per_rank"))
        assert np.array_equal(o["rbase"], iv(pfx + "_rbase"))
        assert np.array_equal(o["rank_slot"].ravel(), iv(pfx + "_slot"))
    o = orc.rank_layout(idx, None, E, Tmax, orc.LAYOUT_PACKED)
    assert np.array_equal(o["recv_topk_idx"][:5].ravel(), iv("rank_packed_recv_topk_idx"))
    assert np.array_equal(o["src_info"][:5], iv("rank_packed_src_info"))


@pytest.mark.parametrize("seed", range(40))
def test_rank_layout_brute_force(orc, seed):
    rng = np.random.default_rng(700 + seed)
    R = int(rng.integers(1, 4))
    L = int(rng.integers(1, 4))
    E = R * L
    Tmax = int(rng.integers(1, 5))
    T = int(rng.integers(1, Tmax + 1))
    K = int(rng.integers(1, 5))
    idx = rng.integers(-1, E, size=(R, T, K))
    w = rng.random((R, T, K)).astype(np.float32)
    N = R * T
    flat = idx.reshape(N, K)
    for packed in (False, True):
        lay = orc.LAYOUT_PACKED if packed else orc.LAYOUT_PADDED
        o = orc.rank_layout(idx, w, E, Tmax, lay)
        # enumerate (token, rank) pairs: the carrying k is the first on that rank
        carry = {}
        for gg in range(N):
            for k in range(K):
                e = flat[gg, k]
                if 0 <= e < E and (gg, e // L) not in carry:
                    carry[(gg, e // L)] = k
        counts = np.bincount([d for (_, d) in carry], minlength=R)
        rbase = np.concatenate([[0], np.cumsum(counts)[:-1]]) if packed else np.arange(R) * R * Tmax
        assert np.array_equal(o["tokens_per_rank"], counts)
        assert np.array_equal(o["rbase"], rbase)
        slot = np.full((N, K), -1)
        for d in range(R):
            toks = sorted(gg for (gg, dd) in carry if dd == d)
            for j, gg in enumerate(toks):
                row = rbase[d] + j
                slot[gg, carry[(gg, d)]] = row
                assert o["src_info"][row] == gg * K + carry[(gg, d)]
                for k in range(K):
                    e = flat[gg, k]
                    on_d = 0 <= e < E and e // L == d
                    assert o["recv_topk_idx"][row, k] == (e - d * L if on_d else -1)
                    assert o["recv_topk_weights"][row, k] == (w.reshape(N, K)[gg, k] if on_d else 0.0)
        assert np.array_equal(o["rank_slot"], slot)
        # the same tokens per rank as the expert layout's membership
        assert np.array_equal(o["tokens_per_rank"], orc.layout(idx, E, Tmax, lay)["tokens_per_rank"])


def test_rank_runs_golden(orc):
    g, _ = _read_golden("layout_small.txt")
    iv = lambda k: np.array([int(v) for v in g[k][0]])
    R, T, Tmax, K, E = (int(g[k][0][0]) for k in ("R", "T", "Tmax", "K", "E"))
    idx = iv("topk_idx").reshape(R, T, K)
    for lay, pfx in ((orc.LAYOUT_PACKED, "rank_packed"), (orc.LAYOUT_PADDED, "rank_padded")):
        o = orc.rank_layout(idx, None, E, Tmax, lay)
        r = orc.rank_runs(idx, E, o["rbase"])
        assert np.array_equal(r["run_cnt"].ravel(), iv("rank_run_cnt"))
        assert np.array_equal(r["send_off"].ravel(), iv("rank_send_off"))
        assert np.array_equal(r["send_slot"].ravel(), iv("rank_send_slot"))
        assert np.array_equal(r["recv_off"].ravel(), iv(pfx + "_recv_off"))
        assert r["send_rows"] == int(iv("rank_run_cnt").sum())


@pytest.mark.parametrize("seed", range(40))
def test_rank_runs_brute_force(orc, seed):
    """Send rows by enumeration (carried (token, rank) pairs sorted by source
    rank, destination rank, token), and the run copies checked end to end:
    copying every run from the send buffer to its receive rows puts each
    token where the rank layout says."""
    rng = np.random.default_rng(900 + seed)
    R = int(rng.integers(1, 5))
    L = int(rng.integers(1, 4))
    E = R * L
    Tmax = int(rng.integers(1, 6))
    T = int(rng.integers(0, Tmax + 1))
    K = int(rng.integers(1, 6))
    idx = rng.integers(-1, E, size=(R, T, K))
    N = R * T
    flat = idx.reshape(N, K)
    carry = {}
    for gg in range(N):
        for k in range(K):
            e = flat[gg, k]
            if 0 <= e < E and (gg, e // L) not in carry:
                carry[(gg, e // L)] = k
    pairs = sorted(carry, key=lambda p: (p[0] // max(T, 1), p[1], p[0]))  # (r, d, t)
    cnt = np.zeros((R, R), np.int64)
    for gg, d in pairs:
        cnt[gg // T, d] += 1
    send_off = np.concatenate([[0], np.cumsum(cnt.ravel())[:-1]]).reshape(R, R)
    slot = np.full((N, K), -1)
    for row, (gg, d) in enumerate(pairs):
        slot[gg, carry[(gg, d)]] = row
    for lay in (orc.LAYOUT_PACKED, orc.LAYOUT_PADDED):
        o = orc.rank_layout(idx, None, E, Tmax, lay)
        r = orc.rank_runs(idx, E, o["rbase"])
        recv_off = o["rbase"][None, :] + np.concatenate([np.zeros((1, R), np.int64), np.cumsum(cnt, 0)[:-1]], 0)
        assert np.array_equal(r["run_cnt"], cnt)
        assert np.array_equal(r["send_off"], send_off)
        assert np.array_equal(r["recv_off"], recv_off)
        assert np.array_equal(r["send_slot"], slot)
        assert r["send_rows"] == len(pairs)
        # the copies: a token id per send row, moved run by run
        send = np.full(max(len(pairs), 1), -1)
        m = slot >= 0
        send[slot[m]] = np.nonzero(m)[0]
        recv = np.full(o["rows"], -1)
        for a in range(R):
            for d in range(R):
                n = cnt[a, d]
                recv[recv_off[a, d]:recv_off[a, d] + n] = send[send_off[a, d]:send_off[a, d] + n]
        rs = o["rank_slot"]
        assert np.array_equal(m, rs >= 0)
        assert np.array_equal(recv[rs[m]], np.nonzero(m)[0])


def test_rank_runs_carry_bytes(orc):
    """BF16 rows dispatched into the send order and copied run by run equal
    the rank layout's own dispatch, bit for bit (ragged T, masked entries)."""
    w = wl.NORMAL.with_(tokens_per_rank=37, max_tokens_per_rank=40, hidden=256)
    d = wl.generate(w)
    idx = wl.inject_masks(d["topk_idx"], 0.1, 4)
    x = d["x_bits"].reshape(w.num_tokens, w.hidden)
    o = orc.rank_layout(idx, None, w.num_experts, w.max_tokens_per_rank)
    r = orc.rank_runs(idx, w.num_experts, o["rbase"])
    send = orc.dispatch(x, r["send_slot"], r["send_rows"], use_fp8=False)
    recv = np.zeros((o["rows"], w.hidden), np.uint16)
    R = w.num_ranks
    for a in range(R):
        for dd in range(R):
            n = r["run_cnt"][a, dd]
            so, ro = r["send_off"][a, dd], r["recv_off"][a, dd]
            recv[ro:ro + n] = send[so:so + n]
    assert np.array_equal(recv, orc.dispatch(x, o["rank_slot"], o["rows"], use_fp8=False))


def test_rank_round_trip_bf16(orc):
    """Rank dispatch, an identity expert per rank that returns the token times
    the sum of its local weights, rank combine: weights summing to one give x
    back within two bf16 roundings."""
    w = wl.NORMAL.with_(tokens_per_rank=64, max_tokens_per_rank=64, hidden=256)
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    o = orc.rank_layout(d["topk_idx"], d["topk_weights"], w.num_experts, w.max_tokens_per_rank)
    x = d["x_bits"].reshape(N, H)
    recv = orc.dispatch(x, o["rank_slot"], o["rows"], use_fp8=False)
    used = o["rank_slot"][o["rank_slot"] >= 0]
    scale = o["recv_topk_weights"][used].sum(axis=1, dtype=np.float64)
    y = np.zeros((o["rows"], H), np.uint16)
    y[used] = _torch_bf16_bits((orc.bf16_to_f32(recv[used]) * scale[:, None]).astype(np.float32))
    out = orc.combine(y, o["rank_slot"], None)
    xf = _bits_to_bf16_float(x).astype(np.float64)
    of = _bits_to_bf16_float(out).astype(np.float64)
    nr = (o["rank_slot"] >= 0).sum(axis=1)[:, None]
    assert np.all(np.abs(of - xf) <= (nr + 2) * _ulp_bf16(xf))


def test_layout_identity_case(orc):
    idx = np.zeros((1, 9, 1), np.int64)  # R = 1, E = 1, K = 1
    for lay in (orc.LAYOUT_PADDED, orc.LAYOUT_PACKED):
        o = orc.layout(idx, 1, 9, lay)
        assert np.array_equal(o["slot"].ravel(), np.arange(9))
        assert np.array_equal(o["src_info"], np.arange(9))


@pytest.mark.parametrize("name", ["tiny", "skew"])
def test_layout_invariants(orc, name):
    w = wl.WORKLOADS[name]
    idx = wl.generate(w)["topk_idx"] if name == "tiny" else wl.inject_masks(
        wl.generate(w.with_(hidden=128))["topk_idx"], 0.05, 3)
    R, T, K = idx.shape
    E = w.num_experts
    for lay in (orc.LAYOUT_PADDED, orc.LAYOUT_PACKED):
        o = orc.layout(idx, E, w.max_tokens_per_rank, lay)
        slot = o["slot"].ravel()
        valid = idx.ravel() >= 0
        M = int(valid.sum())
        assert o["tokens_per_expert"].sum() == M == o["cnt_er"].sum()
        assert np.all(slot[~valid] == -1)
        s = slot[valid]
        assert len(np.unique(s)) == M  # every entry has its own row
        assert np.array_equal(o["src_info"][s], np.nonzero(valid)[0])
        for e in range(E):  # rows of an expert: contiguous from base, ascending (g, k)
            rows = np.sort(s[idx.ravel()[valid] == e])
            assert np.array_equal(rows, o["base"][e] + np.arange(len(rows)))
            assert np.all(np.diff(o["src_info"][rows]) > 0)
        assert np.array_equal(o["tokens_per_rank"], o["is_token_in_rank"].sum(0))
        if lay == orc.LAYOUT_PADDED:
            assert np.all(o["tokens_per_expert"] <= R * w.max_tokens_per_rank)


# ------------------------------------------------------------------ FP8 cast

def test_fp8_golden_blocks(orc):
    _, _ = _read_golden("fp8_block.txt")
    lines = [l.split("#", 1)[0].split() for l in open(os.path.join(GOLDEN, "fp8_block.txt"))]
    lines = [l for l in lines if l]
    i = 0
    n = 0
    while i < len(lines):
        assert lines[i][0] == "block"
        x = np.zeros(128, np.float32)
        vals = [float(Fraction(v)) for v in lines[i][1:]]
        x[:len(vals)] = vals
        qx = [int(h, 16) for h in lines[i + 1][1:]]
        sc = float(Fraction(lines[i + 2][1]))
        xb = _torch_bf16_bits(x)
        assert np.array_equal(_bits_to_bf16_float(xb), x)  # inputs are bf16-exact
        q, s = orc.quant_token(xb[None, :])
        assert list(q[0, :len(qx)]) == qx
        assert np.all(q[0, len(qx):] == 0)
        assert s[0, 0] == sc
        i += 3
        n += 1
    assert n == 3


def test_dequant_rows_golden_and_bound(orc):
    # codes of the first golden FP8 block at scale 2^-7: 448 -> 3.5, -224 -> -1.75, 56 -> 0.4375
    q = np.zeros((2, 128), np.uint8)
    q[1, :3] = [0x7E, 0xF6, 0x66]
    sc = np.array([[1.0], [0.0078125]], np.float32)
    y = orc.dequant_rows(q, sc, np.array([[1, -1]], np.int32))
    assert list(_bits_to_bf16_float(y[1, :4])) == [3.5, -1.75, 0.4375, 0.0]
    assert np.all(y[0] == 0)  # a row no entry received is left alone
    # dequantised rows are within the FP8 bound of the token they came from
    rng = np.random.default_rng(15)
    x = _random_tokens(rng, 16, 512)
    qq, ss = orc.quant_token(x)
    yy = orc.dequant_rows(qq, ss, np.arange(16, dtype=np.int32).reshape(16, 1))
    xf = _bits_to_bf16_float(x).astype(np.float64)
    s_full = np.repeat(ss, 128, axis=1).astype(np.float64)
    bound = (2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * s_full) * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(xf) * 1.07
    assert np.all(np.abs(_bits_to_bf16_float(yy).astype(np.float64) - xf) <= bound)


def test_fp8_zero_block_uses_floor(orc):
    q, s = orc.quant_token(np.zeros((1, 256), np.uint16))
    assert np.all(q == 0)
    assert s[0, 0] == np.float32(1e-4) / np.float32(448.0)


def _random_tokens(rng, n, H, spread=True):
    x = rng.standard_normal((n, H)).astype(np.float32)
    if spread:
        x *= (10.0 ** rng.uniform(-2, 2, (n, 1))).astype(np.float32)
    return _torch_bf16_bits(x)


def test_fp8_matches_torch_cast_of_products(orc):
    rng = np.random.default_rng(11)
    xb = _random_tokens(rng, 64, 1024)
    q, s = orc.quant_token(xb)
    x = torch.from_numpy(_bits_to_bf16_float(xb)).reshape(64, 8, 128)
    amax = x.abs().amax(-1, keepdim=True).clamp_min(torch.tensor(1e-4, dtype=torch.float32))
    inv = torch.tensor(448.0) / amax
    ref_q = (x * inv).to(torch.float8_e4m3fn).view(torch.uint8).reshape(64, 1024).numpy()
    ref_s = (amax / torch.tensor(448.0)).reshape(64, 8).numpy()
    assert np.array_equal(q, ref_q)
    assert np.array_equal(s.view(np.uint32), ref_s.view(np.uint32))


def test_fp8_error_bound(orc):
    rng = np.random.default_rng(12)
    xb = _random_tokens(rng, 128, 2048)
    q, s = orc.quant_token(xb)
    x = _bits_to_bf16_float(xb).astype(np.float64)
    deq = orc.e4m3_to_f32(q).astype(np.float64) * np.repeat(s, 128, axis=1)
    # 3 mantissa bits: half-ulp 2^-4 relative in the normal range, half of the
    # 2^-9 subnormal step (times the scale) below it, plus binary32 rounding
    bound = 2.0 ** -4 * np.abs(x) + np.repeat(s, 128, axis=1) * 2.0 ** -10 + 2.0 ** -22 * np.abs(x)
    assert np.all(np.abs(deq - x) <= bound)


def test_fp8_power_of_two_scaling(orc):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((16, 512)).astype(np.float32)
    xb = _torch_bf16_bits(x)
    q0, s0 = orc.quant_token(xb)
    for j in (-3, 5):
        xj = _torch_bf16_bits(_bits_to_bf16_float(xb) * np.float32(2.0 ** j))
        qj, sj = orc.quant_token(xj)
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj, s0 * np.float32(2.0 ** j))


# ------------------------------------------------------------------ combine

def test_combine_golden(orc):
    _, cases = _read_golden("combine_small.txt")
    assert len(cases) == 5
    for c in cases:
        y = _torch_bf16_bits(np.array(c["y"], np.float32))
        assert np.array_equal(_bits_to_bf16_float(y), np.array(c["y"], np.float32))
        slot = np.array([[int(v) for v in c["slot"]]], np.int32)
        w = np.array([[float(Fraction(v)) for v in c["w"]]], np.float32)
        assert np.array_equal(w.astype(np.float64), np.array([[float(Fraction(v)) for v in c["w"]]]))
        out = orc.combine(y, slot, w)
        assert [f"{v:04X}" for v in out[0]] == [v.upper() for v in c["out"]], c["name"]


def _round_to_f32(q: Fraction) -> Fraction:
    """Nearest binary32 to an exact rational, ties to even (no overflow)."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    n, r = divmod(a, ulp)
    if r * 2 > ulp or (r * 2 == ulp and n % 2 == 1):
        n += 1
    return sign * n * ulp


@pytest.mark.parametrize("seed", range(12))
def test_combine_exact_rational(orc, seed):
    rng = np.random.default_rng(300 + seed)
    N, K, H, rows = 3, int(rng.integers(1, 9)), 16, 12
    y = _random_tokens(rng, rows, H)
    slot = rng.integers(-1, rows, size=(N, K)).astype(np.int32)
    w = rng.random((N, K)).astype(np.float32) * np.float32(2.0) - np.float32(0.5)
    use_w = seed % 3 != 0
    out = orc.combine(y, slot, w if use_w else None)
    yf = _bits_to_bf16_float(y)
    ref = np.zeros((N, H), np.float32)
    for g in range(N):
        for c in range(H):
            acc = Fraction(0)
            for k in range(K):
                if slot[g, k] < 0:
                    continue
                wk = Fraction(float(w[g, k])) if use_w else Fraction(1)
                acc = _round_to_f32(wk * Fraction(float(yf[slot[g, k], c])) + acc)
            ref[g, c] = float(acc)
    assert np.array_equal(out, _torch_bf16_bits(ref))


def test_combine_special_cases(orc):
    rng = np.random.default_rng(14)
    y = _random_tokens(rng, 40, 256)
    slot = rng.permutation(40)[:32].reshape(8, 4).astype(np.int32)
    # K = 1, weight 1: a pure gather
    assert np.array_equal(orc.combine(y, slot[:, :1], np.ones((8, 1), np.float32)), y[slot[:, 0]])
    # one-hot weights: a copy of the selected expert row
    w = np.zeros((8, 4), np.float32)
    w[np.arange(8), np.arange(8) % 4] = 1.0
    out = orc.combine(y, slot, w)
    assert np.array_equal(out, y[slot[np.arange(8), np.arange(8) % 4]])
    # no weights: a plain sum
    sum_ref = np.zeros((8, 256), np.float32)
    yf = _bits_to_bf16_float(y)
    for k in range(4):
        sum_ref = sum_ref + yf[slot[:, k]]
    assert np.array_equal(orc.combine(y, slot, None), _torch_bf16_bits(sum_ref))


# ------------------------------------------------------------------ round trip

def _ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def test_round_trip_bf16(orc):
    w = wl.TINY
    d = wl.generate(w)
    lay = orc.layout(d["topk_idx"], w.num_experts, w.max_tokens_per_rank)
    x = d["x_bits"].reshape(w.num_tokens, w.hidden)
    recv = orc.dispatch(x, lay["slot"], lay["rows"], use_fp8=False)
    out = orc.combine(recv, lay["slot"], d["topk_weights"].reshape(w.num_tokens, -1))
    xf = _bits_to_bf16_float(x).astype(np.float64)
    of = _bits_to_bf16_float(out).astype(np.float64)
    assert np.all(np.abs(of - xf) <= _ulp_bf16(xf))


def test_round_trip_fp8(orc):
    w = wl.TINY.with_(use_fp8=True, x_scale="loguniform")
    d = wl.generate(w)
    lay = orc.layout(d["topk_idx"], w.num_experts, w.max_tokens_per_rank)
    x = d["x_bits"].reshape(w.num_tokens, w.hidden)
    q, s = orc.dispatch(x, lay["slot"], lay["rows"], use_fp8=True)
    # identity expert: dequantise each received row and return it in bf16
    used = lay["slot"][lay["slot"] >= 0]
    y = np.zeros((lay["rows"], w.hidden), np.uint16)
    deq = orc.e4m3_to_f32(q[used]) * np.repeat(s[used], 128, axis=1)
    y[used] = orc.f32_to_bf16(deq.astype(np.float32))
    out = orc.combine(y, lay["slot"], d["topk_weights"].reshape(w.num_tokens, -1))
    xf = _bits_to_bf16_float(x).astype(np.float64)
    of = _bits_to_bf16_float(out).astype(np.float64)
    scale = np.repeat(orc.quant_token(x)[1], 128, axis=1).astype(np.float64)
    K = w.topk
    bound = (2.0 ** -4 * np.abs(xf) + 2.0 ** -10 * scale) * (1 + 2.0 ** -8) \
        + 2.0 ** -8 * np.abs(xf) * (1 + 2.0 ** -4) + 2.0 ** -8 * np.abs(of) \
        + K * 2.0 ** -22 * np.abs(xf)
    assert np.all(np.abs(of - xf) <= bound)
