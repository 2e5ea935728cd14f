"""Property search over the oracle's shapes (CPU only).

The seeded brute-force pins sample routings at a few fixed shapes; these
tests let hypothesis search the shape edge cases as well: one rank, one
expert per rank, no tokens on a rank, more choices per token than experts,
every entry masked, ids below -1 or past the last expert.  Expected values
come from enumeration and exact arithmetic, never from the oracle itself.

Sources: "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南" (cyqw.cn),
section 核心API示例 (dispatch and combine from topk_idx / topk_weights) and
section 性能调优 (fixed-size receive buffers); the layout readings are the
oracle's (expert e on rank e / (E/R), one expert's rows in (token, k) order,
combine as the weighted sum over a token's top-k in ascending k)."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")

from hypothesis import HealthCheck, given, settings  # noqa: E402

import oracle  # noqa: E402
import test_oracle_mutants as mutants  # noqa: E402
import test_oracle_pins as pins  # noqa: E402

# derandomized and without an example database: the same search every run
SETTINGS = settings(max_examples=150, deadline=None, derandomize=True, database=None,
                    suppress_health_check=[HealthCheck.function_scoped_fixture])


@st.composite
def routing(draw, max_ranks=4, max_local=3, max_tmax=5, max_k=6):
    """(topk_idx [R, T, K], E, Tmax): T may be 0 and K may exceed E; ids are
    drawn from [-3, E+2] so masked (-1) and invalid entries both appear."""
    R = draw(st.integers(1, max_ranks))
    L = draw(st.integers(1, max_local))
    E = R * L
    Tmax = draw(st.integers(1, max_tmax))
    T = draw(st.integers(0, Tmax))
    K = draw(st.integers(1, max_k))
    n = R * T * K
    mode = draw(st.sampled_from(["mixed", "valid", "masked", "one_expert"]))
    if mode == "valid":
        ids = draw(st.lists(st.integers(0, E - 1), min_size=n, max_size=n))
    elif mode == "masked":
        ids = [-1] * n
    elif mode == "one_expert":  # every entry on one expert: its buffer fills first
        e = draw(st.integers(0, E - 1))
        ids = [e] * n
    else:
        ids = draw(st.lists(st.integers(-3, E + 2), min_size=n, max_size=n))
    return np.array(ids, np.int64).reshape(R, T, K), E, Tmax


@SETTINGS
@given(case=routing(), packed=st.booleans())
def test_layout_matches_enumeration(orc, case, packed):
    idx, E, Tmax = case
    o = orc.layout(idx, E, Tmax, orc.LAYOUT_PACKED if packed else orc.LAYOUT_PADDED)
    b = pins._brute_layout(idx, E, Tmax, packed)
    assert o["n_bad"] == b["n_bad"]
    assert o["n_overflow"] == b["overflow"]
    assert np.array_equal(o["tokens_per_expert"], b["counts"])
    assert np.array_equal(o["base"], b["base"])
    assert np.array_equal(o["slot"], b["slot"])
    assert np.array_equal(o["cnt_er"], b["cnt_er"])
    assert np.array_equal(o["is_token_in_rank"], b["in_rank"])
    assert np.array_equal(o["tokens_per_rank"], b["in_rank"].sum(0))
    # the exclusive prefix of the (expert, source rank) counts
    cnt = b["cnt_er"]
    assert np.array_equal(o["off_er"], np.cumsum(cnt, axis=1) - cnt)
    v = b["slot"] >= 0
    assert np.array_equal(o["src_info"][b["slot"][v]], b["src"][v])
    # rows nobody writes keep -1, and no row is written twice
    written = np.zeros(o["rows"], bool)
    written[b["slot"][v]] = True
    assert (o["src_info"][~written] == -1).all()
    assert np.unique(b["slot"][v]).size == int(v.sum())


@SETTINGS
@given(case=routing(), packed=st.booleans())
def test_rank_layout_matches_enumeration(orc, case, packed):
    idx, E, Tmax = case
    R, T, K = idx.shape
    L = E // R
    N = R * T
    flat = idx.reshape(N, K)
    w = (np.arange(N * K, dtype=np.float32).reshape(R, T, K) + 1) / 8
    o = orc.rank_layout(idx, w, E, Tmax, orc.LAYOUT_PACKED if packed else orc.LAYOUT_PADDED)
    carry = {}  # (token, destination rank) -> the first choice on that rank
    for g in range(N):
        for k in range(K):
            e = int(flat[g, k])
            if 0 <= e < E and (g, e // L) not in carry:
                carry[(g, e // L)] = k
    counts = np.bincount([d for (_, d) in carry], minlength=R)
    rbase = np.concatenate([[0], np.cumsum(counts)[:-1]]) if packed else np.arange(R) * R * Tmax
    assert np.array_equal(o["tokens_per_rank"], counts)
    assert np.array_equal(o["rbase"], rbase)
    slot = np.full((N, K), -1)
    for d in range(R):
        for j, g in enumerate(sorted(g for (g, dd) in carry if dd == d)):
            row = rbase[d] + j
            slot[g, carry[(g, d)]] = row
            assert o["src_info"][row] == g * K + carry[(g, d)]
            for k in range(K):
                e = int(flat[g, k])
                on_d = 0 <= e < E and e // L == d
                assert o["recv_topk_idx"][row, k] == (e - d * L if on_d else -1)
                assert o["recv_topk_weights"][row, k] == (w.reshape(N, K)[g, k] if on_d else 0)
    assert np.array_equal(o["rank_slot"], slot)


def _bf16_exact(v):
    """bf16 bits of an fp32-exact value (round to nearest even)."""
    t = torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@SETTINGS
@given(case=routing(max_k=5), packed=st.booleans(), data=st.data())
def test_bf16_round_trip_exact(orc, case, packed, data):
    """Dispatch of BF16 rows, the identity expert, then the weighted combine.
    Tokens are +-m * 2^s with an 8-bit m, weights are powers of two: every
    partial sum is exact in fp32, so each output is the bf16 rounding of the
    exact rational sum over the token's rows that landed."""
    idx, E, Tmax = case
    R, T, K = idx.shape
    N, H = R * T, 128
    lay = orc.LAYOUT_PACKED if packed else orc.LAYOUT_PADDED
    o = orc.layout(idx, E, Tmax, lay)
    seed = data.draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    m = rng.integers(128, 256, size=(N, H)) * rng.choice([-1, 1], size=(N, H))
    s = rng.integers(-6, 4, size=(N, H))
    x = (m * np.exp2(s - 7)).astype(np.float32)
    wexp = rng.integers(-3, 4, size=(N, K))
    w = np.exp2(wexp).astype(np.float32)
    recv = orc.dispatch(_bf16_exact(x), o["slot"], o["rows"], False)
    out = orc.combine(recv, o["slot"], w)
    for g in range(N):
        acc = [Fraction(0)] * H
        for k in range(K):
            if o["slot"][g, k] >= 0:
                acc = [a + Fraction(float(w[g, k])) * Fraction(float(xv)) for a, xv in zip(acc, x[g])]
        exact = np.array([float(a) for a in acc], np.float64)
        assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
        assert np.array_equal(out[g], _bf16_exact(exact))


# Mistakes planted in a copy of the oracle's C source that the searches above
# must find on their own, with no seeded pin's help.  (The two combine
# mutants that only change rounding order are left to the seeded pins: with
# exact partial sums the order cannot show.)
SEARCH_MUTANTS = {
    "combine: bf16 by truncation": "round_trip",
    "layout: rows ordered k-major": "layout",
    "layout: inclusive prefix for packed bases": "layout",
    "layout: expert owner e mod R": "layout",
    "layout: off_er inclusive": "layout",
    "layout: padded buffers sized by T instead of Tmax": "layout",
    "layout: invalid ids not reported": "layout",
    "layout: padded overflow not dropped": "layout",
    "layout: padded counts not capped": "layout",
    "layout: source rank taken as g mod R": "layout",
    "layout: tokens per rank counts entries": "layout",
    "rank layout: every entry carries its token": "rank_layout",
    "rank layout: weights of other ranks' experts kept": "rank_layout",
    "rank layout: rank buffers sized by T instead of Tmax": "rank_layout",
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    yield tmp_path_factory.mktemp("search_mutants")
    oracle.use_library(None)


@pytest.mark.parametrize("name", list(SEARCH_MUTANTS))
def test_search_finds_mutant(orc, name, mutant_dir):
    old, new = mutants.MUTANTS[name]
    text = open(mutants.SRC).read()
    assert text.count(old) == 1, "mutation site not found (oracle source changed?)"
    stem = f"s{list(SEARCH_MUTANTS).index(name)}"
    src = os.path.join(mutant_dir, stem + ".c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    oracle.use_library(oracle.compile_source(src, os.path.join(mutant_dir, stem + ".so")))
    prop = {"layout": test_layout_matches_enumeration,
            "rank_layout": test_rank_layout_matches_enumeration,
            "round_trip": test_bf16_round_trip_exact}[SEARCH_MUTANTS[name]]
    try:
        with pytest.raises(AssertionError):
            prop(orc)
    finally:
        oracle.use_library(None)
