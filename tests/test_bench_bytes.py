"""The byte accounting behind the bench's roofline fractions, pinned to
values worked out by hand from the operation definitions (CPU only)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from combine_get_dispatch_02_gb300 import workloads as wl  # noqa: E402


def _mb(b):
    return round(b / 1e6, 1)


def test_low_latency_bytes():
    # N = 4096 tokens, K = 8, H = 7168, M = 32768 received rows, FP8 payload
    N, K, H, M, E, R = 4096, 8, 7168, 32768, 256, 32
    disp, disp_kernel, comb = bench._algorithmic_bytes(wl.LL, M)
    # read x once, topk_idx, write each row's codes and scales, slots, src_info, (e, r) counts
    assert disp == N * H * 2 + N * K * 8 + M * H + M * (H // 128) * 4 + N * K * 4 + M * 4 + E * R * 4
    assert _mb(disp) == 301.5
    assert disp_kernel == N * H * 2 + M * H + M * (H // 128) * 4 + N * K * 4
    # read each received row, weights and slots, write the combined tokens
    assert comb == M * H * 2 + 2 * N * K * 4 + N * H * 2
    assert _mb(comb) == 528.7


@pytest.mark.parametrize("fp8,dispatch_mb", [(False, 4232.1), (True, 2411.7)])
def test_normal_bytes(fp8, dispatch_mb):
    disp, _, comb = bench._algorithmic_bytes(wl.NORMAL.with_(use_fp8=fp8), 262144)
    assert _mb(disp) == dispatch_mb
    assert _mb(comb) == 4230.0


def test_skew_and_identity_bytes():
    disp, _, comb = bench._algorithmic_bytes(wl.SKEW, 49152)
    assert (_mb(disp), _mb(comb)) == (275.5, 470.2)
    # identity expert at ll: read codes + scales, write bf16 rows, read slots
    assert bench._identity_bytes(wl.LL, 32768) == 32768 * (7168 + 56 * 4) + 32768 * 7168 * 2 + 4096 * 8 * 4


def test_peak_lookup(tmp_path):
    """The roofline denominator: the measured copy bandwidth when the file
    holds one (as a number or an object with a burst figure), else the
    fallback, which is said."""
    p = tmp_path / "peaks.json"
    assert bench._peaks(str(p)) == (bench.FALLBACK_HBM_GBS, "fallback")
    p.write_text('{"hbm_gbs": 7012.5, "bf16_tflops": 1900}')
    assert bench._peaks(str(p)) == (7012.5, "measured")
    p.write_text('{"hbm_gbs": {"burst": 7100, "sustained": 6900}}')
    assert bench._peaks(str(p)) == (7100.0, "measured")
    for bad in ('{"hbm_gbs": null}', '{"hbm_gbs": "n/a"}', "not json", "[1, 2]", '{"hbm_gbs": 0}'):
        p.write_text(bad)
        assert bench._peaks(str(p)) == (bench.FALLBACK_HBM_GBS, "fallback")
