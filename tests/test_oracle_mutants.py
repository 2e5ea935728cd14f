"""The pins catch plausible mistakes: each case plants one mistake in a copy of
the oracle's C source (on the CPU), builds it, binds the oracle module to it
and checks that at least one pin of test_oracle_pins fails."""
import os
import shutil

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")

MUTANTS = {
    "combine: product rounded before the add": (
        "acc = fmaf(wk, orc_bf16_to_f32(y[s * H + c]), acc);",
        "acc = acc + wk * orc_bf16_to_f32(y[s * H + c]);"),
    "combine: k summed in descending order": (
        "            for (int k = 0; k < K; k++) {\n                int64_t s = slot[g * K + k];\n"
        "                if (s < 0)\n                    continue;\n                float wk",
        "            for (int k = K - 1; k >= 0; k--) {\n                int64_t s = slot[g * K + k];\n"
        "                if (s < 0)\n                    continue;\n                float wk"),
    "combine: bf16 by truncation": (
        "out[g * H + c] = orc_f32_to_bf16(acc);",
        "out[g * H + c] = (uint16_t)(f32_bits(acc) >> 16);"),
    "fp8: no floor on amax": (
        "float amax_c = amax < 1e-4f ? 1e-4f : amax;",
        "float amax_c = amax;"),
    "fp8: inverse taken from the rounded scale": (
        "float inv = 448.0f / amax_c;",
        "float inv = 1.0f / s;"),
    "fp8: amax over the first 64 channels only": (
        "    for (int i = 0; i < 128; i++) {\n        float a = fabsf",
        "    for (int i = 0; i < 64; i++) {\n        float a = fabsf"),
    "e4m3: ties rounded up": (
        "pick = (c & 1) ? c + 1 : c;",
        "pick = c + 1;"),
    "e4m3: overflow to NaN instead of saturating": (
        "    if (ax >= 448.0)\n        return (uint8_t)(sign | 0x7E);",
        "    if (ax >= 448.0)\n        return (uint8_t)(sign | 0x7F);"),
    "e4m3: subnormal step 2^-10": (
        "v = ldexp((double)m / 8.0, -6);",
        "v = ldexp((double)m / 8.0, -7);"),
    "bf16: ties rounded up": (
        "pick = (lo & 1u) ? hi : lo;",
        "pick = hi;"),
    "layout: rows ordered k-major": (
        "    for (int64_t g = 0; g < N; g++) {\n        for (int k = 0; k < K; k++) {\n"
        "            int64_t e = topk_idx[g * K + k];\n            if (e < 0 || e >= E) {",
        "    for (int k = 0; k < K; k++) {\n        for (int64_t g = 0; g < N; g++) {\n"
        "            int64_t e = topk_idx[g * K + k];\n            if (e < 0 || e >= E) {"),
    "layout: inclusive prefix for packed bases": (
        "            base[e] = acc;\n            acc += tokens_per_expert[e];",
        "            acc += tokens_per_expert[e];\n            base[e] = acc;"),
    "layout: expert owner e mod R": (
        "if (e >= 0 && e < E && e / L == d)",
        "if (e >= 0 && e < E && e % R == d)"),
    "layout: off_er inclusive": (
        "            off_er[e * R + r] = run;\n            run += cnt_er[e * R + r];",
        "            run += cnt_er[e * R + r];\n            off_er[e * R + r] = run;"),
    "layout: padded buffers sized by T instead of Tmax": (
        "base[e] = (int64_t)e * R * Tmax;",
        "base[e] = (int64_t)e * R * T;"),
    "layout: invalid ids not reported": (
        "                bad++;\n",
        ""),
    "rank layout: every entry carries its token": (
        "            if (!first)\n                continue;\n            int64_t row = rbase[d] + fill[d];",
        "            int64_t row = rbase[d] + fill[d];"),
    "rank layout: weights of other ranks' experts kept": (
        "recv_topk_w[row * K + k2] = on_d ? (w ? w[g * K + k2] : 1.0f) : 0.0f;",
        "recv_topk_w[row * K + k2] = w ? w[g * K + k2] : 1.0f;"),
    "rank layout: rank buffers sized by T instead of Tmax": (
        "rbase[d] = layout == ORC_LAYOUT_PADDED ? (int64_t)d * R * Tmax : acc;",
        "rbase[d] = layout == ORC_LAYOUT_PADDED ? (int64_t)d * R * T : acc;"),
    "identity expert: scale of the wrong block": (
        "float v = orc_e4m3_to_f32(q[s * H + c]) * scales[s * (H / 128) + c / 128];",
        "float v = orc_e4m3_to_f32(q[s * H + c]) * scales[s * (H / 128)];"),
    "layout: padded overflow not dropped": (
        "            if (layout == ORC_LAYOUT_PADDED && pos >= cap) {",
        "            if (0) {"),
    "layout: padded counts not capped": (
        "tokens_per_expert[e] = (int32_t)cap;",
        "tokens_per_expert[e] = tokens_per_expert[e];"),
    "layout: source rank taken as g mod R": (
        "int r = (int)(g / T);",
        "int r = (int)(g % R);"),
    "layout: tokens per rank counts entries": (
        "hit = 1;",
        "hit += 1;"),
    "fp8: scale from a rounded 1/448": (
        "float s = amax_c / 448.0f;",
        "float s = amax_c * (1.0f / 448.0f);"),
    "fp8: amax of signed values": (
        "float a = fabsf(orc_bf16_to_f32(x[i]));",
        "float a = orc_bf16_to_f32(x[i]);"),
    "fp8 dispatch: scales written to the source token's row": (
        "orc_quant_token(xg, H, (uint8_t *)recv + s * H, scales + s * (H / 128));",
        "orc_quant_token(xg, H, (uint8_t *)recv + s * H, scales + g * (H / 128));"),
    "combine: NULL weights read as 0": (
        "float wk = w ? w[g * K + k] : 1.0f;",
        "float wk = w ? w[g * K + k] : 0.0f;"),
    "rank runs: send offsets in destination-major order": (
        "    for (int r = 0; r < R; r++)\n        for (int d = 0; d < R; d++) {\n            send_off[r * R + d] = acc;",
        "    for (int d = 0; d < R; d++)\n        for (int r = 0; r < R; r++) {\n            send_off[r * R + d] = acc;"),
    "rank runs: receive offsets without the rank's base": (
        "int64_t run = rbase[d];",
        "int64_t run = 0;"),
    "rank runs: every entry on a rank gets a send row": (
        "                        break; /* later k on d are not carrying entries */\n",
        ""),
    "rank runs: tokens in descending order within a run": (
        "            for (int t = 0; t < T; t++) {\n                int64_t g = (int64_t)r * T + t;",
        "            for (int t = T - 1; t >= 0; t--) {\n                int64_t g = (int64_t)r * T + t;"),
}


def _pins():
    cheap = [pins.test_layout_golden, pins.test_fp8_golden_blocks, pins.test_combine_golden,
             pins.test_e4m3_definition_values, pins.test_e4m3_saturates,
             pins.test_fp8_zero_block_uses_floor, pins.test_e4m3_every_midpoint_ties_to_even,
             pins.test_e4m3_decode_matches_torch, pins.test_combine_special_cases]
    for f in cheap:
        yield f.__name__, (lambda f=f: f(oracle))
    yield "rank_golden", lambda: pins.test_rank_layout_golden(oracle)
    yield "rank_runs_golden", lambda: pins.test_rank_runs_golden(oracle)
    for seed in range(10):
        yield f"rank_runs_brute_force[{seed}]", (lambda seed=seed: pins.test_rank_runs_brute_force(oracle, seed))
    for seed in range(30):
        yield f"brute_force[{seed}]", (lambda seed=seed: pins.test_layout_brute_force(oracle, seed))
    for seed in range(20):
        yield f"rank_brute_force[{seed}]", (lambda seed=seed: pins.test_rank_layout_brute_force(oracle, seed))
    for name in ("tiny", "skew"):
        yield f"invariants[{name}]", (lambda name=name: pins.test_layout_invariants(oracle, name))
    yield "dequant", lambda: pins.test_dequant_rows_golden_and_bound(oracle)
    yield "bf16_torch", lambda: pins.test_bf16_matches_torch(oracle)
    yield "fp8_torch", lambda: pins.test_fp8_matches_torch_cast_of_products(oracle)
    yield "e4m3_torch", lambda: pins.test_e4m3_encode_matches_torch(oracle)
    for seed in range(4):
        yield f"exact_rational[{seed}]", (lambda seed=seed: pins.test_combine_exact_rational(oracle, seed))
    yield "round_trip_bf16", lambda: pins.test_round_trip_bf16(oracle)
    yield "round_trip_fp8", lambda: pins.test_round_trip_fp8(oracle)


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    d = tmp_path_factory.mktemp("mutants")
    yield d
    oracle.use_library(None)
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_mutant(name, workdir):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation site not found (oracle source changed?)"
    idx = list(MUTANTS).index(name)
    src = os.path.join(workdir, f"m{idx}.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    lib = oracle.compile_source(src, os.path.join(workdir, f"m{idx}.so"))
    oracle.use_library(lib)
    try:
        caught = None
        for pin_name, run in _pins():
            try:
                run()
            except AssertionError:
                caught = pin_name
                break
        assert caught is not None, f"no pin caught: {name}"
    finally:
        oracle.use_library(None)
