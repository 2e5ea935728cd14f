"""C ABI checks that need no GPU: the library loads, exports every entry point
include/ep.h declares, and rejects bad arguments on the host before touching
the device."""
import ctypes
import os
import re

import pytest

from combine_get_dispatch_02_gb300 import build as epbuild
from combine_get_dispatch_02_gb300 import ep

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ep.h")


@pytest.fixture(scope="module")
def lib():
    epbuild.build()
    return ep.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|ep_status)\s*(ep_\w+)\s*\(", text, re.M)))


def test_header_declares_entry_points():
    assert _declared() == sorted(ep.ENTRY_POINTS)


def _prototypes():
    """{name: (return type, [(parameter type, parameter name)])} of every
    entry point, parsed from the header (comments removed)."""
    text = re.sub(r"/\*.*?\*/", " ", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(const\s+char\s*\*|ep_status)\s*(ep_\w+)\s*\(([^)]*)\)\s*;", text, re.M):
        params = []
        for a in " ".join(m.group(3).split()).split(","):
            a = a.strip()
            name = re.findall(r"(\w+)$", a)[0]
            params.append((a[: -len(name)].replace(" ", ""), name))
        out[m.group(2)] = (m.group(1).replace(" ", ""), params)
    return out


def _ctype_of(ctype: str, name: str):
    """The ctypes type a C parameter must be bound with: device pointers
    (d_*), streams and opaque context / handle pointers pass as void*, host
    out-parameters and structs as typed pointers."""
    base = ctype.replace("const", "")
    stars = base.count("*")
    base = base.replace("*", "")
    scalars = {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64, "uint64_t": ctypes.c_uint64}
    structs = {"ep_config": ep.ep_config, "ep_handle_info": ep.ep_handle_info, "ep_tuning": ep.ep_tuning,
               "ep_tune_record": ep.ep_tune_record, "ep_test_hooks": ep.ep_test_hooks}
    if stars == 0:
        return scalars[base]
    if stars == 2:  # ep_ctx ** / ep_handle **: an opaque pointer written back
        return ctypes.POINTER(ctypes.c_void_p)
    if name.startswith("d_") or base in ("void", "ep_ctx", "ep_handle"):
        return ctypes.c_void_p
    if base in structs:
        return ctypes.POINTER(structs[base])
    return ctypes.POINTER(scalars[base])


def test_binding_signatures_match_header(lib):
    protos = _prototypes()
    assert sorted(protos) == sorted(ep.ENTRY_POINTS)
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.restype == (ctypes.c_char_p if ret.startswith("const") else ctypes.c_int32), name
        want = [_ctype_of(t, n) for t, n in params]
        assert list(fn.argtypes) == want, (name, [n for _, n in params])


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(10):
        assert ep.status_str(s) and ep.status_str(s) != "unknown status"
    assert ep.status_str(99) == "unknown status"


def test_config_limits(lib):
    ok = ep.make_config(32, 128, 7168, 256, 8)
    assert ep.ep_config_check(ok) == ep.EP_OK
    bad = [
        (ep.make_config(0, 128, 7168, 256, 8), ep.EP_ERR_INVALID_ARG),
        (ep.make_config(32, 0, 7168, 256, 8), ep.EP_ERR_INVALID_ARG),
        (ep.make_config(32, 128, 7170, 256, 8), ep.EP_ERR_INVALID_ARG),   # H % 8
        (ep.make_config(32, 128, 7168, 250, 8), ep.EP_ERR_INVALID_ARG),   # E % R
        (ep.make_config(32, 128, 7168, 256, 0), ep.EP_ERR_INVALID_ARG),
        (ep.make_config(32, 128, 7168, 256, 8, layout=5), ep.EP_ERR_INVALID_ARG),
        (ep.make_config(32, 128, 7168, 256, 8, max_sms=-1), ep.EP_ERR_INVALID_ARG),
        (ep.make_config(32, 128, 7168, 256, 33), ep.EP_ERR_UNSUPPORTED),
        (ep.make_config(32, 128, 7168, 2048, 8), ep.EP_ERR_UNSUPPORTED),
        (ep.make_config(64, 128, 7168, 512, 8), ep.EP_ERR_UNSUPPORTED),   # E*R > 16384
        (ep.make_config(32, 1 << 20, 7168, 256, 8), ep.EP_ERR_UNSUPPORTED),  # rows >= 2^31
    ]
    for cfg, want in bad:
        assert ep.ep_config_check(cfg) == want, (cfg.num_ranks, cfg.hidden, cfg.num_experts)
    assert lib.ep_config_check(None) == ep.EP_ERR_INVALID_ARG


def _limits_of_header(R, Tmax, H, E, K, layout, max_sms):
    """The status ep_config_check must give, read off the limits the header
    states for ep_config: a malformed size is INVALID_ARG, a well-formed one
    past the library's limits UNSUPPORTED."""
    if min(R, Tmax, H, E, K) < 1 or max_sms < 0 or layout not in (0, 1):
        return ep.EP_ERR_INVALID_ARG
    if E % R or H % 8:
        return ep.EP_ERR_INVALID_ARG
    if R > 1024 or K > 32 or E > 1024 or H > 65536 or E * R > 16384:
        return ep.EP_ERR_UNSUPPORTED
    rows = E * R * Tmax if layout == 0 else R * Tmax * K
    if rows >= 2**31 or R * Tmax * K >= 2**31:
        return ep.EP_ERR_UNSUPPORTED
    return ep.EP_OK


def test_config_limits_search(lib):
    """Hypothesis walks the edges of every limit (and the 2^31 row bound)."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    def near(*edges):
        return st.one_of([st.integers(e - 2, e + 2) for e in edges] + [st.integers(-3, 2**31 - 1)])

    @hyp.settings(max_examples=600, deadline=None, derandomize=True, database=None)
    @hyp.given(R=near(1, 32, 1024), Tmax=near(1, 128, 1 << 16, 1 << 21), H=near(8, 7168, 65536),
               E=near(1, 256, 1024, 16384), K=near(1, 8, 32), layout=st.integers(-1, 2),
               max_sms=st.integers(-2, 200))
    def check(R, Tmax, H, E, K, layout, max_sms):
        cfg = ep.make_config(R, Tmax, H, E, K, layout=layout, max_sms=max_sms)
        want = _limits_of_header(R, Tmax, H, E, K, layout, max_sms)
        assert ep.ep_config_check(cfg) == want, (R, Tmax, H, E, K, layout, max_sms)
        if want == ep.EP_OK:
            rows = E * R * Tmax if layout == 0 else R * Tmax * K
            assert ep.ep_recv_rows(cfg) == rows

    check()


def test_size_queries(lib):
    cfg = ep.make_config(32, 128, 7168, 256, 8)
    assert ep.ep_recv_rows(cfg) == 256 * 32 * 128
    assert ep.ep_recv_bytes(cfg, True) == (256 * 4096 * 7168, 256 * 4096 * 56 * 4)
    assert ep.ep_recv_bytes(cfg, False) == (256 * 4096 * 7168 * 2, 0)
    packed = ep.make_config(8, 4096, 7168, 256, 8, layout=ep.EP_LAYOUT_PACKED)
    assert ep.ep_recv_rows(packed) == 8 * 4096 * 8
    odd = ep.make_config(4, 32, 200, 32, 4)
    with pytest.raises(ep.EPError) as e:
        ep.ep_recv_bytes(odd, True)  # FP8 needs H % 128 == 0
    assert e.value.status == ep.EP_ERR_UNSUPPORTED


def test_host_rejections_touch_no_device(lib):
    P = ctypes.c_void_p
    # invalid config: rejected before any CUDA call
    out = P(123)
    assert lib.ep_create(ctypes.byref(ep.make_config(0, 1, 8, 1, 1)), ctypes.byref(out)) == ep.EP_ERR_INVALID_ARG
    assert out.value is None
    assert lib.ep_create(None, ctypes.byref(out)) == ep.EP_ERR_INVALID_ARG
    # NULL context / handle
    assert lib.ep_dispatch(None, None, None, 1, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_combine(None, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_get_dispatch_layout(None, None, 0, None, None, None, None, None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_get_device_status(None, None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_destroy(None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_handle_destroy(None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_handle_create(None, ctypes.byref(out)) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_handle_get_info(None, None) == ep.EP_ERR_INVALID_ARG


def test_host_rejections_of_the_range_split_and_tuning_calls(lib):
    """Every entry point added for the round trip, the split calls and the
    launch-shape tuning rejects a NULL context before any CUDA call."""
    P = ctypes.c_void_p
    E = ep.EP_ERR_INVALID_ARG
    assert lib.ep_dispatch_range(None, None, 0, None, 0, 0, None, None, None) == E
    assert lib.ep_combine_range(None, None, None, None, 0, 0, None, None) == E
    assert lib.ep_expert_identity(None, None, 0, None, None, None, 0, 0, None) == E
    assert lib.ep_round_trip(None, None, None, 0, None, 0, None, None, None, None, None, 0, None) == E
    n = ctypes.c_int32(0)
    assert lib.ep_round_trip_auto_chunk(None, 0, 0, ctypes.byref(n)) == E
    assert lib.ep_dispatch_send(None, None, None, 0, 0, None, None, None, None) == E
    assert lib.ep_dispatch_recv(None, None, 0, None, None, None, None, None, 0, None) == E
    assert lib.ep_combine_send(None, None, None, None, 0, None) == E
    assert lib.ep_combine_recv(None, None, None, None, None, None) == E
    t = ep.ep_tuning()
    assert lib.ep_get_tuning(None, ctypes.byref(t)) == E
    assert lib.ep_set_tuning(None, ctypes.byref(t)) == E
    assert lib.ep_autotune(None, None, None, 1, None, 0, None, None, None, None, 1, ctypes.byref(t), None) == E
    assert lib.ep_get_autotune_log(None, None, 0, ctypes.byref(n)) == E
    assert lib.ep_status_str(ep.EP_ERR_TIMEOUT).decode() == "a bounded wait on the device gave up"
    h = ep.ep_test_hooks(-1, 0)
    assert lib.ep_set_test_hooks(None, ctypes.byref(h)) == E


def test_host_rejections_of_the_rank_transport(lib):
    """The rank transport's calls reject a NULL context / handle before any
    CUDA call, and its send-buffer size query answers R*Tmax*min(K, R)."""
    E = ep.EP_ERR_INVALID_ARG
    assert lib.ep_rank_dispatch_send(None, None, None, None, 0, 0, None, None, None, None, None, None) == E
    assert lib.ep_rank_dispatch_recv(None, None, 0, None, None, None, None, None, 0, None, None) == E
    assert lib.ep_rank_combine_send(None, None, None, None, 0, None, None) == E
    assert lib.ep_rank_combine_recv(None, None, None, None, None) == E
    assert lib.ep_rank_runs(None, None, None, None) == E
    for R, Tmax, K in ((8, 4096, 8), (32, 128, 8), (4, 32, 2), (2, 7, 6)):
        cfg = ep.make_config(R, Tmax, 1024, 4 * R, K)
        assert ep.ep_rank_send_rows(cfg) == R * Tmax * min(K, R)


def test_receive_row_counts_match_the_definitions_and_the_oracle(lib):
    """Host-only size queries: padded E·R·Tmax / packed R·Tmax·K rows, and for
    the rank-deduplicated layout R·R·Tmax / R·Tmax·min(K, R) — the same
    numbers the oracle's own (independent) definitions give."""
    import oracle
    for R, Tmax, E, K in [(32, 128, 256, 8), (8, 4096, 256, 8), (4, 32, 32, 4), (16, 512, 64, 6), (2, 8, 4, 4),
                          (8, 100, 16, 12)]:
        for layout in (ep.EP_LAYOUT_PADDED, ep.EP_LAYOUT_PACKED):
            cfg = ep.make_config(R, Tmax, 1024, E, K, layout=layout)
            rows = ep.ep_recv_rows(cfg)
            rank_rows = ep.ep_rank_recv_rows(cfg)
            if layout == ep.EP_LAYOUT_PADDED:
                assert rows == E * R * Tmax and rank_rows == R * R * Tmax
            else:
                assert rows == R * Tmax * K and rank_rows == R * Tmax * min(K, R)
            assert rows == oracle.recv_rows(R, Tmax, E, K, layout)
            assert rank_rows == oracle.rank_recv_rows(R, Tmax, K, layout)


def test_struct_layouts_match_header(tmp_path):
    """The binding's ctypes structures have the sizes and field offsets the C
    compiler gives the header's structs."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("needs gcc")
    structs = {"ep_config": ep.ep_config, "ep_tuning": ep.ep_tuning,
               "ep_tune_record": ep.ep_tune_record, "ep_handle_info": ep.ep_handle_info,
               "ep_test_hooks": ep.ep_test_hooks}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ep.h"', "int main(void) {"]
    for s, cls in structs.items():
        lines.append(f'    printf("{s} size %zu\\n", sizeof({s}));')
        for f, _ in cls._fields_:
            lines.append(f'    printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        s, f, v = line.split()
        got[(s, f)] = int(v)
    for s, cls in structs.items():
        assert got[(s, "size")] == ctypes.sizeof(cls), s
        for f, _ in cls._fields_:
            assert got[(s, f)] == getattr(cls, f).offset, (s, f)


def test_c_program_uses_the_abi(lib, tmp_path):
    """A plain C11 program compiled against include/ep.h and linked with
    libep.so makes the calls that need no GPU (tests/c/abi_host.c)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("needs gcc")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c", "abi_host.c")
    libdir = os.path.dirname(ep._LIB_PATH)
    exe = tmp_path / "abi_host"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER), src,
                    "-L", libdir, "-l:libep.so", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
