"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments before touching the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkg():
    from tests.buildlib import ensure_built
    ensure_built()
    import selective_state_space_123_b300 as m
    return m


def _declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "ssm_scan.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_]+)\s*\(", hdr)))


def test_exports_every_declared_symbol(pkg):
    declared = _declared_symbols()
    assert set(declared) == set(pkg.EXPORTS), declared
    raw = ctypes.CDLL(pkg.LIB_PATH)
    for name in declared:
        assert hasattr(raw, name), name


def _declared_param_counts():
    hdr = open(os.path.join(ROOT, "include", "ssm_scan.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(ssm_[a-z_]+)\s*\(([^)]*)\)\s*;", hdr):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_header(pkg):
    """Every function the binding calls is declared with as many parameters
    in ssm_scan.h as the binding passes (a miscount would shift every later
    argument)."""
    counts = _declared_param_counts()
    assert set(counts) == set(pkg.EXPORTS)
    for name, n in counts.items():
        argtypes = getattr(pkg.lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes and len(argtypes))


def test_strerror_covers_codes(pkg):
    for code in range(-9, 1):
        s = pkg.ssm_strerror(code)
        assert s and s != "unknown status"
    assert pkg.ssm_strerror(-99) == "unknown status"


def _call_fwd(pkg, shape, ptrs=None, ws_bytes=1 << 20, ws=0x10000):
    p = dict(u=0x1000, dr=0x2000, A=0x3000, B=0x4000, C=0x5000, D=None, z=None, bias=None,
             h0=None, y=0x6000, hL=None)
    if ptrs:
        p.update(ptrs)
    V = lambda x: None if x is None else ctypes.c_void_p(x)
    return pkg.lib.ssm_scan_fwd(ctypes.byref(shape) if shape is not None else None,
                                V(p["u"]), V(p["dr"]), V(p["A"]), V(p["B"]), V(p["C"]),
                                V(p["D"]), V(p["z"]), V(p["bias"]), V(p["h0"]), V(p["y"]),
                                V(p["hL"]), V(ws), ws_bytes, None)


def test_fwd_argument_errors(pkg):
    S = lambda **k: pkg.make_shape(k.get("b", 2), k.get("d", 8), k.get("n", 16), k.get("l", 64),
                                   k.get("ti", 1), k.get("to", 0))
    assert _call_fwd(pkg, None) == pkg.SSM_ERR_NULL
    assert _call_fwd(pkg, S(n=0)) == pkg.SSM_ERR_SHAPE
    assert _call_fwd(pkg, S(n=65)) == pkg.SSM_ERR_SHAPE
    assert _call_fwd(pkg, S(b=-1)) == pkg.SSM_ERR_SHAPE
    assert _call_fwd(pkg, S(l=-5)) == pkg.SSM_ERR_SHAPE
    assert _call_fwd(pkg, S(ti=7)) == pkg.SSM_ERR_DTYPE
    assert _call_fwd(pkg, S(to=-1)) == pkg.SSM_ERR_DTYPE
    assert _call_fwd(pkg, S(b=1 << 40, d=1 << 40)) == pkg.SSM_ERR_SHAPE
    assert _call_fwd(pkg, S(), {"u": None}) == pkg.SSM_ERR_NULL
    assert _call_fwd(pkg, S(), {"A": None}) == pkg.SSM_ERR_NULL
    assert _call_fwd(pkg, S(), {"y": None}) == pkg.SSM_ERR_NULL
    assert _call_fwd(pkg, S(), {"B": 0x4008}) == pkg.SSM_ERR_ALIGN
    assert _call_fwd(pkg, S(), {"hL": 0x7004}) == pkg.SSM_ERR_ALIGN
    assert _call_fwd(pkg, S(), ws=None) == pkg.SSM_ERR_WORKSPACE
    assert _call_fwd(pkg, S(), ws_bytes=16) == pkg.SSM_ERR_WORKSPACE
    # nothing to do: empty batch or no channels succeed without touching the GPU
    assert _call_fwd(pkg, S(b=0), {"u": None, "y": None}) == pkg.SSM_OK
    assert _call_fwd(pkg, S(d=0), {"u": None, "y": None}) == pkg.SSM_OK


def _call_fwd_conv(pkg, shape, conv_w=0x8000, conv_k=4, ws_bytes=1 << 24, ws=0x10000):
    V = lambda x: None if x is None else ctypes.c_void_p(x)
    return pkg.lib.ssm_scan_fwd_conv(ctypes.byref(shape), V(0x1000), V(conv_w), None, conv_k,
                                     V(0x2000), V(0x3000), V(0x4000), V(0x5000), None, None, None,
                                     None, V(0x6000), None, V(ws), ws_bytes, None)


def test_fwd_conv_argument_errors(pkg):
    """The conv entry point refuses what it does not build before any GPU work."""
    S = lambda n=16, l=64, ti=1: pkg.make_shape(2, 8, n, l, ti, 0)
    assert _call_fwd_conv(pkg, S(), conv_w=None) == pkg.SSM_ERR_NULL
    assert _call_fwd_conv(pkg, S(), conv_k=0) == pkg.SSM_ERR_SHAPE
    assert _call_fwd_conv(pkg, S(), conv_k=5) == pkg.SSM_ERR_SHAPE
    assert _call_fwd_conv(pkg, S(), conv_w=0x8004) == pkg.SSM_ERR_ALIGN
    # built for 9..16 states and 16-byte token rows
    assert _call_fwd_conv(pkg, S(n=32)) == pkg.SSM_ERR_UNSUPPORTED
    assert _call_fwd_conv(pkg, S(n=4)) == pkg.SSM_ERR_UNSUPPORTED
    assert _call_fwd_conv(pkg, S(l=63)) == pkg.SSM_ERR_UNSUPPORTED
    assert _call_fwd_conv(pkg, S(l=62, ti=0)) == pkg.SSM_ERR_UNSUPPORTED


def _call_fwd_varlen(pkg, shape, cu=0x9000, nseq=3, conv_w=None, conv_k=0, ws_bytes=1 << 24):
    V = lambda x: None if x is None else ctypes.c_void_p(x)
    return pkg.lib.ssm_scan_fwd_varlen(ctypes.byref(shape), V(0x1000), V(cu), nseq, V(conv_w), None,
                                       conv_k, V(0x2000), V(0x3000), V(0x4000), V(0x5000), None,
                                       None, None, None, V(0x6000), None, V(0x10000), ws_bytes, None)


def test_fwd_varlen_argument_errors(pkg):
    """The packed-sequence entry point refuses what it does not build before
    any GPU work."""
    S = lambda n=16, l=64, ti=1: pkg.make_shape(2, 8, n, l, ti, 0)
    assert _call_fwd_varlen(pkg, S(), cu=None) == pkg.SSM_ERR_NULL
    assert _call_fwd_varlen(pkg, S(), nseq=0) == pkg.SSM_ERR_SHAPE
    assert _call_fwd_varlen(pkg, S(), conv_w=0x8000, conv_k=5) == pkg.SSM_ERR_SHAPE
    assert _call_fwd_varlen(pkg, S(), cu=0x9002) == pkg.SSM_ERR_ALIGN
    assert _call_fwd_varlen(pkg, S(n=32)) == pkg.SSM_ERR_UNSUPPORTED
    assert _call_fwd_varlen(pkg, S(l=60)) == pkg.SSM_ERR_UNSUPPORTED
    assert _call_fwd_varlen(pkg, S(), ws_bytes=16) == pkg.SSM_ERR_WORKSPACE
    assert pkg.lib.ssm_strerror(pkg.SSM_ERR_SEQLENS).startswith(b"packed-sequence")


def test_fwd_bidir_argument_errors(pkg):
    """The bidirectional entry point refuses what it does not build before
    any GPU work; its workspace holds the second pass's fp32 output."""
    V = lambda x: None if x is None else ctypes.c_void_p(x)

    def call(shape, A_r=0x3100, B_r=0x4100, ws_bytes=1 << 26):
        return pkg.lib.ssm_scan_fwd_bidir(
            ctypes.byref(shape), V(0x1000), None, V(0x2000), V(0x3000), V(0x4000), V(0x5000),
            None, None, None, V(0x2100), V(A_r), V(B_r), V(0x5100), None, None, None,
            V(0x6000), None, None, V(0x10000), ws_bytes, None)
    S = lambda n=16, l=64, ti=1: pkg.make_shape(2, 8, n, l, ti, 0)
    assert call(S(), A_r=None) == pkg.SSM_ERR_NULL
    assert call(S(), B_r=None) == pkg.SSM_ERR_NULL
    assert call(S(), B_r=0x4108) == pkg.SSM_ERR_ALIGN
    assert call(S(n=32)) == pkg.SSM_ERR_UNSUPPORTED
    assert call(S(l=60)) == pkg.SSM_ERR_UNSUPPORTED
    assert call(S(), ws_bytes=1024) == pkg.SSM_ERR_WORKSPACE
    big = pkg.make_shape(4, 4096, 16, 4096, 1, 1)
    extra = pkg.ssm_scan_workspace_bytes(big, 2) - pkg.ssm_scan_workspace_bytes(big, False)
    assert extra >= 4 * 4096 * 4096 * 4 + 4 * 4096 * 32 * 4


def test_workspace_query(pkg):
    ok = pkg.make_shape(4, 4096, 16, 4096, 1, 1)
    n = pkg.ssm_scan_workspace_bytes(ok)
    # header + prepared B/C (batch * L * 2 * 16 fp32)
    assert n >= 256 + 4 * 4096 * 32 * 4
    assert pkg.ssm_scan_workspace_bytes(pkg.make_shape(1, 1, 0, 1, 1, 1)) == 0
    assert pkg.ssm_scan_workspace_bytes(pkg.make_shape(1, 1, 4, 1, 5, 1)) == 0
    # a million-length sequence with few channels takes the segmented plan
    long = pkg.make_shape(1, 1536, 16, 1 << 20, 1, 1)
    assert pkg.ssm_scan_workspace_bytes(long) > 256 + (1 << 20) * 32 * 4


def test_step_argument_errors(pkg):
    V = ctypes.c_void_p
    f = pkg.lib.ssm_scan_step
    args = [V(0x1000), V(0x2000), V(0x3000), V(0x4000), V(0x5000), None, None, None, V(0x6000),
            V(0x7000), None, None]
    assert f(2, 8, 0, 1, 1, *args) == pkg.SSM_ERR_SHAPE
    assert f(2, 8, 16, 3, 1, *args) == pkg.SSM_ERR_DTYPE
    assert f(0, 8, 16, 1, 1, *args) == pkg.SSM_OK
    bad = list(args); bad[0] = None
    assert f(2, 8, 16, 1, 1, *bad) == pkg.SSM_ERR_NULL
    bad = list(args); bad[8] = V(0x6004)
    assert f(2, 8, 16, 1, 1, *bad) == pkg.SSM_ERR_ALIGN
    bad = list(args); bad[10] = V(0x8002)   # the status word needs 4-byte alignment only
    assert f(2, 8, 16, 1, 1, *bad) == pkg.SSM_ERR_ALIGN


def test_noalloc_scratch_size_matches_header(pkg):
    """The binding's copy of the no-alloc scratch size is the header's macro."""
    import re
    with open(os.path.join(ROOT, "include", "ssm_scan.h")) as f:
        m = re.search(r"#define\s+SSM_NOALLOC_SCRATCH_BYTES\s+(\d+)", f.read())
    assert m is not None
    assert int(m.group(1)) == pkg.NOALLOC_SCRATCH_BYTES


def test_status_and_debug_argument_errors(pkg):
    assert pkg.lib.ssm_get_status(None, None) == pkg.SSM_ERR_NULL
    assert pkg.lib.ssm_debug_expired_wait(None, 256, 10, None) == pkg.SSM_ERR_NULL
    assert pkg.lib.ssm_debug_expired_wait(ctypes.c_void_p(0x1000), 8, 10, None) == pkg.SSM_ERR_WORKSPACE
    assert pkg.lib.ssm_debug_expired_wait(ctypes.c_void_p(0x1008), 256, 10, None) == pkg.SSM_ERR_ALIGN


def test_binding_refuses_cpu_tensors(pkg):
    import torch
    u = torch.zeros(1, 2, 8)
    A, Bm = torch.zeros(2, 4), torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        pkg.ssm_scan_fwd(u, u, A, Bm, Bm)
    with pytest.raises(ValueError):
        pkg.ssm_scan_fwd_conv(u, torch.zeros(2, 4), None, u, A, Bm, Bm)
    with pytest.raises(ValueError):
        pkg.ssm_scan_fwd_varlen(u, torch.tensor([0, 8], dtype=torch.int32), u, A, Bm, Bm)
    d = dict(delta_raw=u, A=A, B=Bm, C=Bm)
    with pytest.raises(ValueError):
        pkg.ssm_scan_fwd_bidir(u, None, d, d)


def _call_bwd(pkg, shape, ptrs=None, ws_bytes=1 << 30, ws=0x10000):
    p = dict(u=0x1000, dr=0x2000, A=0x3000, B=0x4000, C=0x5000, D=None, z=None, bias=None,
             h0=None, dy=0x6000, dhL=None, du=0x7000, ddr=0x8000, dA=0x9000, dB=0xa000,
             dC=0xb000, dD=None, dz=None, dbias=None, dh0=None)
    if ptrs:
        p.update(ptrs)
    V = lambda x: None if x is None else ctypes.c_void_p(x)
    order = ("u", "dr", "A", "B", "C", "D", "z", "bias", "h0", "dy", "dhL", "du", "ddr", "dA",
             "dB", "dC", "dD", "dz", "dbias", "dh0")
    return pkg.lib.ssm_scan_bwd(ctypes.byref(shape) if shape is not None else None,
                                *[V(p[k]) for k in order], V(ws), ws_bytes, None)


def test_bwd_argument_errors(pkg):
    S = lambda **k: pkg.make_shape(k.get("b", 2), k.get("d", 8), k.get("n", 16), k.get("l", 64),
                                   k.get("ti", 1), k.get("to", 0))
    assert _call_bwd(pkg, None) == pkg.SSM_ERR_NULL
    assert _call_bwd(pkg, S(n=0)) == pkg.SSM_ERR_SHAPE
    assert _call_bwd(pkg, S(n=65)) == pkg.SSM_ERR_SHAPE
    assert _call_bwd(pkg, S(ti=2)) == pkg.SSM_ERR_DTYPE
    for name in ("u", "dr", "A", "B", "C", "dy", "du", "ddr", "dA", "dB", "dC"):
        assert _call_bwd(pkg, S(), {name: None}) == pkg.SSM_ERR_NULL, name
    for name in ("u", "dy", "dB", "dz", "dh0", "dhL"):
        assert _call_bwd(pkg, S(), {name: 0x20004}) == pkg.SSM_ERR_ALIGN, name
    assert _call_bwd(pkg, S(), ws=None) == pkg.SSM_ERR_WORKSPACE
    assert _call_bwd(pkg, S(), ws_bytes=1024) == pkg.SSM_ERR_WORKSPACE


def test_bwd_workspace_query(pkg):
    s = pkg.make_shape(2, 5120, 16, 8192, 1, 1)
    n = pkg.ssm_scan_workspace_bytes(s, True)
    # header + prepared B/C + one fp32 number per (batch, channel, token) + final state
    assert n >= 256 + 2 * 8192 * 32 * 4 + 2 * 5120 * 8192 * 4 + 2 * 5120 * 16 * 4
    # small state sizes are padded to 8 in the backward
    assert pkg.ssm_scan_workspace_bytes(pkg.make_shape(1, 4, 4, 64, 0, 0), True) >= \
        256 + 64 * 16 * 4 + 4 * 64 * 4


@pytest.mark.parametrize("for_backward", [False, True])
def test_workspace_query_edge_shapes(pkg, for_backward):
    """The host planner handles every edge shape (no GPU involved)."""
    for sh in [(1, 8, 16, 0), (0, 8, 16, 64), (2, 0, 16, 64), (1, 1, 1, 1), (1, 1, 64, 1),
               (3, 1000, 5, 63), (1, 7, 16, 1 << 20), (1, 1536, 16, 1 << 20),
               (65535, 1, 16, 8), (1, 100000, 16, 64)]:
        for ti in (0, 1):
            n = pkg.ssm_scan_workspace_bytes(pkg.make_shape(*sh, ti, ti), for_backward)
            assert n >= 256, sh
    for var in ("SSM_FWD_NSEG", "SSM_BWD_NSEG"):
        for forced in ("1", "2", "3", "7", "1000"):
            os.environ[var] = forced
            try:
                for sh in [(1, 8, 16, 0), (1, 8, 16, 1), (2, 40, 16, 64 * 29 + 13)]:
                    for ti in (0, 1):
                        n = pkg.ssm_scan_workspace_bytes(pkg.make_shape(*sh, ti, ti), for_backward)
                        assert n >= 256, (var, forced, sh)
            finally:
                del os.environ[var]


def test_backward_segments_enlarge_the_workspace(pkg, monkeypatch):
    """A segmented backward plan (forced, or the planner's for a few-channel
    long sequence) adds its per-segment buffers after the whole-row ones."""
    sh = pkg.make_shape(1, 48, 16, 64 * 40, 1, 1)
    monkeypatch.setenv("SSM_BWD_NSEG", "1")
    whole = pkg.ssm_scan_workspace_bytes(sh, True)
    monkeypatch.setenv("SSM_BWD_NSEG", "4")
    seg4 = pkg.ssm_scan_workspace_bytes(sh, True)
    # initial states, end states, adjoint sums and inputs, tangent sums:
    # 6 arrays of (nseg, batch, dim, 16) fp32 at least
    assert seg4 >= whole + 6 * 4 * 48 * 16 * 4
    monkeypatch.delenv("SSM_BWD_NSEG")
    assert pkg.ssm_scan_workspace_bytes(pkg.make_shape(1, 1536, 16, 1 << 20, 1, 1), True) > \
        pkg.ssm_scan_workspace_bytes(pkg.make_shape(1, 1536, 16, 1 << 20, 1, 1), False)


def test_plan_overrides_that_do_not_fit_fall_back(pkg, monkeypatch):
    """Tile-shape overrides that exceed the shared memory leave the planner's
    own choice in place (same workspace), instead of an unsized plan."""
    shapes = [(2, 5120, 16, 8192), (1, 64, 64, 1000), (1, 8, 8, 100)]
    base = [pkg.ssm_scan_workspace_bytes(pkg.make_shape(*sh, 1, 1), True) for sh in shapes]
    for nt, w in (("2", "6"), ("2", "7"), ("4", "9"), ("3", "1")):
        monkeypatch.setenv("SSM_BWD_NT", nt)
        monkeypatch.setenv("SSM_BWD_W", w)
        for sh, b in zip(shapes, base):
            n = pkg.ssm_scan_workspace_bytes(pkg.make_shape(*sh, 1, 1), True)
            assert n >= 256, (sh, nt, w)
    for nt, w in (("2", "9"), ("3", "1")):
        monkeypatch.setenv("SSM_FWD_NT", nt)
        monkeypatch.setenv("SSM_FWD_W", w)
        for sh in shapes:
            assert pkg.ssm_scan_workspace_bytes(pkg.make_shape(*sh, 1, 1), False) >= 256


def test_binding_fails_loudly_without_the_library(tmp_path):
    """No CPU fallback: without libssmscan.so the package does not import."""
    import importlib.util
    import shutil
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "selective_state_space_123_b300", "__init__.py")
    pkg_dir = tmp_path / "ssm_copy"
    pkg_dir.mkdir()
    shutil.copy(src, pkg_dir / "__init__.py")
    spec = importlib.util.spec_from_file_location("ssm_copy", pkg_dir / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_header_is_plain_c_and_links(pkg, tmp_path):
    """include/ssm_scan.h compiles as C99 with warnings as errors, and a C
    program that takes the address of every declared function links against
    the library (no torch, no C++ in the interface)."""
    import subprocess
    names = _declared_symbols()
    src = tmp_path / "use_abi.c"
    src.write_text('#include "ssm_scan.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   "    const void* fns[] = {%s};\n"
                   "    ssm_shape s = {1, 1, 16, 64, SSM_BF16, SSM_F32};\n"
                   "    printf(\"%%d %%d\\n\", (int)(sizeof(fns) / sizeof(fns[0])),\n"
                   "           ssm_scan_workspace_bytes(&s, 0) > 0);\n"
                   "    return 0;\n}\n" % ", ".join("(const void*)%s" % n for n in names))
    exe = tmp_path / "use_abi"
    lib_dir = os.path.dirname(pkg.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o",
                           str(exe), "-L", lib_dir, "-lssmscan", "-Wl,-rpath," + lib_dir])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(len(names)), "1"]
