"""The C-ABI library on the host: it loads, exports what the header declares, and
rejects bad arguments before touching the GPU (no compute call is made here)."""
import os
import re

import pytest

from selective_state_space_133_b300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mamba_scan.h")


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba_[a-z_]+)\s*\(", text)))


def test_header_declares_expected_api():
    assert declared_functions() == sorted(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_checked_bounds_build_exports_the_same_abi(L):
    """The checked-bounds testing build loads, exports every declared symbol and says which it is."""
    C = _lib.load(build.build_library(checked=True))
    for name in declared_functions():
        assert hasattr(C, name), name
    assert C.mamba_checked_bounds() == 1 and L.mamba_checked_bounds() == 0
    assert C.mamba_status_string(-9).decode().startswith("MAMBA_ERR_DEVICE_BOUNDS")


SPAN_HARNESS = r"""
#include <cstdio>
#include "common.cuh"
using mscan::span_inside;
int main() {
    static float t[10];
    const float* b = t;
    int bad = 0;
    auto expect = [&](bool got, bool want, int line) { if (got != want) { std::printf("case %d\n", line); ++bad; } };
    expect(span_inside(b, 10, b, 10), true, __LINE__);                      // the whole tensor
    expect(span_inside(b, 10, b + 9, 1), true, __LINE__);                   // the last element
    expect(span_inside(b, 10, b + 9, 2), false, __LINE__);                  // one past the end
    expect(span_inside(b, 10, b + 10, 1), false, __LINE__);                 // starts at the end
    expect(span_inside(b, 10, b - 1, 1), false, __LINE__);                  // before the start
    expect(span_inside(b, 10, b + 10, 0), true, __LINE__);                  // empty access at the end
    expect(span_inside(b, 10, b, -1), false, __LINE__);                     // negative count
    expect(span_inside(static_cast<const float*>(nullptr), 10, b, 1), false, __LINE__);  // null tensor
    expect(span_inside(b, 10, reinterpret_cast<const float4*>(b + 6), 1), true, __LINE__);   // 16 bytes, last 4
    expect(span_inside(b, 10, reinterpret_cast<const float4*>(b + 7), 1), false, __LINE__);  // 16 bytes, 1 over
    expect(span_inside(reinterpret_cast<const unsigned short*>(b), 20, b + 4, 6), true, __LINE__);  // mixed types
    expect(span_inside(reinterpret_cast<const unsigned short*>(b), 19, b + 4, 6), false, __LINE__);
    std::printf("%d bad\n", bad);
    return bad != 0;
}
"""


def test_span_check_of_the_checked_build(tmp_path):
    """The extent test the checked build applies to every access, run on the host over its edge cases."""
    import subprocess
    src = tmp_path / "span.cu"
    src.write_text(SPAN_HARNESS)
    exe = tmp_path / "span"
    subprocess.run([build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-DMAMBA_DEBUG_BOUNDS",
                    "-I", build.CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0 bad", r.stdout


def test_status_strings(L):
    for code in range(0, -10, -1):
        s = L.mamba_status_string(code).decode()
        assert s.startswith(_lib.STATUS[code])
    assert L.mamba_status_string(42).decode() == "unknown mamba_status"
    assert L.mamba_version() == 300


# Fake, never-dereferenced addresses: validation fails before any CUDA call.
P = 0x10000  # 16-byte aligned


def scan(L, **kw):
    args = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, sp=1, y=P, fs=None,
                batch=2, dim=32, seqlen=64, dstate=16, dtype=0, stream=None)
    args.update(kw)
    return L.mamba_scan_fwd(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"], args["z"],
                            args["bias"], args["sp"], args["y"], args["fs"], args["batch"], args["dim"],
                            args["seqlen"], args["dstate"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), -3), (dict(dtype=-1), -3),
    (dict(dstate=4), -2), (dict(dstate=12), -2), (dict(dstate=128), -2), (dict(dstate=0), -2),
    (dict(batch=-1), -2), (dict(dim=-5), -2),
    (dict(sp=4), -8), (dict(sp=-1), -8), (dict(sp=1 << 20), -8),
    (dict(dstate=8, u=P + 8), -4), (dict(dstate=32, y=P + 4), -4), (dict(dstate=64, B=None), -1),
    (dict(seqlen=-1), -2), (dict(batch=70000), -2),
    (dict(dim=1 << 20, seqlen=1 << 20), -2),
    (dict(u=None), -1), (dict(delta=None), -1), (dict(A=None), -1), (dict(B=None), -1),
    (dict(C=None), -1), (dict(y=None), -1),
    (dict(u=P + 8), -4), (dict(y=P + 4), -4), (dict(B=P + 2), -4), (dict(z=P + 8), -4),
    (dict(fs=P + 4), -4), (dict(A=P + 4), -4), (dict(D=P + 2), -4), (dict(bias=P + 1), -4),
])
def test_scan_rejects(L, kw, code):
    assert scan(L, **kw) == code


def test_scan_empty_length_allows_null_io(L):
    # seqlen == 0 with a null A is still rejected before any launch
    assert scan(L, seqlen=0, u=None, delta=None, B=None, C=None, y=None, A=None) == -1


def test_scan_empty_is_noop(L):
    # batch or dim of 0: nothing to do, nothing launched, even with null pointers
    assert scan(L, batch=0, u=None, y=None) == 0
    assert scan(L, dim=0, u=None, y=None) == 0


def update(L, **kw):
    args = dict(state=P, u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, sp=1, y=P,
                batch=4, dim=8, dstate=16, dtype=1, stream=None)
    args.update(kw)
    return L.mamba_state_update(args["state"], args["u"], args["delta"], args["A"], args["B"], args["C"],
                                args["D"], args["z"], args["bias"], args["sp"], args["y"], args["batch"],
                                args["dim"], args["dstate"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), -3), (dict(dstate=4), -2), (dict(dstate=128), -2), (dict(batch=-2), -2),
    (dict(sp=6), -8), (dict(dstate=64, state=P + 4), -4), (dict(dstate=8, y=None), -1),
    (dict(state=None), -1), (dict(u=None), -1), (dict(y=None), -1), (dict(A=None), -1),
    (dict(state=P + 4), -4), (dict(A=P + 8), -4), (dict(B=P + 2), -4), (dict(u=P + 1), -4),
    (dict(C=P + 8), -4), (dict(batch=70000), -2),
])
def test_update_rejects(L, kw, code):
    assert update(L, **kw) == code


def test_update_empty_is_noop(L):
    assert update(L, batch=0, state=None) == 0


def scan_ws(L, ws=P, ws_bytes=1 << 30, **kw):
    args = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, sp=1, y=P, fs=None,
                batch=2, dim=32, seqlen=64, dstate=16, dtype=1, stream=None)
    args.update(kw)
    return L.mamba_scan_fwd_ws(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"], args["z"],
                               args["bias"], args["sp"], args.get("h0"), args["y"], args["fs"], args.get("ck"),
                               args["batch"],
                               args["dim"], args["seqlen"], args["dstate"], args["dtype"], ws, ws_bytes,
                               args["stream"])


def test_workspace_size(L):
    # The forward's only workspace is the carries of a split sequence, planned
    # from the current device's SM count: nothing without a device, and
    # nothing for arguments out of range.
    have_device = L.mamba_scan_workspace_size(1, 16, 1 << 20, 16, 1) > 0
    if not have_device:
        assert L.mamba_scan_workspace_size(1, 64, 131072, 16, 1) == 0
    assert L.mamba_scan_workspace_size(8, 2048, 4096, 16, 1) == 0   # enough channel rows: no split
    assert L.mamba_scan_workspace_size(1, 1, 0, 16, 1) == 0
    assert L.mamba_scan_workspace_size(1, 1, 16, 24, 1) == 0
    assert L.mamba_scan_workspace_size(1, 64, 4096, 16, 7) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=5), -3), (dict(dstate=48), -2), (dict(u=P + 2), -4), (dict(C=None), -1),
    (dict(sp=8), -8), (dict(h0=P + 8), -4), (dict(ck=P + 4), -4), (dict(batch=-1), -2), (dict(y=None), -1),
])
def test_scan_ws_rejects(L, kw, code):
    assert scan_ws(L, **kw) == code


def conv_scan(L, **kw):
    args = dict(x=P, w=P, cb=None, cs=None, width=4, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, sp=1,
                h0=None, y=P, fs=None, batch=2, dim=32, seqlen=64, dstate=16, dtype=1, ws=P, ws_bytes=1 << 30)
    args.update(kw)
    return L.mamba_conv_scan_fwd_ws(args["x"], args["w"], args["cb"], args["cs"], args["width"], args["delta"],
                                    args["A"], args["B"], args["C"], args["D"], args["z"], args["bias"], args["sp"],
                                    args["h0"], args["y"], args["fs"], args["batch"], args["dim"], args["seqlen"],
                                    args["dstate"], args["dtype"], args["ws"], args["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(width=3), -2), (dict(width=5), -2), (dict(w=None), -1), (dict(w=P + 8), -4), (dict(cb=P + 2), -4),
    (dict(cs=P + 1), -4), (dict(x=None), -1), (dict(dtype=3), -3),
    (dict(sp=16), -8), (dict(dstate=20), -2),
])
def test_conv_scan_rejects(L, kw, code):
    assert conv_scan(L, **kw) == code


def scan_bwd(L, **kw):
    args = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, sp=1, h0=None, ck=None, dy=P, du=P, ddl=P,
                dA=P, dB=P, dC=P, dD=None, dz=None, dbias=None, dh0=None, batch=2, dim=32, seqlen=64, dstate=16,
                dtype=1, ws=P, ws_bytes=1 << 30)
    args.update(kw)
    return L.mamba_scan_bwd(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"], args["z"],
                            args["bias"], args["sp"], args["h0"], args["ck"], args["dy"], args["du"], args["ddl"],
                            args["dA"], args["dB"], args["dC"], args["dD"], args["dz"], args["dbias"], args["dh0"],
                            args["batch"], args["dim"], args["seqlen"], args["dstate"], args["dtype"], args["ws"],
                            args["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dstate=12), -2), (dict(dstate=128), -2), (dict(sp=4), -8), (dict(sp=-1), -8),
    (dict(dstate=8, du=P + 4), -4), (dict(dstate=64, sp=3, dA=None), -1),
    (dict(dA=None), -1), (dict(z=P, dz=None), -1), (dict(dD=P), -1), (dict(du=P + 4), -4),
    (dict(ws_bytes=100), -7),
])
def test_scan_bwd_rejects(L, kw, code):
    assert scan_bwd(L, **kw) == code


def test_bwd_workspace_size(L):
    # packed B/C rows + one state per 16 steps + fp32 dB/dC sums, each rounded to 256 bytes
    for n in (8, 16, 32, 64):
        want = 2 * 64 * 2 * n * 4 + 2 * 32 * 4 * n * 4 + 2 * 2 * n * 64 * 4
        assert L.mamba_scan_bwd_workspace_size(2, 32, 64, n, 1) == want
    assert L.mamba_scan_bwd_workspace_size(2, 32, 64, 24, 1) == 0


def ssd(L, **kw):
    args = dict(x=P, delta=P, A=P, B=P, C=P, D=None, bias=None, flags=1, h0=None, y=P, fs=None, batch=2, nheads=4,
                headdim=64, seqlen=128, dstate=128, dtype=1, ws=None, ws_bytes=0)
    args.update(kw)
    return L.mamba_ssd_fwd(args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"], args["bias"],
                           args["flags"], args["h0"], args["y"], args["fs"], args["batch"], args["nheads"],
                           args["headdim"], args["seqlen"], args["dstate"], args["dtype"], args["ws"],
                           args["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=0), -3), (dict(dtype=4), -3), (dict(flags=2), -8), (dict(flags=4), -8),
    (dict(headdim=32), -2), (dict(headdim=128), -2), (dict(dstate=16), -2), (dict(dstate=512), -2),
    (dict(batch=-1), -2), (dict(nheads=-1), -2), (dict(seqlen=-3), -2), (dict(batch=70000), -2),
    (dict(A=None), -1), (dict(x=None), -1), (dict(delta=None), -1), (dict(B=None), -1), (dict(y=None), -1),
    (dict(x=P + 8), -4), (dict(y=P + 4), -4), (dict(C=P + 2), -4), (dict(delta=P + 1), -4), (dict(fs=P + 8), -4),
    (dict(h0=P + 4), -4), (dict(D=P + 2), -4),
    (dict(seqlen=100), -1), (dict(seqlen=100, ws=P, ws_bytes=10), -7), (dict(seqlen=100, ws=P + 16, ws_bytes=1 << 30), -4),
])
def test_ssd_rejects(L, kw, code):
    assert ssd(L, **kw) == code


def test_ssd_empty_is_noop(L):
    assert ssd(L, batch=0, x=None, y=None) == 0
    assert ssd(L, nheads=0, x=None, y=None) == 0


def test_ssd_workspace_size(L):
    assert L.mamba_ssd_workspace_size(2, 4, 64, 128, 128, 1) == 0            # 256-byte rows: no copies
    w = L.mamba_ssd_workspace_size(2, 4, 64, 100, 128, 1)                    # 200-byte rows: pitched copies
    assert w >= 2 * (2 * 4 * 64 + 2 * 2 * 128) * 104
    assert L.mamba_ssd_workspace_size(2, 4, 64, 100, 128, 0) == 0            # fp32 I/O is not supported
    assert L.mamba_ssd_workspace_size(2, 4, 32, 100, 128, 1) == 0


def ssd_update(L, **kw):
    args = dict(state=P, x=P, delta=P, A=P, B=P, C=P, D=None, bias=None, flags=1, y=P, batch=4, nheads=2, headdim=64,
                dstate=128, dtype=1)
    args.update(kw)
    return L.mamba_ssd_update(args["state"], args["x"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                              args["bias"], args["flags"], args["y"], args["batch"], args["nheads"], args["headdim"],
                              args["dstate"], args["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=3), -3), (dict(flags=2), -8), (dict(headdim=32), -2), (dict(dstate=16), -2), (dict(batch=-1), -2),
    (dict(batch=70000), -2), (dict(state=None), -1), (dict(x=None), -1), (dict(delta=None), -1), (dict(C=None), -1),
    (dict(y=None), -1), (dict(A=None), -1), (dict(state=P + 8), -4), (dict(B=P + 8), -4), (dict(x=P + 1), -4),
    (dict(dtype=0, y=P + 2), -4), (dict(D=P + 2), -4),
])
def test_ssd_update_rejects(L, kw, code):
    assert ssd_update(L, **kw) == code


def test_ssd_update_empty_is_noop(L):
    assert ssd_update(L, batch=0, state=None) == 0
