"""The C ABI on the host, no GPU: the library loads, exports every entry
point include/moe_prefill.h declares, sizes its workspace, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import quantized_moe_expert_quantize_gb300 as M
from quantized_moe_expert_quantize_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return M.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(M.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_bytes_layout(lib):
    d = M.make_desc(16384, 2560, 640, 512, 10)
    n = M.workspace_bytes(d)
    R = 16384 * 10
    # per routed row: hq, dh, dm (which gu shares), row_src + dst_of,
    # scattered xq and dx
    minimum = R * (640 * 2 + 20 * 4 + 2560 * 4 + 8 + 2560 * 2 + 80 * 4)
    assert minimum <= n <= minimum + 64 * 2**20
    assert n % 256 == 0
    assert M.host_io_bytes(d) >= 2 * 16384 * 2560 * 4


@pytest.mark.parametrize("d,n_ff", [(2560, 640), (256, 1024)])
def test_gu_shares_the_dm_region(lib, d, n_ff):
    """gu (live from the gate/up product to swiglu_quant) and dm (from the
    down product to the combine) are one region, as large as the larger."""
    desc = M.make_desc(64, d, n_ff, 8, 2)
    need = lib.moe_prefill_workspace_bytes(ctypes.byref(desc))
    base = 1 << 40  # never dereferenced: the view is host arithmetic
    v = M.MoeWorkspaceView()
    assert lib.moe_workspace_view(ctypes.byref(desc), ctypes.c_void_p(base), need,
                                  ctypes.byref(v)) == 0
    gu = ctypes.cast(v.gu, ctypes.c_void_p).value
    dm = ctypes.cast(v.dm, ctypes.c_void_p).value
    assert gu == dm
    assert dm + 64 * 2 * max(d, 2 * n_ff) * 4 <= base + need


@pytest.mark.parametrize("field,value,code", [
    ("d", 100, M.MOE_ERR_SHAPE), ("d", 32, M.MOE_ERR_SHAPE), ("n_ff", 96, M.MOE_ERR_SHAPE),
    ("E", 0, M.MOE_ERR_SHAPE), ("E", 2048, M.MOE_ERR_SHAPE), ("k", 0, M.MOE_ERR_SHAPE),
    ("k", 9, M.MOE_ERR_SHAPE), ("T", -1, M.MOE_ERR_SHAPE), ("gu_fmt", 4, M.MOE_ERR_FORMAT),
    ("down_fmt", 0, M.MOE_ERR_FORMAT), ("gu_layout", 2, M.MOE_ERR_FORMAT),
    ("flags", 4, M.MOE_ERR_FORMAT), ("flags", 7, M.MOE_ERR_FORMAT)])
def test_bad_descriptor_rejected(lib, field, value, code):
    d = M.make_desc(64, 256, 64, 8, 2)
    setattr(d, field, value)
    assert lib.moe_prefill_workspace_bytes(ctypes.byref(d)) == 0
    ws = ctypes.create_string_buffer(1 << 20)
    rc = lib.moe_prefill_layer(ctypes.byref(d), 16, 16, 16, 16, 16, 16, ctypes.addressof(ws),
                               1 << 20, None)
    assert rc == code


def test_layer_flags_are_accepted(lib):
    """MOE_FLAG_FUSED_COMBINE and MOE_FLAG_HOST_OUT_DEFERRED are the known
    flags: the layer keeps its workspace size (the fused combine's counters
    are always laid out), and any other bit is refused."""
    d0 = M.make_desc(64, 256, 64, 8, 2)
    for f in (M.MOE_FLAG_FUSED_COMBINE, M.MOE_FLAG_HOST_OUT_DEFERRED,
              M.MOE_FLAG_FUSED_COMBINE | M.MOE_FLAG_HOST_OUT_DEFERRED):
        d1 = M.make_desc(64, 256, 64, 8, 2, flags=f)
        assert M.workspace_bytes(d1) == M.workspace_bytes(d0) > 0
    bad = M.make_desc(64, 256, 64, 8, 2, flags=4)
    assert lib.moe_prefill_workspace_bytes(ctypes.byref(bad)) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_null_misaligned_and_small_workspace(lib):
    d = M.make_desc(64, 256, 64, 8, 2, weight_pack_bytes=1 << 20)
    need = lib.moe_prefill_workspace_bytes(ctypes.byref(d))
    ws = 1 << 40  # never dereferenced: every case below fails validation first
    dp = ctypes.byref(d)
    call = lambda *a: lib.moe_prefill_layer(dp, *a)
    ok = [_fake(0x1000), _fake(0x2000), _fake(0x3000), _fake(0x4000), _fake(0x5000),
          _fake(0x6000)]
    # null workspace / inputs
    assert call(*ok, None, need, None) == M.MOE_ERR_NULL
    assert call(None, *ok[1:], _fake(ws), need, None) == M.MOE_ERR_NULL
    assert call(ok[0], ok[1], ok[2], None, ok[4], ok[5], _fake(ws), need, None) == M.MOE_ERR_NULL
    # workspace too small / misaligned
    assert call(*ok, _fake(ws), need - 1, None) == M.MOE_ERR_WORKSPACE
    assert call(*ok, _fake(ws + 16), need, None) == M.MOE_ERR_ALIGN
    # misaligned x, weight pack
    assert call(_fake(0x1004), *ok[1:], _fake(ws), need, None) == M.MOE_ERR_ALIGN
    assert call(ok[0], ok[1], ok[2], _fake(0x4008), ok[4], ok[5], _fake(ws), need,
                None) == M.MOE_ERR_ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_no_device_is_reported(lib):
    assert M.moe_check_device() == M.MOE_ERR_DEVICE


def test_status_strings(lib):
    for code in range(-8, 1):
        assert M.status_string(code) != "unknown status code"
    assert M.status_string(-99) == "unknown status code"


def test_noalloc_route_rejects_sizes_beyond_its_scratch(lib):
    """The fixed-scratch routing entry point refuses a problem its 1 MiB
    scratch cannot hold, before touching the device."""
    d = M.make_desc(1_000_000, 256, 64, 512, 10)
    fake = ctypes.c_void_p(1 << 40)  # never dereferenced
    rc = lib.moe_route_noalloc(ctypes.byref(d), fake, fake, fake, fake, fake, None)
    assert rc == M.MOE_ERR_SCRATCH
    assert "scratch" in M.status_string(rc)
    d = M.make_desc(64, 256, 64, 8, 2)
    assert lib.moe_route_noalloc(ctypes.byref(d), fake, None, fake, fake, fake, None) == M.MOE_ERR_NULL


@pytest.mark.parametrize("gu_fmt", [M.MOE_FMT_W2, M.MOE_FMT_W4NL, M.MOE_FMT_Q8_0])
@pytest.mark.parametrize("down_fmt", [M.MOE_FMT_W2, M.MOE_FMT_W4NL, M.MOE_FMT_Q8_0])
@pytest.mark.parametrize("layout", [M.MOE_GU_SPLIT, M.MOE_GU_INTERLEAVED])
def test_every_format_and_layout_is_accepted(lib, gu_fmt, down_fmt, layout):
    """Every weight format for either matrix and both gate/up layouts pass
    validation, and the tiled pack is exactly the row-major matrices' bytes."""
    import synth
    T, d, n_ff, E, k = 64, 640, 320, 6, 2
    desc = M.make_desc(T, d, n_ff, E, k, gu_fmt, down_fmt, 0, layout)
    assert lib.moe_prefill_workspace_bytes(ctypes.byref(desc)) > 0
    want = E * (2 * n_ff * synth.row_bytes(gu_fmt, d) + d * synth.row_bytes(down_fmt, n_ff))
    assert M.tiled_pack_bytes(desc) == want


def test_plain_c_consumer(lib, tmp_path):
    """The boundary is a C ABI: a C99 program that includes only the header
    compiles warning-free, links the library, and gets from the host-side
    entry points what the Python binding gets."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "consumer"
    pkg = os.path.dirname(M.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_consumer.c"),
                    "-L", pkg, "-lmoeprefill", f"-Wl,-rpath,{pkg}", "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split(" ", 6)
    d = M.make_desc(16384, 2560, 640, 512, 10, M.MOE_FMT_W2, M.MOE_FMT_W4NL, 0,
                    M.MOE_GU_INTERLEAVED)
    assert int(out[0]) == M.workspace_bytes(d)
    assert int(out[1]) == M.tiled_pack_bytes(d)
    assert int(out[2]) == M.host_io_bytes(d)
    assert int(out[3]) == 0
    assert int(out[4]) == M.MOE_ERR_NULL
    assert int(out[5]) == M.MOE_ERR_SHAPE
    assert out[6].strip() == M.status_string(M.MOE_ERR_SHAPE)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: with the library absent, the binding raises instead of
    computing anything."""
    monkeypatch.setattr(M, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(M, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        M.lib()
    d = M.make_desc(8, 256, 64, 4, 2)
    with pytest.raises(RuntimeError):
        M.workspace_bytes(d)


def test_product_code_never_touches_the_oracle():
    """The package and the library sources neither import, include, load nor
    call the oracle: it is test infrastructure only."""
    pkg = os.path.join(ROOT, "quantized_moe_expert_quantize_gb300")
    uses = re.compile(r"^\s*(import|from)\s+oracle\b|#\s*include\s*[<\"][^>\"]*oracle"
                      r"|liboracle|moe_oracle|\borc_\w+\s*\(", re.M)
    paths = [os.path.join(d, f) for d, _, fs in os.walk(pkg) for f in fs]
    paths += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    checked = 0
    for path in paths:
        if path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            assert not uses.search(open(path).read()), path
            checked += 1
    assert checked >= 10


def test_oracle_never_touches_the_cuda_path():
    """The oracle neither imports the package nor loads or includes the CUDA
    library: the two sides share only the seeded inputs."""
    uses = re.compile(r"^\s*(import|from)\s+quantized_moe_expert_quantize_gb300|libmoeprefill"
                      r"|#\s*include\s*[<\"][^>\"]*(moe_prefill\.h|\.cuh)|\bmoe_\w+\s*\(", re.M)
    odir = os.path.join(ROOT, "oracle")
    checked = 0
    for fn in os.listdir(odir):
        if fn.endswith((".py", ".c", ".h")):
            assert not uses.search(open(os.path.join(odir, fn)).read()), fn
            checked += 1
    assert checked >= 3


def test_wait_selftest_validates_before_enqueueing(lib):
    fake = ctypes.c_void_p(1 << 20)
    assert lib.moe_selftest_wait_timeout(None, 1, None) == M.MOE_ERR_NULL
    assert lib.moe_selftest_wait_timeout(ctypes.c_void_p((1 << 20) + 2), 1, None) == M.MOE_ERR_ALIGN
    assert lib.moe_selftest_wait_timeout(fake, 2, None) == M.MOE_ERR_SHAPE
    assert lib.moe_selftest_wait_timeout(fake, 1, None) == M.MOE_ERR_DEVICE   # no GPU here
