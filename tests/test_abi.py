"""The C ABI of libqz without a GPU: the library loads, exports every function that
include/qz.h declares, its structs have the header's layout, and argument errors come
back synchronously (they are checked before any CUDA call)."""
import ctypes as C
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qz.h")


@pytest.fixture(scope="module")
def qz():
    import __graft_entry__
    __graft_entry__.build_library()
    import precision_quantization_gb300 as qz
    qz.lib()
    return qz


def declared_functions():
    txt = open(HEADER, encoding="utf-8").read()
    return set(re.findall(r"QZ_API\s+[\w\s\*]+?\b(qz_\w+)\s*\(", txt))


def test_exports_every_declared_symbol(qz):
    decl = declared_functions()
    assert decl == set(qz.ABI_SYMBOLS)
    out = subprocess.run(["nm", "-D", "--defined-only", qz.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    assert decl <= exported
    for name in decl:
        assert hasattr(qz.lib(), name)


def test_struct_layout_matches_header(qz, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "qz.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu\\n\","
        " sizeof(qz_desc), offsetof(qz_desc, rows), offsetof(qz_desc, ld),"
        " sizeof(qz_stats), offsetof(qz_stats, mse), offsetof(qz_stats, max_rel_err),"
        " offsetof(qz_stats, max_abs_err), offsetof(qz_stats, n)); return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [C.sizeof(qz.QzDesc), qz.QzDesc.rows.offset, qz.QzDesc.ld.offset,
            C.sizeof(qz.QzStats), qz.QzStats.mse.offset, qz.QzStats.max_rel_err.offset,
            qz.QzStats.max_abs_err.offset, qz.QzStats.n.offset]
    assert got == want


def test_enum_values_match_header(qz):
    txt = open(HEADER, encoding="utf-8").read()
    for name, val in re.findall(r"\b(QZ_[A-Z0-9_]+)\s*=\s*(\d+)", txt):
        assert getattr(qz, name) == int(val), name
    for name, val in re.findall(r"#define\s+(QZ_FLAG_\w+)\s+(0x[0-9a-fA-F]+)u", txt):
        assert getattr(qz, name) == int(val, 16)


def test_status_strings(qz):
    for s in range(8):
        assert qz.qz_status_string(s) and qz.qz_status_string(s) != "unknown status"
    assert qz.qz_status_string(99) == "unknown status"


def test_workspace_size(qz):
    n = qz.qz_workspace_size()
    assert n >= 256 and n % 16 == 0
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 128, 256)
    assert qz.qz_workspace_size(d) == n


FAKE = 1 << 20  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("mutate,want", [
    (lambda d: setattr(d, "format", 9), "QZ_ERR_ENUM"),
    (lambda d: setattr(d, "granularity", 0), "QZ_ERR_ENUM"),
    (lambda d: setattr(d, "elem_round", 1), "QZ_ERR_ENUM"),
    (lambda d: setattr(d, "scale_round", 2), "QZ_ERR_ENUM"),
    (lambda d: setattr(d, "in_dtype", 7), "QZ_ERR_ENUM"),
    (lambda d: setattr(d, "rows", -1), "QZ_ERR_SHAPE"),
    (lambda d: setattr(d, "ld", 10), "QZ_ERR_SHAPE"),
    (lambda d: setattr(d, "cols", 40), "QZ_ERR_SHAPE"),         # not a multiple of 16
    (lambda d: setattr(d, "block_size", 32), "QZ_ERR_UNSUPPORTED"),
    (lambda d: setattr(d, "granularity", 2), "QZ_ERR_UNSUPPORTED"),  # NVFP4 per row
])
def test_quantize_argument_errors(qz, mutate, want):
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 4, 64)
    mutate(d)
    rc = qz.qz_quantize(d, FAKE, FAKE, FAKE, FAKE, FAKE, None, None)
    assert rc == getattr(qz, want)


def test_quantize_null_and_workspace_errors(qz):
    assert qz.lib().qz_quantize(None, FAKE, FAKE, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_NULL
    d = qz.make_desc("e4m3", qz.QZ_BF16, "tensor", 4, 64)
    # per-tensor scale computed in the library: needs a workspace
    assert qz.qz_quantize(d, FAKE, FAKE, None, FAKE, None, None, None) == qz.QZ_ERR_WORKSPACE
    # ... and a tensor-scale output
    assert qz.qz_quantize(d, FAKE, FAKE, None, None, FAKE, None, None) == qz.QZ_ERR_NULL
    # misaligned workspace / stats
    assert qz.qz_quantize(d, FAKE, FAKE, None, FAKE, None, None, FAKE + 4) == qz.QZ_ERR_ALIGN
    assert qz.qz_quantize(d, FAKE, FAKE, None, FAKE, FAKE, FAKE + 4, FAKE) == qz.QZ_ERR_ALIGN
    # missing x / codes / row scales
    d_row = qz.make_desc("int8", qz.QZ_F32, "row", 4, 64)
    assert qz.qz_quantize(d_row, None, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_NULL
    assert qz.qz_quantize(d_row, FAKE, FAKE, None, None, None, None, None) == qz.QZ_ERR_NULL
    # misaligned fp32 input
    assert qz.qz_quantize(d_row, FAKE + 2, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_ALIGN
    # 8-bit formats take no block size and no BLOCK granularity
    d_bad = qz.make_desc("int8", qz.QZ_F32, "block", 4, 64)
    assert qz.qz_quantize(d_bad, FAKE, FAKE, FAKE, FAKE, None, None, FAKE) == qz.QZ_ERR_UNSUPPORTED


def test_quantize_delayed_argument_errors(qz):
    qd = qz.qz_quantize_delayed
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 4, 64)
    # amax_out is required; NVFP4 BLOCK also needs amax_in and the tensor-scale output
    assert qd(d, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE) == qz.QZ_ERR_NULL
    assert qd(d, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, FAKE) == qz.QZ_ERR_NULL
    assert qd(d, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE) == qz.QZ_ERR_NULL
    # the workspace is always required (the amax of this tensor is folded through it)
    assert qd(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == qz.QZ_ERR_WORKSPACE
    assert qd(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None, FAKE) == qz.QZ_ERR_ALIGN
    # MXFP4 BLOCK and ROW scales need no amax_in
    d_mx = qz.make_desc("mxfp4", qz.QZ_BF16, "block", 4, 64)
    assert qd(d_mx, None, FAKE, FAKE, None, None, FAKE, None, FAKE) == qz.QZ_ERR_NULL  # x
    d_row = qz.make_desc("e4m3", qz.QZ_F32, "row", 4, 64)
    assert qd(d_row, FAKE, FAKE, None, None, None, FAKE, None, FAKE) == qz.QZ_ERR_NULL  # scales
    assert qz.lib().qz_quantize_delayed(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                        None) == qz.QZ_ERR_NULL


def test_int4_descriptor_rules(qz):
    for bs in (16, 32, 64, 128):
        d = qz.make_desc("int4", qz.QZ_BF16, "block", 4, 256, block_size=bs)
        assert qz.qz_quantize(d, None, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_NULL  # x
    for bs in (0, 8, 48, 256):
        d = qz.make_desc("int4", qz.QZ_BF16, "block", 4, 256)
        d.block_size = bs
        assert qz.qz_quantize(d, FAKE, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_UNSUPPORTED
    d = qz.make_desc("int4", qz.QZ_BF16, "tensor", 4, 256)
    assert qz.qz_quantize(d, FAKE, FAKE, FAKE, FAKE, None, None, FAKE) == qz.QZ_ERR_UNSUPPORTED
    d = qz.make_desc("int4", qz.QZ_F32, "block", 4, 80, block_size=32)   # cols % 32 != 0
    assert qz.qz_quantize(d, FAKE, FAKE, FAKE, None, None, None, None) == qz.QZ_ERR_SHAPE
    d = qz.make_desc("int4", qz.QZ_F32, "block", 4, 64, block_size=32)
    assert qz.qz_quantize(d, FAKE, FAKE, None, None, None, None, None) == qz.QZ_ERR_NULL  # scales
    assert qz.qz_quantize(d, FAKE, FAKE, FAKE + 2, None, None, None, None) == qz.QZ_ERR_ALIGN


def test_asym4_argument_errors_host(qz):
    F = FAKE
    assert qz.qz_dequantize_asym4(F, F, F, 2, 20, 4, F, 20, qz.QZ_F32) == qz.QZ_ERR_SHAPE
    assert qz.qz_dequantize_asym4(F, F, F, 2, 64, 24, F, 64, qz.QZ_F32) == qz.QZ_ERR_SHAPE
    assert qz.qz_dequantize_asym4(F, F, F, 2, 64, 16, F, 32, qz.QZ_F32) == qz.QZ_ERR_SHAPE  # ld
    assert qz.qz_dequantize_asym4(None, F, F, 2, 64, 16, F, 64, qz.QZ_F32) == qz.QZ_ERR_NULL
    assert qz.qz_dequantize_asym4(F, F, F, 2, 64, 16, F + 2, 64, qz.QZ_F32) == qz.QZ_ERR_ALIGN
    assert qz.qz_dequantize_asym4(F, F, F, 2, 64, 16, F, 64, 9) == qz.QZ_ERR_ENUM


def test_quant_dot_argument_errors_host(qz):
    F = FAKE
    qd = qz.qz_quant_dot
    big = 1 << 30
    assert qd(F, F, F, 4, 64, 16, F, big, big, F, big) == qz.QZ_ERR_UNSUPPORTED  # n1 >= 2^30
    assert qd(None, F, F, 4, 64, 16, F, 300, 300, F, 300) == qz.QZ_ERR_NULL     # many columns
    assert qd(F, F, F, 4, 64, 16, F + 1, 300, 300, F, 300) == qz.QZ_ERR_ALIGN
    assert qd(F, F, F, 4, 60, 4, F, 8, 8, F, 8) == qz.QZ_ERR_SHAPE              # mid % 8
    assert qd(F, F, F, 4, 64, 24, F, 8, 8, F, 8) == qz.QZ_ERR_SHAPE             # mid % group
    assert qd(F, F, F, 4, 64, 16, F, 4, 8, F, 8) == qz.QZ_ERR_SHAPE             # ld_y < n1
    assert qd(None, F, F, 4, 64, 16, F, 8, 8, F, 8) == qz.QZ_ERR_NULL
    assert qd(F, F, F, 4, 64, 16, F + 1, 8, 8, F, 8) == qz.QZ_ERR_ALIGN


def test_dequantize_and_stats_argument_errors(qz):
    d = qz.make_desc("mxfp4", qz.QZ_BF16, "block", 4, 64)
    assert qz.qz_dequantize(d, FAKE, FAKE, None, FAKE, 5) == qz.QZ_ERR_ENUM
    assert qz.qz_dequantize(d, None, FAKE, None, FAKE, qz.QZ_BF16) == qz.QZ_ERR_NULL
    assert qz.qz_dequantize(d, FAKE, None, None, FAKE, qz.QZ_BF16) == qz.QZ_ERR_NULL
    assert qz.qz_dequantize(d, FAKE, FAKE, None, FAKE + 1, qz.QZ_BF16) == qz.QZ_ERR_ALIGN
    dn = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 4, 64)
    assert qz.qz_dequantize(dn, FAKE, FAKE, None, FAKE, qz.QZ_F32) == qz.QZ_ERR_NULL
    assert qz.qz_error_stats(d, FAKE, FAKE, FAKE, None, None, FAKE) == qz.QZ_ERR_NULL
    assert qz.qz_error_stats(d, FAKE, FAKE, FAKE, None, FAKE, None) == qz.QZ_ERR_WORKSPACE
    assert qz.qz_amax(d, FAKE, None, FAKE) == qz.QZ_ERR_NULL
    assert qz.qz_workspace_init(None, 1 << 20) == qz.QZ_ERR_NULL
    assert qz.qz_workspace_init(FAKE, 16) == qz.QZ_ERR_WORKSPACE
    st, _ = qz.qz_get_device_status(None)
    assert st == qz.QZ_ERR_NULL


def test_binding_fails_loudly_without_library(qz, monkeypatch, tmp_path):
    import precision_quantization_gb300 as mod
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(ImportError):
        mod.lib()


def test_host_io_layout_matches_header(qz, tmp_path):
    src = tmp_path / "hostio.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "qz.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %d\\n\", sizeof(qz_host_io),"
        " offsetof(qz_host_io, y), offsetof(qz_host_io, stats), offsetof(qz_host_io, codes_host),"
        " offsetof(qz_host_io, stats_host), QZ_HOST_MAX_RUNS); return 0;}\n")
    exe = tmp_path / "hostio"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    io = qz.QzHostIo
    assert got == [C.sizeof(io), io.y.offset, io.stats.offset, io.codes_host.offset,
                   io.stats_host.offset, qz.QZ_HOST_MAX_RUNS]


def test_host_plan_argument_errors(qz):
    """Every argument error of qz_host_plan_create comes back before a CUDA call, with the
    plan handle left NULL; the other host-plan calls reject a NULL plan."""
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 64, 256)
    e = qz.make_desc("e4m3", qz.QZ_BF16, "tensor", 64, 256)
    create = qz.qz_host_plan_create
    assert create([d, e], 0, qz.QZ_BF16, True) == (qz.QZ_ERR_SHAPE, None)   # chunk_rows
    assert create([], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_NULL, None)       # no runs
    assert create([d] * 17, 16, qz.QZ_BF16, True) == (qz.QZ_ERR_SHAPE, None)
    assert create([d], 16, 9, True) == (qz.QZ_ERR_ENUM, None)               # out dtype
    mixed = qz.make_desc("e4m3", qz.QZ_F32, "tensor", 64, 256)
    assert create([d, mixed], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_ENUM, None)
    other_rows = qz.make_desc("e4m3", qz.QZ_BF16, "tensor", 65, 256)
    assert create([d, other_rows], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_SHAPE, None)
    strided = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 64, 256, 512)
    assert create([strided], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_SHAPE, None)
    bad_fmt = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 64, 256)
    bad_fmt.format = 9
    assert create([bad_fmt], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_ENUM, None)
    ragged = qz.make_desc("e4m3", qz.QZ_BF16, "tensor", 64, 40)
    ragged_nv = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 64, 48)
    ragged_nv.cols, ragged_nv.ld = 40, 40
    assert create([ragged, ragged_nv], 16, qz.QZ_BF16, True) == (qz.QZ_ERR_SHAPE, None)
    assert qz.lib().qz_host_plan_create(None, 1, 16, qz.QZ_BF16, 1, None) == qz.QZ_ERR_NULL
    assert qz.qz_host_run(None, FAKE, [qz.QzHostIo()]) == qz.QZ_ERR_NULL
    assert qz.qz_host_plan_status(None)[0] == qz.QZ_ERR_NULL
    qz.qz_host_plan_destroy(None)  # a no-op
