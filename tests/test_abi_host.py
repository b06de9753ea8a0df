"""The C ABI without a GPU: libob.so loads, exports every entry point that
include/ob.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes as ct
import os
import re

import pytest

import momentum_compression_gb300 as ob

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from momentum_compression_gb300 import _build
    _build.build()


def _declared():
    src = open(os.path.join(ROOT, "include", "ob.h")).read()
    return sorted(set(re.findall(r"^(?:ob_status|const char\*)\s+(ob_\w+)\(", src, re.M)))


def test_header_and_binding_agree():
    assert _declared() == sorted(ob.EXPORTS)


def test_every_declared_symbol_is_exported():
    lib = ct.CDLL(ob.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name


def test_c_programs_compile_against_the_header():
    """The plain-C programs the GPU tests run (tests/cuda/*.c) compile with
    a host C compiler against include/ob.h and the CUDA runtime header:
    the header is valid C and its declarations match their use."""
    import glob
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no host C compiler or CUDA headers")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for src in sorted(glob.glob(os.path.join(root, "tests", "cuda", "*.c"))):
        r = subprocess.run([cc, "-std=c11", "-fsyntax-only", "-Wall", "-Werror",
                            "-I", os.path.join(root, "include"), "-I", cuda_inc, src],
                           capture_output=True, text=True)
        assert r.returncode == 0, src + "\n" + r.stderr


def test_layout_matches_definition():
    ctx = ob.ob_init(109_482_240, 8, 1 << 20)
    lay = ob.ob_get_layout(ctx)
    assert lay["P"] == 13_688_832 and lay["n_pad"] == 8 * 13_688_832
    assert lay["chunks_per_partition"] == 14 and lay["n_chunks"] == 112
    # 13 full chunks of 256 tiles + a last chunk of 57,344 elements (14 tiles)
    assert lay["n_tiles"] == 8 * (13 * 256 + 14)
    assert lay["words_per_worker"] == (lay["n_pad"] // 32 + 3) // 4 * 4
    ob.ob_destroy(ctx)
    ctx = ob.ob_init(5000, 3, 992, 32)
    lay = ob.ob_get_layout(ctx)
    assert lay["P"] == 1696 and lay["chunk"] == 992 and lay["chunks_per_partition"] == 2
    ob.ob_destroy(ctx)


@pytest.mark.parametrize("kw,status", [
    (dict(n=0, W=4, chunk=1024), ob.OB_ERR_INVALID),
    (dict(n=1 << 34, W=4, chunk=1024), ob.OB_ERR_INVALID),
    (dict(n=100, W=0, chunk=1024), ob.OB_ERR_INVALID),
    (dict(n=100, W=65, chunk=1024), ob.OB_ERR_UNSUPPORTED),
    (dict(n=100, W=2, chunk=1000), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=0), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, align=48), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, grad_dtype=7), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, b1=1.0), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, eps=-1.0), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, layer_offsets=[0, 50, 50, 100]), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, layer_offsets=[0, 50, 99]), ob.OB_ERR_INVALID),
    (dict(n=100, W=2, chunk=1024, layer_offsets=[1, 50, 100]), ob.OB_ERR_INVALID),
])
def test_init_rejects(kw, status):
    with pytest.raises(ob.OBError) as ei:
        ob.ob_init(**kw)
    assert ei.value.status == status
    assert ob.ob_last_error(None)


def test_calls_need_a_workspace():
    ctx = ob.ob_init(1 << 16, 2, 4096)
    for call in (
        lambda: ob.ob_compress(ctx, [16, 16], 16, [16, 16], 16, 16, stream=0),
        lambda: ob.ob_server_reduce(ctx, 16, 16, 16, 16, 16, stream=0),
        lambda: ob.ob_adam_step(ctx, 16, 16, 16, 16, 16, stream=0),
        lambda: ob.ob_warmup_step(ctx, [16, 16], 16, 16, 16, stream=0),
        lambda: ob.ob_compress_signm_ls(ctx, [16, 16], 16, 16, [16, 16], 16, 16, stream=0),
        lambda: ob.ob_server_reduce_db(ctx, 16, 16, 16, 16, 16, 32, 32, stream=0),
        lambda: ob.ob_lamb_step_signm(ctx, 16, 16, 32, 32, 16, 16, 16, None, stream=0),
        lambda: ob.ob_step_db(ctx, [16, 16], [16, 16], 16, 16, 16, 16, 16, 32, 32, 16, 16, 16,
                              stream=0),
    ):
        with pytest.raises(ob.OBError) as ei:
            call()
        assert ei.value.status == ob.OB_ERR_STATE
        assert "workspace" in ob.ob_last_error(ctx)
    ob.ob_destroy(ctx)


def test_set_workspace_checks_before_cuda():
    ctx = ob.ob_init(1 << 16, 2, 4096)
    need = ob.ob_workspace_bytes(ctx)
    with pytest.raises(ob.OBError) as ei:
        ob.ob_set_workspace(ctx, 0x1000 + 16, need, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_set_workspace(ctx, 0x1000, need - 1, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
    ob.ob_destroy(ctx)


def test_quant_int8_checks_before_cuda():
    with pytest.raises(ob.OBError) as ei:
        ob.ob_quant_int8(0x1004, 0x2000, 0x3000, 1, 0, n=100, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_quant_int8(0x1000, 0x2001, 0x3000, 1, 0, n=100, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_quant_int8(0x1000, 0x2000, 0x3000, 1, 0, n=0, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_quant_int8(None, 0x2000, 0x3000, 1, 0, n=10, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID


def test_null_ctx():
    lib = ob.lib()
    assert lib.ob_get_layout(None, None) == ob.OB_ERR_INVALID
    assert lib.ob_compress(None, None, None, None, None, None, None, None) == ob.OB_ERR_INVALID
    assert b"NULL" in lib.ob_last_error(None)


def test_codec_calls_check_before_cuda():
    """The mixed-width codec calls reject a bad width, an alignment A that
    is not a multiple of 256, NULL and misaligned pointers on the host."""
    ctx = ob.ob_init(10_000, 2, 4096)
    assert ob.ob_qb_sizes(ctx, 2) == (ob.ob_get_layout(ctx)["n_pad"] * 2 // 32,
                                      ob.ob_get_layout(ctx)["n_pad"] // 256)
    for bits in (0, 1, 3, 16):
        with pytest.raises(ob.OBError) as ei:
            ob.ob_compress_qb(ctx, bits, [16, 16], 16, [16, 16], 16, 16, 1, 1, stream=0)
        assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_qb(ctx, 2, [16, 24], 16, [16, 16], 16, 16, 1, 1, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_server_reduce_qb(ctx, 2, 16, 18, 16, 16, 16, 1, 1, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_adam_step_qb(ctx, 4, 16, 16, None, 16, 16, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_f16(ctx, 1, [16, 16], 16, [16, 16], None, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
    with pytest.raises(ob.OBError) as ei:
        ob.ob_server_reduce_f16(ctx, 16, 16, 8, stream=0)
    assert ei.value.status == ob.OB_ERR_ALIGN
    with pytest.raises(ob.OBError) as ei:
        ob.ob_zero_errors(ctx, [16, None], 16, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
    ob.ob_destroy(ctx)
    ctx = ob.ob_init(10_000, 2, 4096, align=32)
    with pytest.raises(ob.OBError) as ei:
        ob.ob_compress_qb(ctx, 2, [16, 16], 16, [16, 16], 16, 16, 1, 1, stream=0)
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    assert "256" in ob.ob_last_error(ctx)
    with pytest.raises(ob.OBError) as ei:
        ob.ob_adam_step_f16(ctx, 0, None, None, 16, None, stream=0)
    assert ei.value.status == ob.OB_ERR_UNSUPPORTED
    ob.ob_destroy(ctx)


def test_rank_reset_checks_before_cuda():
    """ob_reset_errors_rank rejects a partition outside [0, W) and missing or
    misaligned buffers before any launch (it needs no workspace)."""
    ctx = ob.ob_init(1 << 16, 2, 4096)
    ok = dict(err=0x1000, bits_row=0x2000, scales_row=0x3000, err_s_part=0x4000,
              sbits_part=0x5000, sscales_part=0x6000)
    cases = [
        (dict(j=2), ob.OB_ERR_INVALID, "partition"),
        (dict(j=-1), ob.OB_ERR_INVALID, "partition"),
        (dict(err=None), ob.OB_ERR_INVALID, "err is NULL"),
        (dict(err=0x1004), ob.OB_ERR_ALIGN, "err"),
        (dict(sbits_part=0x5008), ob.OB_ERR_ALIGN, "sbits_part"),
        (dict(sscales_part=0x6001), ob.OB_ERR_ALIGN, "sscales_part"),
    ]
    for over, status, msg in cases:
        kw = dict(ok, j=0)
        kw.update(over)
        with pytest.raises(ob.OBError) as ei:
            ob.ob_reset_errors_rank(ctx, kw.pop("j"), stream=0, **kw)
        assert ei.value.status == status, over
        assert msg in ob.ob_last_error(ctx), (over, ob.ob_last_error(ctx))
    ob.ob_destroy(ctx)
    with pytest.raises(ob.OBError) as ei:
        ob.ob_reset_errors_rank(None, 0, **ok, stream=0)
    assert ei.value.status == ob.OB_ERR_INVALID
