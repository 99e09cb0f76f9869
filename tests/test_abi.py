"""The C-ABI library loads, exports every symbol include/awq.h declares, and
rejects bad arguments on the host before touching a GPU (no compute call)."""
import ctypes
import re

import pytest

awq = pytest.importorskip("weight_only_bit_05_b300")
lib = awq.lib

AWQ_OK, AWQ_ERR_SHAPE, AWQ_ERR_NULL, AWQ_ERR_ALIGN = 0, 1, 2, 3
AWQ_ERR_UNSUPPORTED, AWQ_ERR_WORKSPACE = 5, 6
FAKE = 0x10000          # never dereferenced: validation fails first
MIS = FAKE + 4          # misaligned pointer


def test_every_declared_symbol_is_exported():
    names = awq.exported_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_header_declares_what_the_binding_uses():
    with open(awq.HEADER) as f:
        txt = f.read()
    for n in awq._SIGS:
        assert re.search(r"\b%s\s*\(" % n, txt), n


def test_default_config_and_workspace_sizes():
    c = lib.awq_default_config()
    assert (c.w_bit, c.group, c.zero_point, c.n_grid) == (4, 128, 1, 20)
    assert lib.awq_gemm_workspace_size(16, 512, 512) == 16 * 512 * 2
    # few 128-row tiles: the plans split K, and the workspace also holds the
    # fp32 partial sums, at most 8 parts of [M][N] for the narrow-token kernel
    # (up to 128 tokens) or of each [bn][128] tile (bn = the token tile) for
    # the wide one
    for M, N, K, bn in ((16, 256, 4096, 16), (120, 256, 4096, 128), (48, 640, 8192, 64),
                        (300, 1024, 8192, 160)):
        xt = ((M * K * 2 + 255) // 256) * 256
        part = lib.awq_gemm_workspace_size(M, N, K) - xt
        padded = -(-M // bn) * bn * -(-N // 128) * 128 * 4
        assert part > 0 and part % 4 == 0 and part <= 8 * max(padded, M * N * 4), (M, N, K)
    assert lib.awq_gemm_workspace_size(0, 512, 512) == 0
    # Without a device the library plans for 148 SMs.  160-token tiles:
    # 2048 x 3584 has 28 x 13 = 364 tiles, two full rounds and 68 left, so
    # only those 68 tiles are split over K, 2 parts each (68 x 2 <= 148
    # SMs), one [160][128] fp32 block per part; 160 x 18944 has exactly one
    # round of 148 tiles and no split.
    xt = 2048 * 4096 * 2
    assert lib.awq_gemm_workspace_size(2048, 3584, 4096) == xt + 68 * 2 * 160 * 128 * 4
    assert lib.awq_gemm_workspace_size(160, 18944, 4096) == 160 * 4096 * 2
    assert lib.awq_absmean_workspace_size(4096, 4096) % 8 == 0
    assert lib.awq_absmean_workspace_size(4096, 4096) >= 4096 * 8
    ws = lib.awq_search_workspace_size(65536, 57344, 8192)
    # Yref chunk <= 4 GiB, X~ 1 GiB, plus the packed chunk: a few GiB, not 15
    assert (1 << 30) * 5 < ws < (1 << 30) * 7


def _err():
    return lib.awq_last_error_string().decode()


def test_gemv_validation():
    f = lib.awq_gemv
    assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 512, 100, FAKE, None) == AWQ_ERR_SHAPE
    assert "multiple of 128" in _err()
    assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 12, 512, FAKE, None) == AWQ_ERR_SHAPE
    assert f(FAKE, 9, FAKE, FAKE, FAKE, None, 512, 512, FAKE, None) == AWQ_ERR_SHAPE
    assert f(FAKE, 0, FAKE, FAKE, FAKE, None, 512, 512, FAKE, None) == AWQ_ERR_SHAPE
    assert f(None, 1, FAKE, FAKE, FAKE, None, 512, 512, FAKE, None) == AWQ_ERR_NULL
    assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 512, 512, None, None) == AWQ_ERR_NULL
    assert f(FAKE, 1, MIS, FAKE, FAKE, None, 512, 512, FAKE, None) == AWQ_ERR_ALIGN
    assert f(FAKE, 1, FAKE, FAKE, FAKE, MIS, 512, 512, FAKE, None) == AWQ_ERR_ALIGN


def test_gemm_validation():
    f = lib.awq_gemm
    assert f(FAKE, 0, FAKE, FAKE, FAKE, None, 512, 512, FAKE, None, 0, None) == AWQ_ERR_SHAPE
    assert f(FAKE, 4, FAKE, FAKE, FAKE, None, 512, 384 + 64, FAKE, None, 0, None) == AWQ_ERR_SHAPE
    # inv_s given: the workspace must hold X~
    assert f(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 512, 512, FAKE, None, 0, None) == AWQ_ERR_WORKSPACE
    assert f(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 512, 512, FAKE, FAKE, 100, None) == AWQ_ERR_WORKSPACE
    assert f(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 512, 512, FAKE, MIS, 1 << 20, None) == AWQ_ERR_WORKSPACE


def test_pack_validation_and_config():
    f = lib.awq_pack
    cfg = lib.awq_default_config()
    assert f(FAKE, None, 8, 100, ctypes.byref(cfg), FAKE, FAKE, FAKE, None) == AWQ_ERR_SHAPE
    assert f(FAKE, None, 8, 128, ctypes.byref(cfg), None, FAKE, FAKE, None) == AWQ_ERR_NULL
    for field, val in (("w_bit", 3), ("w_bit", 2), ("group", 256), ("group", 96),
                       ("zero_point", 2), ("n_grid", 0)):
        bad = lib.awq_default_config()
        setattr(bad, field, val)
        assert f(FAKE, None, 8, 128, ctypes.byref(bad), FAKE, FAKE, FAKE, None) == AWQ_ERR_UNSUPPORTED


def test_stats_and_search_validation():
    assert lib.awq_absmean(FAKE, 0, 128, FAKE, FAKE, 1 << 20, None) == AWQ_ERR_SHAPE
    assert lib.awq_absmean(FAKE, 16, 128, FAKE, None, 0, None) == AWQ_ERR_WORKSPACE
    assert lib.awq_channel_scales(FAKE, 128, 1.0, FAKE, FAKE, None) == AWQ_ERR_SHAPE
    assert lib.awq_channel_scales(FAKE, 128, -0.5, FAKE, FAKE, None) == AWQ_ERR_SHAPE
    best = ctypes.c_int32()
    mse = (ctypes.c_double * 20)()
    cfg = lib.awq_default_config()
    args = [FAKE, 256, FAKE, 512, 512, ctypes.byref(cfg), FAKE, 1 << 40, FAKE, FAKE,
            ctypes.byref(best), mse, None, None]
    bad = list(args)
    bad[4] = 100
    assert lib.awq_search_scales(*bad) == AWQ_ERR_SHAPE
    bad = list(args)
    bad[7] = 16
    assert lib.awq_search_scales(*bad) == AWQ_ERR_WORKSPACE
    bad = list(args)
    bad[10] = None
    assert lib.awq_search_scales(*bad) == AWQ_ERR_NULL


def test_fused_gate_up_validation():
    for f, extra in ((lib.awq_gemv_silu_mul, ()), (lib.awq_gemm_silu_mul, (None, 0))):
        # I must be a positive multiple of 4 (2I rows, a multiple of 8)
        assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 6, 512, FAKE, *extra, None) == AWQ_ERR_SHAPE
        assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 0, 512, FAKE, *extra, None) == AWQ_ERR_SHAPE
        assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 256, 200, FAKE, *extra, None) == AWQ_ERR_SHAPE
        assert f(FAKE, 1, None, FAKE, FAKE, None, 256, 512, FAKE, *extra, None) == AWQ_ERR_NULL
        assert f(FAKE, 1, FAKE, FAKE, FAKE, None, 256, 512, MIS, *extra, None) == AWQ_ERR_ALIGN
    assert lib.awq_gemv_silu_mul(FAKE, 9, FAKE, FAKE, FAKE, None, 256, 512, FAKE,
                                 None) == AWQ_ERR_SHAPE
    # the tensor-core form needs the workspace when inv_s is given
    assert lib.awq_gemm_silu_mul(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 256, 512, FAKE, None, 0,
                                 None) == AWQ_ERR_WORKSPACE


def test_fold_validation():
    f = lib.awq_fold_inv_scales
    assert f(FAKE, 0, 4, FAKE, FAKE, None) == AWQ_ERR_SHAPE
    assert f(FAKE, 4, 0, FAKE, FAKE, None) == AWQ_ERR_SHAPE
    assert f(None, 4, 4, FAKE, FAKE, None) == AWQ_ERR_NULL
    assert f(FAKE, 4, 4, None, FAKE, None) == AWQ_ERR_NULL
    assert f(FAKE, 4, 4, FAKE, MIS, None) == AWQ_ERR_ALIGN


def test_variant_configs_are_accepted_by_validation():
    # the variants pass configuration checks (and then fail on a later, shape check)
    f = lib.awq_pack
    for w_bit, group, zp in ((4, 64, 1), (4, 32, 0), (8, 128, 1), (8, 32, 0)):
        c = lib.awq_default_config()
        c.w_bit, c.group, c.zero_point = w_bit, group, zp
        assert f(FAKE, None, 8, 100, ctypes.byref(c), FAKE, FAKE, FAKE, None) == AWQ_ERR_SHAPE
        assert lib.awq_gemv_ex(ctypes.byref(c), FAKE, 9, FAKE, FAKE, FAKE, None, 512, 512, FAKE,
                               None) == AWQ_ERR_SHAPE
    bad = lib.awq_default_config()
    bad.w_bit = 3
    assert lib.awq_gemm_ex(ctypes.byref(bad), FAKE, 4, FAKE, FAKE, FAKE, None, 512, 512, FAKE,
                           None, 0, None) == AWQ_ERR_UNSUPPORTED


def test_debug_stall_hook_validates_its_arguments():
    """The test hook rejects a kernel selection outside 0..3 and a wait limit
    outside [1e3, 1e10] ns before any CUDA call (runs without a GPU)."""
    for which, ns in ((1, 0), (1, 999), (2, 10_000_000_001), (4, 1_000_000), (-1, 1_000_000)):
        assert awq.lib.awq_debug_stall(which, ns) == 1   # AWQ_ERR_SHAPE
        assert b"awq_debug_stall" in awq.lib.awq_last_error_string()
