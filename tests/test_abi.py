"""The C-ABI library builds, loads and exports every entry point include/tg.h declares.

No GPU is needed: only argument checks that return before any CUDA call are exercised.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tg_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from persistent_warp_specialized_gb300 import _build

    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tg_gemm_persistent", "tg_tile_schedule", "tg_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing


def test_binding_covers_every_declared_symbol():
    import persistent_warp_specialized_gb300 as tg

    assert sorted(tg.EXPORTED) == declared_functions()


def test_config_query(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    cfg = tg.tg_gemm_config()
    assert cfg == {"block_m": 128, "block_n": 256, "block_k": 64, "stages": 4, "group": 8}


def test_host_side_rejections_need_no_gpu(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent(16, 16, 16, 8, 8, 8, 7, stream=0)      # unknown dtype
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent(16, 16, 16, -1, 8, 8, "bf16", stream=0)  # negative size
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent(16, 16, 16, 8, 12, 8, "bf16", stream=0)  # N % 8 != 0
    assert e.value.code == tg.TG_ERR_ALIGN
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent(16, 24, 8, 8, 8, 8, "f16", stream=0)     # C not 16-byte aligned
    assert e.value.code == tg.TG_ERR_ALIGN
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent(None, 16, 16, 8, 8, 8, "f16", stream=0)  # null A
    assert e.value.code == tg.TG_ERR_ARG
    # empty problems are a successful no-op
    assert tg.tg_gemm_persistent(None, None, None, 0, 8, 8, "f16", stream=0) == 0
    assert tg.tg_gemm_persistent(None, None, None, 8, 0, 8, "f16", stream=0) == 0
    with pytest.raises(tg.TgError) as e:
        tg.tg_tile_schedule(0, 3, 148, 8)
    assert e.value.code == tg.TG_ERR_ARG
    assert "must be" in tg.tg_last_error()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "persistent_warp_specialized_gb300")
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|oracle/", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f


def test_mxfp8_host_side_rejections_need_no_gpu(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    cases = [
        ((16, 16, 16, 16, 16, 8, 8, 128, 7), tg.TG_ERR_ARG),         # unknown output dtype
        ((16, 16, 16, 16, 16, 8, 8, -128, "bf16"), tg.TG_ERR_ARG),   # negative size
        ((16, 16, 16, 16, 16, 8, 8, 96, "bf16"), tg.TG_ERR_ALIGN),   # K % 128 != 0
        ((16, 16, 16, 16, 16, 8, 12, 128, "bf16"), tg.TG_ERR_ALIGN),  # N % 8 != 0
        ((16, 16, None, 16, 16, 8, 8, 128, "bf16"), tg.TG_ERR_ARG),  # null B
        ((16, 16, 16, None, 16, 8, 8, 128, "bf16"), tg.TG_ERR_ARG),  # null SFB
        ((16, 24, 16, 16, 16, 8, 8, 128, "bf16"), tg.TG_ERR_ALIGN),  # SFA not 16-byte aligned
        ((24, 16, 16, 16, 16, 8, 8, 128, "bf16"), tg.TG_ERR_ALIGN),  # A not 16-byte aligned
    ]
    for args, code in cases:
        with pytest.raises(tg.TgError) as e:
            tg.tg_gemm_mxfp8(*args, stream=0)
        assert e.value.code == code, args
    rc = tg.load_library().tg_gemm_mxfp8_debug(16, 16, 16, 16, 16, 8, 8, 128, 1, 0, 0x400, None,
                                               0, -1)    # dynamic is not an MXFP8 option
    assert rc == tg.TG_ERR_ARG
    assert tg.tg_gemm_mxfp8(None, None, None, None, None, 0, 8, 128, "bf16", stream=0) == 0
    assert tg.tg_gemm_mxfp8(None, None, None, None, None, 8, 0, 128, "bf16", stream=0) == 0


def test_mxfp8_packed_scale_sizes_and_rejections(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    # k-blocks x row blocks (rows padded to a multiple of 256) x 512 bytes
    assert tg.tg_mxfp8_scale_bytes(0, 128) == 0
    assert tg.tg_mxfp8_scale_bytes(1, 128) == 1 * 2 * 512
    assert tg.tg_mxfp8_scale_bytes(256, 128) == 1 * 2 * 512
    assert tg.tg_mxfp8_scale_bytes(257, 256) == 2 * 4 * 512
    assert tg.tg_mxfp8_scale_bytes(8192, 8192) == 64 * 64 * 512
    for args, code in [((-1, 128), tg.TG_ERR_ARG), ((8, 96), tg.TG_ERR_ALIGN)]:
        with pytest.raises(tg.TgError) as e:
            tg.tg_mxfp8_scale_bytes(*args)
        assert e.value.code == code
    with pytest.raises(tg.TgError) as e:
        tg.tg_mxfp8_pack_scales(16, None, 8, 128, stream=0)        # null output
    assert e.value.code == tg.TG_ERR_ARG
    with pytest.raises(tg.TgError) as e:
        tg.tg_mxfp8_pack_scales(16, 24, 8, 128, stream=0)          # output not 16-byte aligned
    assert e.value.code == tg.TG_ERR_ALIGN
    assert tg.tg_mxfp8_pack_scales(None, None, 0, 0, stream=0) == 0


def test_group_width_option_rejections(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    with pytest.raises(ValueError):
        tg._group(0)
    with pytest.raises(ValueError):
        tg._group(256)
    assert tg._group(12) == 12 << 16
    # a bit above the group field is not a known variant
    with pytest.raises(tg.TgError) as e:
        tg.tg_gemm_persistent_ex(16, 16, 16, 8, 8, 8, "bf16", stream=0, variant=1 << 24)
    assert e.value.code == tg.TG_ERR_ARG


def test_mxfp8_rejects_the_dense_only_wide_variant(lib):
    import persistent_warp_specialized_gb300 as tg

    tg.load_library()
    with pytest.raises(tg.TgError) as e:     # rejected before any CUDA call
        tg.tg_gemm_mxfp8_ex(16, 16, 16, 16, 16, 256, 256, 128, "bf16", stream=0, variant="wide")
    assert e.value.code == tg.TG_ERR_ARG
