"""The C-ABI library loads on the host and exports every function include/*.h declares; host-side
argument checks return their status codes without touching a GPU."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_block_scaled_03_gb300 import build_ext
    build_ext.build()
    import mxfp8_block_scaled_03_gb300 as mx
    return mx.lib()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+\**([a-z][a-z0-9_]*)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("mxfp8_quantize", "grouped_mlp_fwd", "grouped_mlp_workspace_size", "mxfp8_check_device_error"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    import mxfp8_block_scaled_03_gb300 as mx
    assert mx.mxfp8_abi_version() == 1
    assert mx.mxfp8_status_string(0) == "ok"
    assert "split" in mx.mxfp8_status_string(6)


def test_sf_bytes(lib):
    import mxfp8_block_scaled_03_gb300 as mx
    assert mx.mxfp8_sf_bytes(77, 96, mx.ROWWISE, mx.SF_COMPACT) == 77 * 3
    assert mx.mxfp8_sf_bytes(77, 96, mx.COLWISE, mx.SF_COMPACT) == 3 * 96
    assert mx.mxfp8_sf_bytes(256, 384, mx.ROWWISE, mx.SF_MMA) == 2 * 3 * 512
    assert mx.mxfp8_sf_bytes(256, 384, mx.COLWISE, mx.SF_MMA) == 3 * 2 * 512
    assert mx.mxfp8_sf_bytes(4, 48, mx.ROWWISE, mx.SF_COMPACT) == 0


def test_workspace_layout(lib):
    import mxfp8_block_scaled_03_gb300 as mx
    L = mx.grouped_mlp_workspace_layout(32768, 4096, 14336, 8)
    assert L["r_pad"] == 34816          # 32768 + 255*8 rounded up to 256
    assert L["xq"] % 256 == 0 and L["hq"] % 256 == 0
    assert L["xsf"] - L["xq"] >= 34816 * 4096
    assert mx.grouped_mlp_workspace_size(32768, 4096, 14336, 8) >= L["hsf"] + 34816 * 14336 // 32
    assert mx.grouped_mlp_workspace_size(10, 100, 128, 1) > 0      # H need not be valid for the size query
    assert mx.grouped_mlp_workspace_size(10, 128, 128, 0) == 0


def test_host_argument_checks(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)        # never dereferenced: every call below fails its host checks first
    assert lib.mxfp8_quantize(fake, 4, 48, 1, 0, fake, fake, None, None, None) == 1       # K % 32
    assert lib.mxfp8_quantize(fake, 4, 64, 0, 0, fake, fake, None, None, None) == 1       # no direction
    assert lib.mxfp8_quantize(fake, 4, 64, 1, 7, fake, fake, None, None, None) == 1       # layout
    assert lib.mxfp8_quantize(None, 4, 64, 1, 0, fake, fake, None, None, None) == 1       # null x
    assert lib.mxfp8_quantize(P((1 << 20) + 8), 4, 64, 1, 0, fake, fake, None, None, None) == 1  # alignment
    assert lib.mxfp8_quantize(fake, 4, 64, 2, 0, fake, fake, None, None, None) == 1       # missing col outputs
    assert lib.mxfp8_quantize(fake, 100, 128, 1, 1, fake, fake, None, None, None) == 2    # MMA layout, M % 128
    assert lib.mxfp8_quantize(fake, 0, 64, 1, 0, None, None, None, None, None) == 0      # empty: no-op
    g = lib.grouped_mlp_fwd
    args = [fake, 256, 256, 256, 2, fake, None, fake, fake, fake, fake, fake, fake, 1 << 40, None]
    bad = list(args); bad[2] = 200
    assert g(*bad) == 2                                                                   # H % 128
    bad = list(args); bad[4] = 0
    assert g(*bad) == 1                                                                   # E
    bad = list(args); bad[5] = None
    assert g(*bad) == 1                                                                   # split_sizes
    bad = list(args); bad[0] = None
    assert g(*bad) == 1                                                                   # null x with rows
    bad = list(args); bad[11] = None
    assert g(*bad) == 1                                                                   # null y with rows
    bad = list(args); bad[13] = 1000
    assert g(*bad) == 3                                                                   # workspace too small
    bad = list(args); bad[12] = P((1 << 20) + 16)
    assert g(*bad) == 3                                                                   # workspace alignment
    assert lib.mxfp8_check_device_error(None, None, None) == 1
