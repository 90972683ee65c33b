"""CPU checks of the C ABI: the library builds, loads and exports every declared symbol, and
host-side argument validation rejects bad calls before anything reaches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dcp.h")


@pytest.fixture(scope="module")
def lib():
    from decode_context_paged_gb300 import _build
    _build.build()
    import decode_context_paged_gb300 as dcp
    return dcp.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dcp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("dcp_reshard_pages", "dcp_partial_decode_attn", "dcp_lse_merge"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dcp.h but not exported"


def test_status_strings_and_version(lib):
    import decode_context_paged_gb300 as dcp
    assert dcp.version() >= 10000
    assert dcp.status_string(0) == "ok"
    assert "workspace" in dcp.status_string(-4)
    assert dcp.device_error_status(0) == 0
    assert dcp.device_error_status(dcp.DEVERR_TIMEOUT | dcp.DEVERR_OUT_OF_RANGE) == -6
    assert dcp.device_error_status(dcp.DEVERR_OUT_OF_RANGE) == -2


def test_layer_range_worked_example(lib):
    import decode_context_paged_gb300 as dcp
    got = [dcp.layer_range(78, 8, r) for r in range(8)]
    assert got == [(0, 10), (10, 20), (20, 30), (30, 40), (40, 50), (50, 60), (60, 69), (69, 78)]
    s = ctypes.c_int()
    assert lib.dcp_layer_range(8, 0, 0, ctypes.addressof(s), ctypes.addressof(s)) == -1
    assert lib.dcp_layer_range(8, 4, 4, ctypes.addressof(s), ctypes.addressof(s)) == -1


def test_host_validation_rejects_bad_arguments(lib):
    null = None
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # merge: bad part count, bad width, unaligned
    assert lib.dcp_lse_merge(0, 10, 512, fake, fake, fake, fake, null) == -1
    assert lib.dcp_lse_merge(2, 10, 500, fake, fake, fake, fake, null) == -1
    assert lib.dcp_lse_merge(2, 10, 512, ctypes.c_void_p(0x1004), fake, fake, fake, null) == -1
    assert lib.dcp_lse_merge(2, 0, 512, null, null, null, null, null) == 0  # nothing to do
    # reshard: page size, row width, rank counts, path coordinates
    ptrs = (ctypes.c_void_p * 1)(0x1000)
    args = [1, fake, 4, fake, fake, 64, 576, 0, 1, 1, ctypes.addressof(ptrs), 4, 1,
            ctypes.addressof(ptrs), 4, -1, -1, null, null]
    bad = list(args); bad[5] = 32
    assert lib.dcp_reshard_pages(*bad) == -1
    bad = list(args); bad[6] = 512
    assert lib.dcp_reshard_pages(*bad) == -1
    bad = list(args); bad[9] = 0
    assert lib.dcp_reshard_pages(*bad) == -1
    bad = list(args); bad[16] = 3
    assert lib.dcp_reshard_pages(*bad) == -1
    bad = list(args); bad[7] = 7
    assert lib.dcp_reshard_pages(*bad) == -1
    # filter: rank outside [0, n_dcp)
    assert lib.dcp_filter_page_indices(4, fake, null, 4, 4, fake, null, fake, null) == -1
    assert lib.dcp_filter_page_indices(4, fake, fake, 4, 0, fake, null, fake, null) == -1
    # attention: shape checks that need no device
    kv = (ctypes.c_void_p * 1)(0x1000)
    a = [1, 1, 64, fake, fake, fake, 4, fake, 64, 0, ctypes.c_float(1.0), ctypes.c_float(0.07), 1,
         ctypes.addressof(kv), 4, -1, fake, fake, fake, ctypes.c_size_t(1 << 20), null, null]
    bad = list(a); bad[8] = 128
    assert lib.dcp_partial_decode_attn(*bad) == -1
    bad = list(a); bad[12] = 0
    assert lib.dcp_partial_decode_attn(*bad) == -1
    bad = list(a); bad[12] = 17
    assert lib.dcp_partial_decode_attn(*bad) == -1
    bad = list(a); bad[1] = 0
    assert lib.dcp_partial_decode_attn(*bad) == -1
    bad = list(a); bad[11] = ctypes.c_float(0.0)
    assert lib.dcp_partial_decode_attn(*bad) == -1
    bad = list(a); bad[9] = 1; bad[10] = ctypes.c_float(0.0)
    assert lib.dcp_partial_decode_attn(*bad) == -1
