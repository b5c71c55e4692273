"""CPU checks of the C ABI: the library builds, loads, and exports every declared symbol;
host-side argument checks refuse bad calls before any launch (no GPU needed for those)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    from dspark_draft_selection_gb300.build import LIB, build
    if not os.path.exists(LIB):
        build()
    return LIB


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dspark_topk", "dspark_lattice_score", "dspark_chain_select", "dspark_dense_walk",
              "dspark_sample", "dspark_verify", "dspark_d2t_check", "dspark_workspace_size",
              "dspark_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dspark_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(libpath)
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_binding_signatures_cover_the_header(libpath):
    from dspark_draft_selection_gb300._binding import SIGNATURES
    assert sorted(n for n, _, _ in SIGNATURES) == declared_functions()


def test_status_strings_and_host_checks(libpath):
    import dspark_draft_selection_gb300 as ds
    lib = ds.lib()
    assert ds.dspark_status_string(0) == "ok"
    assert "range" in ds.dspark_status_string(2)
    # null pointers and bad sizes are refused on the host, before any launch
    assert lib.dspark_topk(None, 0, 1, 1, 10, 10, None, 8, 1.0, 0.0, None, 10, None, None, None, None, None) == 1
    fake = ctypes.c_void_p(256)
    assert lib.dspark_topk(fake, 0, 1, 1, 10, 10, None, 65, 1.0, 0.0, None, 10, fake, fake, fake, fake, None) == 1
    assert lib.dspark_topk(fake, 7, 1, 1, 10, 10, None, 8, 1.0, 0.0, None, 10, fake, fake, fake, fake, None) == 1
    assert lib.dspark_topk(fake, 0, 1, 1, 10, 9, None, 8, 1.0, 0.0, None, 10, fake, fake, fake, fake, None) == 1  # ld < V_d
    # an empty batch is a no-op that launches nothing
    assert lib.dspark_topk(fake, 0, 0, 1, 10, 10, None, 8, 1.0, 0.0, None, 10, fake, fake, fake, fake, None) == 0
    assert ds.dspark_workspace_size(ds.OP_TOPK, 32, 7, 151936, 64) == 0
    assert lib.dspark_chain_select(fake, fake, fake, 1, 7, 65, 0, 0.0, 1.0, 0.0, None, None, None, None, None, None, fake,
                                   fake, fake, None,
                                   fake, None) == 1
    assert lib.dspark_d2t_check(fake, 10, 10, 1, None, 0, fake, None) == 8      # injectivity needs a workspace
    # grouped convolution: channels not a multiple of the groups, too many taps, no-op on zero rows
    assert lib.dspark_grouped_conv(fake, 0, 4, 10, 10, 3, 4, fake, fake, fake, 10, None) == 1
    assert lib.dspark_grouped_conv(fake, 0, 4, 12, 12, 3, 17, fake, fake, fake, 12, None) == 1
    assert lib.dspark_grouped_conv(None, 0, 0, 12, 12, 3, 4, None, None, None, 12, None) == 0
    assert ds.dspark_workspace_size(ds.OP_D2T_CHECK, 1, 1, 64, 0) >= 8
    # the sampler's optional weight scratch: whole 256-byte rows of V floats, none for an empty row
    ws_s = ds.dspark_workspace_size(ds.OP_SAMPLE, 16, 15, 114688, 0)
    assert ws_s > 0 and ws_s % 256 == 0 and ws_s % (114688 * 4) == 0
    assert ds.dspark_workspace_size(ds.OP_SAMPLE, 16, 15, 0, 0) == 0
