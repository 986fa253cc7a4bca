"""The C-ABI library loads and exports every function include/purlin.h declares
(no GPU needed; nothing here calls into the device)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "purlin.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(purlin_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def P():
    import __graft_entry__

    __graft_entry__.build()
    import collective_datapath_atom_gb300 as P

    return P


def test_header_declares_the_collectives():
    names = declared_functions()
    for n in ("purlin_init", "purlin_finalize", "purlin_all_reduce", "purlin_reduce_scatter",
              "purlin_all_gather", "purlin_all_to_all", "purlin_all_gather_v",
              "purlin_reduce_scatter_v", "purlin_all_to_all_v", "purlin_check",
              "purlin_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(P):
    names = declared_functions()
    lib = ctypes.CDLL(P.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    nm = subprocess.run(["nm", "-D", "--defined-only", P.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(line.split()[-1] for line in nm.splitlines() if line.strip())
    assert set(names) <= exported
    # the binding marshals exactly the declared set
    assert set(P._SIGNATURES) == set(names)


def test_status_strings(P):
    for s in range(0, 8):
        assert P.status_string(s)
    assert P.status_string(99) == "unknown status"


def test_init_without_a_gpu_fails_cleanly(P):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(0)
    st = P.lib.purlin_init(8, None, ctypes.byref(h))
    assert st == P.PURLIN_ERR_CUDA and not h.value
    assert P.lib.purlin_init(0, None, ctypes.byref(h)) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_init(65, None, ctypes.byref(h)) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_finalize(None) == P.PURLIN_OK
    assert P.lib.purlin_check(None) == P.PURLIN_ERR_INVALID_ARG


def test_library_does_not_link_the_oracle(P):
    deps = subprocess.run(["nm", "-D", P.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle_" not in deps


def test_device_coll_layout_matches_the_library(P):
    """The binding's purlin_device_coll has the size the library was built with."""
    assert ctypes.sizeof(P.purlin_device_coll) == P.lib.purlin_device_coll_size()
    # the C layout: two pointer arrays of PURLIN_MAX_RANKS, then the fields
    assert P.purlin_device_coll.segs.offset == 2 * 8 * P.PURLIN_MAX_RANKS


EXAMPLES_HEADER = os.path.join(ROOT, "collective_datapath_atom_gb300", "examples",
                               "device_examples.h")


def test_examples_library_exports_its_header():
    """The device-API example kernels' library exports what its header declares,
    and its binding marshals exactly that set."""
    import __graft_entry__

    __graft_entry__.build()
    from collective_datapath_atom_gb300 import examples

    text = re.sub(r"/\*.*?\*/", "", open(EXAMPLES_HEADER).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(purlin_[a-z_0-9]+)\s*\(", text)))
    assert names, "no declarations found"
    nm = subprocess.run(["nm", "-D", "--defined-only", examples.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(line.split()[-1] for line in nm.splitlines() if line.strip())
    assert set(names) <= exported
    assert set(examples._SIGNATURES) == set(names)


def test_new_entry_points_refuse_bad_arguments_before_any_launch(P):
    """Argument checks that return before the GPU is touched (they run here
    without a GPU): the touch floor needs two 16-byte aligned pointers, and a
    packet channel needs a context, a capacity and a CTA count in range."""
    vp = ctypes.c_void_p
    assert P.lib.purlin_touch_launch(None, vp(0x1000), None) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_touch_launch(vp(0x1000), None, None) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_touch_launch(vp(0x1008), vp(0x2000), None) == P.PURLIN_ERR_ALIGNMENT
    assert P.lib.purlin_touch_launch(vp(0x1000), vp(0x2004), None) == P.PURLIN_ERR_ALIGNMENT
    ch = P.purlin_packet_channel()
    assert P.lib.purlin_packet_channel_create(None, 4096, 2, ctypes.byref(ch)) == \
        P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_packet_channel_check(None, None) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_packet_channel_check(ctypes.byref(ch), None) == P.PURLIN_ERR_INVALID_ARG
    assert P.lib.purlin_packet_channel_release(None, ctypes.byref(ch)) == P.PURLIN_ERR_INVALID_ARG


def test_packet_channel_layout_matches_the_header():
    """The binding's struct mirrors include/purlin.h field for field."""
    import collective_datapath_atom_gb300 as P

    names = [f for f, _ in P.purlin_packet_channel._fields_]
    assert names == ["staging", "state", "capacity", "timeout_ns", "drop_unit", "ctas", "pad",
                     "owner"]
    assert ctypes.sizeof(P.purlin_packet_channel) == 56
    with open(os.path.join(ROOT, "include", "purlin.h")) as f:
        text = f.read()
    body = text[text.index("typedef struct purlin_packet_channel"):]
    body = body[:body.index("} purlin_packet_channel;")]
    declared = re.findall(r"\b(\w+);", body)
    assert declared == names
