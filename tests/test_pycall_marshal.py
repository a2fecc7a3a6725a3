"""The C marshalling module passes each producer exactly the arguments the
ctypes declarations pass (CPU; no GPU, no CUDA library).

Both paths drive a stand-in library (tests/abi_stub.c) with the C ABI's
prototypes (include/nvfp4ap.h) that records every call's arguments; the
arguments are generated from the binding's ctypes declarations, so a swapped,
dropped or mistyped argument in csrc/pycall.c shows up as a differing record.
"""
import ctypes
import importlib.machinery
import importlib.util
import os
import subprocess

import pytest

import nvfp4_activation_producer_gb300 as ap
from nvfp4_activation_producer_gb300 import build as b

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def paths(tmp_path_factory):
    cmd = b.pycall_command()
    if cmd is None:
        pytest.skip("no Python headers or C compiler: the binding uses ctypes")
    d = tmp_path_factory.mktemp("pycall")
    stub = str(d / "libnvfp4ap_stub.so")
    subprocess.run([b.host_cc(), "-O1", "-shared", "-fPIC", "-I", b.INCLUDE, os.path.join(HERE, "abi_stub.c"),
                    "-o", stub], check=True)
    mod = str(d / os.path.basename(b.PYCALL))
    cmd[cmd.index("-o") + 1] = mod
    subprocess.run(cmd, check=True)
    return stub, mod


@pytest.fixture(scope="module")
def apis(paths):
    stub, mod = paths
    loader = importlib.machinery.ExtensionFileLoader("_pycall", mod)
    spec = importlib.util.spec_from_file_location("_pycall", mod, loader=loader)
    fast = importlib.util.module_from_spec(spec)
    loader.exec_module(fast)
    fast.bind(stub)
    L = ctypes.CDLL(stub)
    ap._declare(L)
    L.stub_last.restype = ctypes.c_int
    L.stub_last.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint64)]
    return ap._Api(L, None), ap._Api(L, fast), L


def last(L):
    name = ctypes.create_string_buffer(96)
    words = (ctypes.c_uint64 * 24)()
    n = L.stub_last(name, words)
    return name.value.decode(), list(words[:n])


def make_args(argtypes, seed, null_at=None):
    args = []
    for k, t in enumerate(argtypes):
        if t is ctypes.c_void_p:
            args.append(None if k == null_at else 0x10000 * (seed + 1) + 0x100 * k + 0x10)
        elif t is ctypes.c_int64:
            args.append(1000 * (seed + 1) + 7 * k - 3)
        elif t is ctypes.c_float:
            args.append(0.5 + 0.125 * k + seed)
        else:  # the six output pointers of the six-way producer
            args.append(tuple(0x7000000 + 0x1000 * j + seed for j in range(6)))
    return args


@pytest.mark.parametrize("name", ap._PRODUCERS)
def test_marshalling_matches_ctypes(apis, name):
    slow, fast, L = apis
    argtypes = getattr(L, name).argtypes
    for seed, null_at in ((0, None), (3, 0), (5, len(argtypes) - 1)):
        args = make_args(argtypes, seed, null_at)
        rc_slow = getattr(slow, name)(*args)
        rec_slow = last(L)
        rc_fast = getattr(fast, name)(*args)
        rec_fast = last(L)
        assert rec_slow[0] == name
        assert rec_fast == rec_slow, f"{name}: {rec_fast} != {rec_slow}"
        assert rc_fast == rc_slow and rc_slow >= 101


def test_every_header_producer_is_marshalled():
    # the producers: the header's entry points that take a stream
    import re
    hdr = re.sub(r"/\*.*?\*/", "", open(os.path.join(b.INCLUDE, "nvfp4ap.h")).read(), flags=re.S)
    producers = set()
    for m in re.finditer(r"^int\s+([A-Za-z_0-9]+)\s*\(([^;]*)\);", hdr, flags=re.M):
        if "nvfp4ap_stream_t" in m.group(2):
            producers.add(m.group(1))
    src = open(b.PYCALL_SRC).read()
    listed = set(re.findall(r"X\(([A-Za-z_0-9]+)\)", src))
    wrapped = set(re.findall(r"^BEGIN\(([A-Za-z_0-9]+),", src, flags=re.M))
    assert producers and listed == producers == wrapped
    assert set(ap._PRODUCERS) <= listed


def test_bad_arguments_raise_before_the_call(apis):
    _, fast, L = apis
    name = "ada_layer_norm_quant_fp8_bf16"
    args = make_args(getattr(L, name).argtypes, 9)
    getattr(fast, name)(*args)
    before = last(L)
    with pytest.raises(TypeError):
        getattr(fast, name)(*args[:-1])               # one argument short
    with pytest.raises(TypeError):
        getattr(fast, name)(*(args[:6] + [1.5] + args[7:]))   # a float for rows
    with pytest.raises(TypeError):
        getattr(fast, name)(*(["x"] + args[1:]))      # a string for a pointer
    with pytest.raises(ValueError):
        fast.adaln_modulation6_bf16(1, 2, (1, 2, 3), 1, 2, 3, 4)   # five outputs too few
    assert last(L) == before
