"""The Python binding declares every C entry point with the argument list the
header gives it: the same number of arguments, each of the same kind
(pointer, 32-bit or 64-bit integer, float, size), and the same return kind;
and the statistics structure has the header's fields in the header's order.
ctypes converts arguments by the declared types without looking at the
library, so a binding that drifted from include/pa.h would pass wrong values
silently.  And the in-tree build loads only a library built for this
host's machine.  CPU only: the header is parsed as text and nothing is
called."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_124_gb300 import api

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


def _header_text():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return re.sub(r"//[^\n]*", " ", text)


def _c_kind(decl):
    """The kind of one C parameter or return declaration."""
    decl = decl.strip()
    if "*" in decl:
        return "ptr"
    words = decl.replace("const ", "").split()
    base = words[0] if words else ""
    return {"int": "i32", "int32_t": "i32", "int64_t": "i64", "uint64_t": "u64", "size_t": "u64",
            "float": "f32", "void": None}[base]


def _ctypes_kind(t):
    if t is None:
        return None
    if t in (ctypes.c_void_p, ctypes.c_char_p) or issubclass(t, ctypes._Pointer):
        return "ptr"
    size = ctypes.sizeof(t)
    if t is ctypes.c_float:
        return "f32"
    if t in (ctypes.c_int, ctypes.c_int32):
        return "i32"
    if size == 8 and t(-1).value < 0:
        return "i64"
    if size == 8:
        return "u64"
    raise AssertionError("unexpected ctypes type %r" % t)


def _prototypes():
    """name -> (return kind, [parameter kinds]) for every function the header declares."""
    protos = {}
    pat = re.compile(r"([A-Za-z_][A-Za-z0-9_ ]*?\**)\s*\b(pa_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", re.S)
    for ret, name, params in pat.findall(_header_text()):
        params = " ".join(params.split())
        kinds = [] if params in ("", "void") else [_c_kind(p.rsplit(" ", 1)[0] if not p.strip().endswith("*")
                                                           else p) for p in params.split(",")]
        protos[name] = (_c_kind(ret.split()[-1] if "*" not in ret else ret), kinds)
    return protos


def test_header_parses_into_every_declared_function():
    protos = _prototypes()
    assert sorted(protos) == api.header_functions()
    assert protos["pa_decode"][0] == "i32" and len(protos["pa_decode"][1]) == 21
    assert protos["pa_alloc_create"] == ("ptr", ["i32", "i32"])
    assert protos["pa_version"] == ("ptr", [])


@pytest.mark.parametrize("name", sorted(_prototypes()))
def test_binding_matches_the_header(name):
    ret, kinds = _prototypes()[name]
    assert name in api._SIGS, "%s is declared in include/pa.h but has no binding" % name
    b_ret, b_args = api._SIGS[name]
    assert _ctypes_kind(b_ret) == ret, "%s returns %s in the header" % (name, ret)
    got = [_ctypes_kind(a) for a in b_args]
    assert got == kinds, "%s: header %s, binding %s" % (name, kinds, got)


def test_binding_declares_nothing_the_header_does_not():
    assert set(api._SIGS) <= set(_prototypes())


def test_stats_structure_matches_the_header():
    body = re.search(r"typedef struct pa_alloc_stats \{(.*?)\} pa_alloc_stats_t;", _header_text(), re.S).group(1)
    fields = [tuple(f.split()) for f in body.split(";") if f.strip()]
    want = [(name, {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64}[t]) for t, name in fields]
    assert [(n, t) for n, t in api.AllocStats._fields_] == want


def test_build_freshness_checks_the_library_machine():
    """The in-tree build counts a library as current only if it is a 64-bit
    little-endian ELF object for this host's machine, so a library built on
    the other architecture is rebuilt rather than loaded."""
    from paged_kv_cache_124_gb300 import build as b

    def elf(machine, cls=2, data=1):
        return b"\x7fELF" + bytes([cls, data]) + bytes(12) + machine.to_bytes(2, "little")

    assert b.elf_matches_host(elf(62), "x86_64") and not b.elf_matches_host(elf(183), "x86_64")
    assert b.elf_matches_host(elf(183), "aarch64") and not b.elf_matches_host(elf(62), "aarch64")
    assert not b.elf_matches_host(elf(62, cls=1), "x86_64")          # 32-bit
    assert not b.elf_matches_host(elf(62, data=2), "x86_64")         # big-endian
    assert not b.elf_matches_host(b"#!/bin/sh\n" + bytes(10), "x86_64")
    assert not b.elf_matches_host(elf(62)[:19], "x86_64")
    assert not b.elf_matches_host(elf(62), "riscv64")                # no library for an unknown machine
    with open(b.LIB, "rb") as f:
        assert b.elf_matches_host(f.read(20))                       # the library built here
