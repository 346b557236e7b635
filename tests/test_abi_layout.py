"""The ctypes structures of the Python binding have the C header's layout:
a small C program built against include/si_moe.h prints sizeof and offsetof
of every field, and the binding's ctypes.Structure must agree."""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

from quantized_moe_expert_gemv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = {
    "si_moe_desc": binding.si_moe_desc,
    "si_moe_layer": binding.si_moe_layer,
    "si_moe_route_out": binding.si_moe_route_out,
}


def _c_layout(tmp_path) -> dict:
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "si_moe.h"', "int main(void) {"]
    for name, cls in STRUCTS.items():
        lines.append(f'    printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'    printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for line in out.splitlines():
        name, key, value = line.split()
        got[(name, key)] = int(value)
    return got


def test_binding_structs_match_the_c_header(tmp_path):
    try:
        c = _c_layout(tmp_path)
    except (OSError, subprocess.CalledProcessError) as exc:  # no C compiler on this host
        pytest.skip(f"cannot build the layout probe: {exc}")
    for name, cls in STRUCTS.items():
        assert c[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert c[(name, field)] == getattr(cls, field).offset, (name, field)


def test_binding_constants_match_the_c_header(tmp_path):
    """Every SI_* constant the header defines (status codes, weight types,
    flags, modes, limits) has the same value in the binding: a small C program
    built against include/si_moe.h prints them."""
    import re
    with open(os.path.join(ROOT, "include", "si_moe.h")) as f:
        text = f.read()
    names = sorted(set(re.findall(r"^#define (SI_[A-Z0-9_]+) ", text, flags=re.M)) |
                   set(re.findall(r"^\s+(SI_(?:OK|ERR_[A-Z_]+)) =", text, flags=re.M)))
    assert {"SI_OK", "SI_ERR_RANGE", "SI_MODE_DECODE_HOST", "SI_STATIC_SCRATCH_BYTES"} <= set(names)
    lines = ['#include <stdio.h>', '#include "si_moe.h"', "int main(void) {"]
    lines += [f'    printf("{n} %lld\\n", (long long)({n}));' for n in names]
    lines += ["    return 0;", "}"]
    src = tmp_path / "consts.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "consts"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict((k, int(v)) for k, v in (line.split() for line in out.splitlines()))
    for n in names:
        assert hasattr(binding, n), f"binding lacks {n}"
        assert getattr(binding, n) == got[n], n
