"""The C ABI library loads and exports every function include/treeattn.h declares (CPU)."""
import ctypes

from dag_packed_paged_gb300 import _native, build


def test_library_exports_every_declared_function():
    build.build()
    lib = _native.lib()
    names = _native.header_functions()
    assert {"tree_attn_plan", "tree_attn_fwd", "tree_attn_bwd"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layouts_match_header(tmp_path):
    """Size and field offsets of every struct the binding mirrors, as the C compiler lays them
    out from include/treeattn.h."""
    import subprocess
    structs = {"ta_branch": _native.ta_branch, "ta_mount": _native.ta_mount, "ta_config": _native.ta_config,
               "ta_plan_stats": _native.ta_plan_stats, "ta_plan_arrays": _native.ta_plan_arrays}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "treeattn.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", build.INCLUDE, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split("\n")
    c = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}
    for name, cls in structs.items():
        assert c[(name, "size")] == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert c[(name, f)] == getattr(cls, f).offset, (name, f)
    from dag_packed_paged_gb300 import workloads as W
    assert W.BRANCH_DTYPE.itemsize == ctypes.sizeof(_native.ta_branch)
    assert W.MOUNT_DTYPE.itemsize == ctypes.sizeof(_native.ta_mount)


def test_binding_constants_match_header():
    """Every TA_* value #defined in the header has the same value in the Python binding."""
    import re
    text = open(build.INCLUDE + "/treeattn.h").read()
    defs = dict(re.findall(r"#define\s+(TA_\w+)\s+\(?(-?(?:0x)?[0-9a-fA-F]+)u?\)?", text))
    assert len(defs) == len(re.findall(r"#define\s+TA_", text)) >= 11
    for name, val in defs.items():
        assert hasattr(_native, name), name
        assert getattr(_native, name) == int(val, 0), name
