"""The binding's ctypes mirrors of the C-ABI structs have the header's layout:
a small C program compiled against include/moe_layout.h prints every struct's
size and every field's offset, and each must equal the ctypes structure's.
CPU only (gcc)."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _mirrors():
    import combine_moe_layout_04_gb300 as moe
    return {"moe_tuning": moe._TuningC, "moe_problem": moe._ProblemC,
            "moe_layout_t": moe._LayoutC, "moe_relay_t": moe._RelayC}


def _c_layout(tmp_path, mirrors):
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe_layout.h"', "int main(void) {"]
    for cname, cls in mirrors.items():
        lines.append(f'    printf("{cname} %zu\\n", sizeof({cname}));')
        for field, _ in cls._fields_:
            lines.append(f'    printf("{cname}.{field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_ctypes_mirrors_match_the_header(tmp_path):
    mirrors = _mirrors()
    c = _c_layout(tmp_path, mirrors)
    for cname, cls in mirrors.items():
        assert ctypes.sizeof(cls) == c[cname], cname
        for field, _ in cls._fields_:
            assert getattr(cls, field).offset == c[f"{cname}.{field}"], (cname, field)


def test_header_fields_all_mirrored():
    """Every field the header declares in these structs has a ctypes field of
    the same name, in the same order."""
    import re
    text = open(os.path.join(ROOT, "include", "moe_layout.h")).read()
    for cname, cls in _mirrors().items():
        body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (cname, cname), text, re.S).group(1)
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        names = []
        for decl in body.split(";"):
            decl = decl.strip()
            if not decl:
                continue
            for part in decl.split(","):
                m = re.search(r"(\w+)\s*(\[\s*\w+\s*\])?\s*$", part.strip())
                names.append(m.group(1))
        assert names == [f for f, _ in cls._fields_], (cname, names)


def test_num_hosts_is_the_last_named_header_word():
    """The layout kernel's two record blocks write disjoint header words; the
    one that writes the sizes also zeroes every word after MOE_ST_NUM_HOSTS,
    so no named word may follow it."""
    import re
    text = open(os.path.join(ROOT, "include", "moe_layout.h")).read()
    body = re.search(r"MOE_ST_STATUS = 0,(.*?)\};", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = [n.strip() for n in body.split(",") if n.strip()]
    assert names[-1] == "MOE_ST_NUM_HOSTS", names[-3:]
