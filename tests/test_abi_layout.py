"""The ctypes mirrors of the C-ABI structs match the headers: the same fields in the same order, at the
same offsets, with the same total size, as a C compiler lays them out from include/*.h.  (A field added
to a header but not to the binding, or the other way round, would shift every later field silently.)"""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from speculative_decoding_verify_decode_gb300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")

STRUCTS = [("sd_shape", "sd_verify.h", native.SdShape), ("sd_gdn_shape", "sd_gdn.h", native.SdGdnShape)]


def header_fields(struct: str, header: str) -> list[str]:
    text = open(os.path.join(INC, header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef\s+struct\s+" + struct + r"\s*\{(.*?)\}\s*" + struct + r"\s*;", text, flags=re.S)
    assert body, f"{struct} not found in {header}"
    names = []
    for decl in body.group(1).split(";"):
        decl = decl.strip()
        if decl:
            names.append(re.findall(r"[A-Za-z_]\w*", decl)[-1])
    return names


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
@pytest.mark.parametrize("struct,header,cls", STRUCTS, ids=[s[0] for s in STRUCTS])
def test_ctypes_mirror_matches_the_header(tmp_path, struct, header, cls):
    names = header_fields(struct, header)
    assert names == [f[0] for f in cls._fields_]
    offs = " ".join(f'printf(" %zu", offsetof({struct}, {n}));' for n in names)
    src = tmp_path / "layout.c"
    src.write_text(f'#include <stddef.h>\n#include <stdio.h>\n#include "{header}"\n'
                   f'int main(void) {{ printf("%zu", sizeof({struct})); {offs} printf("\\n"); return 0; }}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", INC, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got[0] == ctypes.sizeof(cls)
    assert got[1:] == [getattr(cls, n).offset for n in names]


def test_with_ctx_stable_sets_only_the_flag():
    base = native.Shape([0, 9, 32], max_pages_per_seq=300, num_pool_pages=700, num_splits=5, window=2048)
    stable = base.with_ctx_stable()
    names = [f[0] for f in native.SdShape._fields_]
    for n in names:
        if n in ("q_indptr_h", "ctx_stable"):
            continue
        assert getattr(stable.c, n) == getattr(base.c, n), n
    assert list(stable.indptr) == list(base.indptr)
    assert base.c.ctx_stable == 0 and stable.c.ctx_stable == 1
    assert stable.with_ctx_stable(False).c.ctx_stable == 0


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_header_constants_match_the_binding(tmp_path):
    """Constants the binding copies from sd_verify.h, as a C compiler evaluates them."""
    consts = {"SD_NOALLOC_SCRATCH_BYTES": native.NOALLOC_SCRATCH_BYTES, "SD_MAX_NODES": native.MAX_NODES,
              "SD_MAX_BATCH": native.MAX_BATCH, "SD_MAX_LAYERS": native.MAX_LAYERS,
              "SD_DEV_TIMEOUT": native.SD_DEV_TIMEOUT, "SD_DEV_BAD_PAGE": native.SD_DEV_BAD_PAGE}
    prints = " ".join(f'printf(" %llu", (unsigned long long)({k}));' for k in consts)
    src = tmp_path / "consts.c"
    src.write_text(f'#include <stdio.h>\n#include "sd_verify.h"\nint main(void) {{ {prints} printf("\\n"); return 0; }}\n')
    exe = tmp_path / "consts"
    subprocess.run(["gcc", "-std=c11", "-I", INC, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert got == list(consts.values())
