"""Build-script host logic: the kernel source digest that ties a committed
ncu traffic record to the kernel sources it was captured on."""
from bmm_reducescatter_alltoall_gb300._build import code_text

SRC = b"""// header comment
#define TILE  128   /* rows */
__global__ void k(int* p) {
    /* block
       comment */
    const char* s = "a // not a comment /* nor this */";
    char q = '"';
    p[0] = TILE;  // trailing
}
"""


def test_comment_and_whitespace_edits_keep_the_code_text():
    edited = SRC.replace(b"// header comment", b"// another header comment\n\n")
    edited = edited.replace(b"/* rows */", b"/* rows of a tile */")
    edited = edited.replace(b"    p[0]", b"\tp[0]")
    assert code_text(edited) == code_text(SRC)


def test_code_edits_change_the_code_text():
    for a, b in [(b"TILE  128", b"TILE  256"), (b"p[0] = TILE", b"p[1] = TILE"),
                 (b"a // not", b"a / / not"), (b"'\"'", b"'x'")]:
        assert a in SRC
        assert code_text(SRC.replace(a, b)) != code_text(SRC), a


def test_literals_survive_and_comments_go():
    t = code_text(SRC)
    assert b'"a // not a comment /* nor this */"' in t
    assert b"header comment" not in t and b"trailing" not in t and b"block" not in t
    assert b"#define TILE 128\n" in t


def test_digest_follows_the_included_headers(tmp_path):
    from bmm_reducescatter_alltoall_gb300._build import included_files
    (tmp_path / "k.cu").write_text('#include "a.h"\n// #include "gone.h"\nint k;\n')
    (tmp_path / "a.h").write_text('#pragma once\n#include "b.h"\n/* #include "c.h" */\n')
    (tmp_path / "b.h").write_text('#include "a.h"\nint b;\n')
    (tmp_path / "c.h").write_text("int c;\n")
    names = [p.rsplit("/", 1)[-1] for p in included_files(str(tmp_path / "k.cu"))]
    assert names == ["k.cu", "a.h", "b.h"]        # commented includes and cycles handled
