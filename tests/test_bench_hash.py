"""The kernel hash that keys the recorded ncu traffic ignores comments and layout only."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = '''// leading comment
__global__ void k(int* p) {  /* block
   comment */ p[0] = 1;  // trailing
  asm("add.s32 %0, %0, 1; // not a comment" : "+r"(p[1]));
  char c = '/';
}
'''


def test_comments_and_layout_do_not_change_the_tokens():
    edited = SRC.replace("// trailing", "// another remark, much longer").replace(
        "/* block\n   comment */", "/* x */").replace("{  ", "{\n\n    ")
    assert bench.code_tokens(edited) == bench.code_tokens(SRC)


def test_code_changes_and_string_contents_do():
    assert bench.code_tokens(SRC.replace("p[0] = 1", "p[0] = 2")) != bench.code_tokens(SRC)
    toks = bench.code_tokens(SRC)
    assert "// not a comment" in toks and "leading" not in toks and "trailing" not in toks
    assert "'/'" in toks


def test_kernel_sources_hash():
    h = bench.kernel_source_hash(["decode.cuh", "ptx.cuh"])
    assert len(h) == 16 and int(h, 16) >= 0
