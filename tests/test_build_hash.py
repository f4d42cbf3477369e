"""The code hash that keeps a committed DRAM-traffic capture tied to the code it was taken on."""
from predicted_token_importance_tb_b300 import build


def test_strip_comments_keeps_code_and_literals():
    a = 'int a = 1; // note\n/* block\n comment */ const char *s = "// not a comment /* */";\nchar c = \'\\\'\';'
    b = 'int a = 1;\nconst char *s = "// not a comment /* */"; char c = \'\\\'\';'
    assert build.strip_comments(a) == build.strip_comments(b)
    assert '"// not a comment /* */"' in build.strip_comments(a)


def test_strip_comments_sees_code_changes():
    assert build.strip_comments("x = a + b; // sum") != build.strip_comments("x = a - b; // sum")
    assert build.strip_comments('s = "a//b";') != build.strip_comments('s = "a";')


def test_code_hash_is_stable():
    assert build.code_hash() == build.code_hash()
    assert len(build.code_hash()) == 64
