"""bench.py's key for the committed DRAM-traffic records: the digest of a
kernel's code follows code edits and ignores comment edits."""
import bench

SRC = {
    "k6_attn_single.cu": 'int f(int x) { return x + 1; }  // add one\n/* block\n comment */\nconst char *s = "a//b /* c */";\n',
    "k6_attn_common.cuh": "#define N 3\n",
    "k6_device.cuh": "// nothing\n",
}


def digest(files):
    return bench.source_digest("attn_tc_single_kernel", read=lambda name: files[name])


def test_strip_comments_keeps_code_and_string_literals():
    out = bench.strip_comments(SRC["k6_attn_single.cu"])
    assert "add one" not in out and "block" not in out
    assert "return x + 1;" in out
    assert '"a//b /* c */"' in out          # comment markers inside a string stay
    assert bench.strip_comments("char c = '/'; // x\n") == "char c = '/'; \n"


def test_comment_edits_keep_the_digest():
    base = digest(SRC)
    edited = dict(SRC)
    edited["k6_attn_single.cu"] = "// a new header\n// over two lines\n\n" + SRC["k6_attn_single.cu"].replace(
        "add one", "increment")
    assert digest(edited) == base


def test_code_edits_change_the_digest():
    base = digest(SRC)
    for name, old, new in (("k6_attn_single.cu", "x + 1", "x + 2"), ("k6_attn_common.cuh", "N 3", "N 4"),
                           ("k6_attn_single.cu", "a//b", "a//c")):
        edited = dict(SRC)
        edited[name] = SRC[name].replace(old, new)
        assert digest(edited) != base, (name, old, new)
