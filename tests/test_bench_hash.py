"""bench.py's kernel hash (which decides whether the committed ncu traffic
still describes the attention kernel) ignores comments and whitespace but
not code (CPU only)."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _hash_of(tmp_path, edit):
    csrc = tmp_path / "speculative_decoding_verify_mla_gb300" / "csrc"
    csrc.mkdir(parents=True)
    import bench
    for fn in bench.ATTENTION_SOURCES:
        shutil.copy(os.path.join(ROOT, "speculative_decoding_verify_mla_gb300", "csrc", fn), csrc / fn)
    edit(csrc / bench.ATTENTION_SOURCES[0])
    old = bench.ROOT
    bench.ROOT = str(tmp_path)
    try:
        return bench.kernel_source_hash()
    finally:
        bench.ROOT = old


def test_hash_ignores_comments_not_code(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    base = bench.kernel_source_hash()

    def add_comments(p):
        p.write_text("// a new line comment\n/* and a\n block comment */\n" + p.read_text().replace("\n", "  \n", 3))

    def change_code(p):
        p.write_text(p.read_text().replace("kRescaleThreshold = 8.0f", "kRescaleThreshold = 7.0f", 1))

    assert _hash_of(tmp_path / "a", add_comments) == base
    assert _hash_of(tmp_path / "b", change_code) != base
