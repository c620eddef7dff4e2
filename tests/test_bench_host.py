"""Host-side logic of bench.py that needs no GPU: the key its recorded GEMM traffic is filed
under ignores comments and blank lines but changes with any code edit."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _key_with(tmp_path, edit):
    """bench.gemm_source_hash() on a copy of the kernel sources with gemm_tc.cu edited."""
    csrc = tmp_path / "matrix_orthogonalizing_optimizer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("gemm_tc.cu", "common.cuh"):
        shutil.copy(os.path.join(ROOT, "matrix_orthogonalizing_optimizer_gb300", "csrc", f), csrc / f)
    p = csrc / "gemm_tc.cu"
    p.write_text(edit(p.read_text()))
    old = bench.ROOT
    bench.ROOT = str(tmp_path)
    try:
        return bench.gemm_source_hash()
    finally:
        bench.ROOT = old


def test_source_key_ignores_comments(tmp_path):
    base = bench.gemm_source_hash()
    assert _key_with(tmp_path / "a", lambda s: s) == base
    assert _key_with(tmp_path / "b", lambda s: "// a new comment line\n" + s) == base
    assert _key_with(tmp_path / "c", lambda s: s.replace("\n", "\n\n", 5)) == base
    assert _key_with(tmp_path / "d", lambda s: "/* a block\n   comment */\n" + s) == base


def test_source_key_follows_code(tmp_path):
    base = bench.gemm_source_hash()
    assert _key_with(tmp_path / "e", lambda s: s.replace("constexpr int SCALE_NPART = 32;",
                                                        "constexpr int SCALE_NPART = 16;")) != base
    assert _key_with(tmp_path / "f", lambda s: s + "\nstatic int unused_marker = 0;\n") != base

