"""Host checks of the bench's profile bookkeeping: a committed ncu summary's
traffic is reported only while the kernel source it was taken on is unchanged
(comments and whitespace aside)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = """// row loop
__global__ void k(float *x) {
    /* one element per thread */
    x[threadIdx.x] *= 2.0f;
}
"""


def _write(path, text):
    with open(path, "w", encoding="utf-8") as f:
        f.write(text)


def test_hash_ignores_comments_and_whitespace(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cu"
    _write(a, SRC)
    _write(b, SRC.replace("// row loop", "// rows, one at a time").replace("    x[", "\tx[")
           .replace("/* one element per thread */", "/* a\n multi-line\n comment */"))
    assert bench.kernel_source_hash([str(a)]) == bench.kernel_source_hash([str(b)])


def test_hash_changes_with_code_and_with_file_boundaries(tmp_path):
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    _write(a, SRC)
    _write(b, SRC.replace("2.0f", "3.0f"))
    assert bench.kernel_source_hash([str(a)]) != bench.kernel_source_hash([str(b)])
    # the same text split differently over two files is another source set
    _write(b, SRC[:40])
    _write(c, SRC[40:])
    assert bench.kernel_source_hash([str(b), str(c)]) != bench.kernel_source_hash([str(a)])


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    _write(src, SRC)
    (tmp_path / "profiles").mkdir()
    summary = tmp_path / "profiles" / "k_case.md"
    h = bench.kernel_source_hash([str(src)])
    _write(summary, "counters\n\ntraffic_bytes_per_launch: 123456\nkernel_source_sha256_16: %s\n" % h)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.PROFILED_SRCS, "k_kernel", [str(src)])
    assert bench.profiled_traffic("k_case.md", "k_kernel") == 123456.0
    _write(src, SRC.replace("// row loop", "// comment edits keep the counters"))
    assert bench.profiled_traffic("k_case.md", "k_kernel") == 123456.0
    _write(src, SRC.replace("*= 2.0f", "+= 1.0f"))
    assert bench.profiled_traffic("k_case.md", "k_kernel") is None
    assert bench.profiled_traffic("missing.md", "k_kernel") is None


def test_every_profiled_kernel_names_existing_sources():
    for kernel, srcs in bench.PROFILED_SRCS.items():
        assert srcs, kernel
        for p in srcs:
            assert os.path.isfile(p), (kernel, p)
