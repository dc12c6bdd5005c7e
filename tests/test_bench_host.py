"""Host-side logic of bench.py that needs no GPU: the code-only source hash
that decides whether the recorded ncu traffic figures still describe the
kernels, and its scope (the encoder's and decoder's translation units)."""
import os
import shutil

import bench


def _copy_sources(tmp_path):
    src = os.path.join(bench.ROOT, "bit_gradient_communication_gb300", "csrc")
    dst = tmp_path / "bit_gradient_communication_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o"))
    return dst


def test_code_only_drops_comments_and_layout():
    a = "int x = 1; // one\n/* block\n comment */ float y;\n"
    b = "int   x = 1;\nfloat y;   // other words\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")


def test_traffic_hash_follows_only_the_two_kernels(tmp_path, monkeypatch):
    dst = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    full0 = bench.kernel_src_hash()
    scoped0 = bench.kernel_src_hash(bench.TRAFFIC_SOURCES)
    assert full0 != scoped0

    # a comment edit in an encoder source changes neither hash
    p = dst / "encode_impl.cuh"
    p.write_text(p.read_text() + "\n// a trailing comment\n")
    assert bench.kernel_src_hash() == full0
    assert bench.kernel_src_hash(bench.TRAFFIC_SOURCES) == scoped0

    # a code edit outside the two kernels' units changes only the full hash
    q = dst / "dequant.cu"
    q.write_text(q.read_text() + "\nnamespace { int unused_marker = 0; }\n")
    assert bench.kernel_src_hash() != full0
    assert bench.kernel_src_hash(bench.TRAFFIC_SOURCES) == scoped0

    # a code edit inside them changes the scoped hash too
    p.write_text(p.read_text() + "\nnamespace { int unused_marker = 1; }\n")
    assert bench.kernel_src_hash(bench.TRAFFIC_SOURCES) != scoped0
