"""Host logic of bench.py, CPU only: the committed ncu summaries count for
the roofline only while the kernels' code is what was profiled (comments
aside), and only on the workload they were taken on."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402

CODE = """// a comment
__global__ void k(float *x) {  // trailing comment
    /* block
       comment */
    x[0] = 1.0f;
}
"""


def write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return str(p)


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a = write(tmp_path, "a.cu", CODE)
    b = write(tmp_path, "b.cu", "\n\n" + CODE.replace("// a comment", "// another comment")
              .replace("/* block", "/* a longer block") + "\n// tail\n")
    assert bench.source_code_hash([a]) == bench.source_code_hash([b])


def test_code_hash_sees_code_changes(tmp_path):
    a = write(tmp_path, "a.cu", CODE)
    b = write(tmp_path, "b.cu", CODE.replace("1.0f", "2.0f"))
    c = write(tmp_path, "c.cu", CODE.replace("x[0] = 1.0f;", "x[0] = 1.0f;\n    x[1] = 0.0f;"))
    ha = bench.source_code_hash([a])
    assert ha != bench.source_code_hash([b])
    assert ha != bench.source_code_hash([c])
    # the order of the files is part of the code
    assert bench.source_code_hash([a, c]) != bench.source_code_hash([c, a])


def test_profiled_traffic_needs_matching_code_and_workload(tmp_path, monkeypatch):
    src = write(tmp_path, "k.cu", CODE)
    summary = write(tmp_path, "k.md", "\n".join([
        "# summary", "",
        "traffic_bytes_per_launch: 12345",
        "source_code_sha256_16: %s" % bench.source_code_hash([src]),
        "workload: c3", ""]))
    monkeypatch.setitem(bench.PROFILES, "k", (summary, [src]))
    assert bench.profiled_traffic("k", "c3") == 12345.0
    assert bench.profiled_traffic("k", "c4") is None
    with open(src, "a") as f:
        f.write("// a comment edit keeps the capture valid\n")
    assert bench.profiled_traffic("k", "c3") == 12345.0
    with open(src, "a") as f:
        f.write("__device__ int changed;\n")
    assert bench.profiled_traffic("k", "c3") is None


def test_profile_sources_cover_every_included_file():
    """Each profiled kernel's hash covers its translation unit and every file
    it reaches through #include "...": a change to any of them (a shared
    header, the C-ABI header) makes the committed capture stale."""
    import re
    for kernel, (_, sources) in bench.PROFILES.items():
        names = {os.path.basename(p) for p in sources}
        assert len(names) == len(sources)
        for path in sources:
            for inc in re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(path).read(), flags=re.M):
                assert os.path.basename(inc) in names, (kernel, path, inc)
    assert {"topp.cu", "common.cuh", "stream.cuh", "spec_verify.h"} <= {
        os.path.basename(p) for p in bench.PROFILES["topp_kernel"][1]}
    assert {"rows.cu", "common.cuh", "stream.cuh", "spec_verify.h"} <= {
        os.path.basename(p) for p in bench.PROFILES["stream_kernel"][1]}


def test_include_closure_follows_nested_includes(tmp_path):
    (tmp_path / "a.cu").write_text('#include "b.cuh"\n__global__ void k() {}\n')
    (tmp_path / "b.cuh").write_text('#pragma once\n#include "c.h"\n')
    (tmp_path / "c.h").write_text("#pragma once\n#include <stdint.h>\n")
    got = [os.path.basename(p) for p in bench.include_closure(str(tmp_path / "a.cu"))]
    assert got == ["a.cu", "b.cuh", "c.h"]
    (tmp_path / "c.h").write_text('#include "missing.h"\n')
    import pytest
    with pytest.raises(FileNotFoundError):
        bench.include_closure(str(tmp_path / "a.cu"))
