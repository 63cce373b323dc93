"""Host logic of bench.py that needs no GPU: the comment-insensitive hash
that keys the committed ncu traffic figures to the code they were taken on,
and the lookup of those figures."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_drops_comments_keeps_literals():
    src = ('int a = 1; // line comment\n'
           'const char* s = "not // a comment";  /* block\n spanning */ int b;\n'
           "char c = '/'; char d = '\\''; const char* e = \"q\\\"/*\"; int f;\n")
    out = bench.code_only(src)
    assert "line comment" not in out and "block" not in out and "spanning" not in out
    assert '"not // a comment"' in out
    assert "'/'" in out and "'\\''" in out and '"q\\"/*"' in out and "int f;" in out
    assert bench.code_only(src) == bench.code_only(src.replace("line comment", "another remark"))
    assert bench.code_only(src) != bench.code_only(src.replace("int b;", "int bb;"))


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SOURCES))
def test_source_hash_follows_code_not_comments(kernel, tmp_path, monkeypatch):
    """A copy of the sources with one comment edited hashes the same; with
    one token of code edited it hashes differently."""
    import shutil
    csrc = os.path.join(ROOT, "block_quantized_routed_gb300", "csrc")
    root = tmp_path / "r"
    (root / "block_quantized_routed_gb300").mkdir(parents=True)
    shutil.copytree(csrc, root / "block_quantized_routed_gb300" / "csrc")
    (root / "include").mkdir()
    shutil.copy(os.path.join(ROOT, "include", "moe_q8k.h"), root / "include" / "moe_q8k.h")
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.kernel_source_hash(kernel)
    hdr = root / "include" / "moe_q8k.h"
    text = hdr.read_text()
    hdr.write_text(text.replace("/*", "/* edited remark:", 1))
    assert bench.kernel_source_hash(kernel) == base
    src = root / "block_quantized_routed_gb300" / "csrc" / bench.KERNEL_SOURCES[kernel][0]
    code = src.read_text()
    src.write_text(code + "\nstatic const int kHashProbe = 1;\n")
    assert bench.kernel_source_hash(kernel) != base


def test_profiled_traffic_lookup():
    """Every traffic line in profiles/ names a kernel the bench knows; the
    ones keyed to the current code are found, a wrong workload is not."""
    import re
    pdir = os.path.join(ROOT, "profiles")
    lines = []
    for f in sorted(os.listdir(pdir)):
        if f.endswith(".md"):
            lines += re.findall(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+kernel:\s*(\S+)\s+workload:\s*(\S+)"
                                r"\s+source_hash:\s*(\w+)", open(os.path.join(pdir, f)).read(), flags=re.M)
    assert lines
    for value, kernel, workload, h in lines:
        assert kernel in bench.KERNEL_SOURCES
        if h == bench.kernel_source_hash(kernel):
            assert bench.profiled_traffic(workload, kernel) == float(value)
        assert bench.profiled_traffic(workload + "_x", kernel) is None
