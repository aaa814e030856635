"""Host-side logic of the benchmark's records (no GPU): the comment-insensitive
source digest and the ncu CSV reader behind the DRAM traffic record."""
import os

import bench
from block_scaled_fp8_gb300 import build


def test_strip_comments_keeps_code_and_literals():
    src = 'int a = 1; // one\n/* two\n lines */ const char *s = "//x /*y*/";  \n\nchar c = \'"\';\n'
    assert build.strip_comments(src) == 'int a = 1;\nconst char *s = "//x /*y*/";\nchar c = \'"\';'


def test_digest_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir()
    inc.mkdir()
    (inc / "dg.h").write_text("int f(void);\n")
    (csrc / "k.cu").write_text("__global__ void k() { int x = 1; }\n")
    monkeypatch.setattr(build, "CSRC", str(csrc))
    monkeypatch.setattr(build, "HERE", str(tmp_path / "pkg"))
    (tmp_path / "pkg").mkdir()
    d0 = build.source_digest()
    (csrc / "k.cu").write_text("// a comment\n__global__ void k() { int x = 1; /* why */ }\n")
    assert build.source_digest() == d0
    (csrc / "k.cu").write_text("__global__ void k() { int x = 2; }\n")
    assert build.source_digest() != d0


def test_read_ncu_csv_units_and_order(tmp_path):
    head = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",' \
           '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
    row = '"{i}","1","p","h","void k<{i}>(int)","1","7","(384, 1, 1)","(152, 1, 1)","0","10.3","s",' \
          '"{m}","{u}","{v}"\n'
    text = "==PROF== Connected\n" + head
    text += row.format(i=1, m="dram__bytes_read.sum", u="Mbyte", v="1.5")
    text += row.format(i=1, m="gpu__time_duration.sum", u="usecond", v="2,000")
    text += row.format(i=0, m="dram__bytes_read.sum", u="byte", v="100")
    p = tmp_path / "x.csv"
    p.write_text(text)
    got = bench.read_ncu_csv(str(p))
    assert [g["kernel"] for g in got] == ["void k<0>(int)", "void k<1>(int)"]
    assert got[0]["dram__bytes_read.sum"] == 100
    assert got[1]["dram__bytes_read.sum"] == 1.5e6 and got[1]["gpu__time_duration.sum"] == 2e6
