"""CPU checks of how bench.py ties a committed ncu summary to the kernel
sources it was taken on: the hash covers the code, not its comments, and a
summary whose hash differs yields no traffic figure."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_keeps_literals():
    src = ('int a = 1; // trailing\n'
           '/* a block\n   comment */ const char *s = "x // y /* z */";\n'
           "char q = '\\''; char r = '/';\n"
           '\n'
           '   int b; /* inline */ int c;  \n')
    got = bench.code_only(src)
    assert got == ('int a = 1;\n'
                   ' const char *s = "x // y /* z */";\n'
                   "char q = '\\''; char r = '/';\n"
                   '   int b;  int c;')


def test_comment_edits_leave_the_hash_and_code_edits_change_it(tmp_path, monkeypatch):
    csrc = tmp_path / "segmented_gemm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    files = {"fused_tc.cu": "__global__ void k() { int x = 1; }\n", "internal.h": "#pragma once\n",
             "ptx.cuh": "// helpers\n#pragma once\n"}
    for name, text in files.items():
        (csrc / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash("lora_tc_kernel")
    (csrc / "ptx.cuh").write_text("// helpers, reworded\n\n#pragma once\n")
    assert bench.kernel_source_hash("lora_tc_kernel") == h0
    (csrc / "fused_tc.cu").write_text("__global__ void k() { int x = 2; }\n")
    assert bench.kernel_source_hash("lora_tc_kernel") != h0


def test_a_summary_on_other_sources_gives_no_traffic(tmp_path, monkeypatch):
    csrc = tmp_path / "segmented_gemm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("fused_tc.cu", "internal.h", "ptx.cuh"):
        (csrc / name).write_text(f"int {name.split('.')[0]};\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("lora_tc_kernel")
    (prof / "lora_tc_kernel_prefill.md").write_text(f"traffic_bytes_per_launch: 1234\nsource_hash: {h}\n")
    assert bench.profiled_traffic("lora_tc_kernel", "prefill") == 1234.0
    (prof / "lora_tc_kernel_prefill.md").write_text("traffic_bytes_per_launch: 1234\nsource_hash: 0000000000000000\n")
    assert bench.profiled_traffic("lora_tc_kernel", "prefill") is None
    assert bench.profiled_traffic("lora_tc_kernel", "qkv") is None   # no summary at all


def test_committed_summaries_name_a_known_kernel_and_their_command():
    """Every ncu summary under profiles/ gives the command that made it (ncu
    with --clock-control none), a source hash, and, for a single kernel's
    capture, its DRAM traffic per launch under the kernel's own name."""
    prof = os.path.join(ROOT, "profiles")
    names = sorted(f for f in os.listdir(prof) if f.endswith(".md"))
    assert names
    for f in names:
        txt = open(os.path.join(prof, f)).read()
        assert "ncu " in txt and "--clock-control none" in txt, f
        assert re.search(r"^source_hash: [0-9a-f]{16}$", txt, re.M), f
        if f.startswith("launches_"):
            continue
        kernel = next((k for k in bench.KERNEL_SOURCES if f.startswith(k + "_")), None)
        assert kernel is not None, f
        assert re.search(r"^traffic_bytes_per_launch: \d+$", txt, re.M), f
