"""Host-side helpers of the benchmark: the kernel source hash that ties a
committed ncu summary to the kernel it was captured on, and the lookup of a
summary's DRAM bytes."""

from __future__ import annotations

import bench


def test_comment_edits_do_not_change_the_code_hash():
    a = 'int a = 1; // note\n/* block\n comment */ asm("mov.u32 %0, 1;");\n'
    b = 'int a   = 1;\n// another note\nasm("mov.u32 %0, 1;");   /* x */\n'
    assert bench._code_only(a) == bench._code_only(b)


def test_code_edits_change_the_code_hash():
    assert bench._code_only("int a = 1;") != bench._code_only("int a = 2;")


def test_literals_are_kept_verbatim():
    src = 'asm("x // not a comment /* nor this */"); char c = \'"\'; s = "a\\"b"; // c'
    out = bench._code_only(src)
    assert '"x // not a comment /* nor this */"' in out
    assert "'\"'" in out and '"a\\"b"' in out
    assert out.endswith(";")


def test_every_committed_summary_matches_the_current_kernels():
    # each summary's DRAM bytes are reported only while its hash matches
    for workload, kernel in [("B4_H8_L1024_d64", "fwd"), ("gate_B1_H32_L8192_d128", "fwd"),
                             ("B1_H16_L32768_d64", "fwd"), ("gate_B1_H32_L8192_d128", "bwd"),
                             ("B1_H16_L32768_d64", "bwd"), ("gate_B1_H32_L8192_d128", "fwd_fp8")]:
        traffic, src = bench.read_traffic(workload, kernel)
        assert traffic is not None and traffic > 0, (workload, kernel)
        assert src.startswith("profiles/")
