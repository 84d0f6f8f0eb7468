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


def test_committed_summaries_carry_the_lookup_fields():
    # every summary names its kernel, workload, code hash and DRAM bytes; its
    # bytes are reported only while the hash matches the current kernel code
    import glob
    import os
    import re
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")))
    assert paths
    for path in paths:
        text = open(path).read()
        fields = {k: re.search(rf"^{k}:\s*(\S+)", text, re.M)
                  for k in ("kernel", "workload", "kernel_source_sha256_16", "dram_bytes_per_launch")}
        assert all(fields.values()), path
        kernel, workload = fields["kernel"].group(1), fields["workload"].group(1)
        assert kernel in bench.KERNEL_SOURCES, path
        traffic, src = bench.read_traffic(workload, kernel)
        if fields["kernel_source_sha256_16"].group(1) == bench.kernel_source_hash(kernel):
            assert traffic == float(fields["dram_bytes_per_launch"].group(1)) and src
        else:
            assert traffic is None or src != os.path.relpath(path, bench.ROOT)


def test_step_stats():
    st = bench.step_stats([3.0, 1.0, 2.0, 10.0, 4.0, 5.0, 6.0, 7.0, 8.0, 9.0])
    assert st["ms_mean"] == 5.5 and st["ms_median"] == 5.5 and st["ms_min"] == 1.0
    assert st["ms_p90"] == 9.0  # the 9th of 10 sorted values
    one = bench.step_stats([2.5])
    assert one["ms_mean"] == one["ms_median"] == one["ms_p90"] == one["ms_min"] == 2.5


def test_row_flops_follow_the_metric():
    from fa_inputs import AttentionWorkload
    w = AttentionWorkload("t", 1, 1, 100, 64, False, 0.125, 1)
    assert bench.row_flops(w, range(100)) == w.flops          # a whole head, non-causal
    assert bench.row_flops(w, [0, 5]) == 2 * 4 * 100 * 64
    wc = AttentionWorkload("t", 1, 1, 100, 64, True, 0.125, 1)
    # causal: row i sees i + 1 keys; a whole head is 2 L (L + 1) d, the
    # metric's halved count up to the diagonal
    assert bench.row_flops(wc, range(100)) == 2 * 100 * 101 * 64
    assert abs(bench.row_flops(wc, range(100)) / wc.flops - 1) < 0.011
