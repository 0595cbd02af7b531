"""bench.py's profile bookkeeping (CPU): a committed ncu summary's DRAM traffic is reported
only while the kernel's device sources are unchanged; comments do not count, code does."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_keeps_code_and_strings():
    src = 'int a = 1; // one\n/* block\n   comment */ const char *s = "x // y /* z */";\n\n  return a;  \n'
    out = bench.strip_comments(src)
    assert out == 'int a = 1;\nconst char *s = "x // y /* z */";\nreturn a;'


def test_comment_edits_keep_the_hash_code_edits_change_it():
    a = "__global__ void k(int *p) { p[0] = 1; }\n"
    b = "// a note\n__global__ void k(int *p) { /* why */ p[0] = 1; }  // end\n"
    c = "__global__ void k(int *p) { p[0] = 2; }\n"
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert bench.strip_comments(a) != bench.strip_comments(c)


def test_every_committed_profile_is_readable_by_the_bench():
    """Each profiles/hsp_<kernel>_kernel_<workload>_m<M>.md names a kernel of the bench and
    a workload, and carries a source hash and an integer traffic figure; the bench reports
    that figure while the hash matches the kernel's sources (else null)."""
    import workloads as W
    pdir = os.path.join(ROOT, "profiles")
    names = [f for f in os.listdir(pdir) if f.startswith("hsp_") and f.endswith(".md")]
    assert names
    for f in names:
        kernel = f.split("_")[1]
        assert kernel in bench.KERNEL_FILES, f
        workload, m = f[len(f"hsp_{kernel}_kernel_"):-3].rsplit("_m", 1)
        assert workload in W.WORKLOADS and int(m) in W.WORKLOADS[workload].Ms, f
        fields = dict(ln.split(":", 1) for ln in open(os.path.join(pdir, f)) if ln[:1].isalpha() and ":" in ln)
        assert len(fields["kernel_sources_sha256_16"].strip()) == 16, f
        traffic = int(fields["traffic_bytes_per_launch"])
        got = bench.profiled_traffic(workload, int(m))
        fresh = fields["kernel_sources_sha256_16"].strip() == bench.kernel_sources_sha16(kernel)
        assert got == (traffic if fresh else None), f
