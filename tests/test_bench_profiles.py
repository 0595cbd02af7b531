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


def test_every_committed_profile_matches_its_kernel_sources():
    """Each profiles/hsp_<kernel>_kernel_<workload>_m<M>.md names a kernel of the bench and
    carries the hash of that kernel's current sources, so its traffic figure is in use."""
    pdir = os.path.join(ROOT, "profiles")
    names = [f for f in os.listdir(pdir) if f.startswith("hsp_") and f.endswith(".md")]
    assert names
    for f in names:
        kernel = f.split("_")[1]
        assert kernel in bench.KERNEL_FILES, f
        workload, m = f[len(f"hsp_{kernel}_kernel_"):-3].rsplit("_m", 1)
        assert bench.profiled_traffic(workload, int(m)) is not None, f"{f}: stale or unreadable"
