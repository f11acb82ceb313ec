"""Host-side logic of bench.py: the comment-stripped source stamps that tie each
ncu summary under profiles/ to the kernel sources it was taken on, the DRAM
traffic the bench line reports from such a summary, and the host description of
the oracle baseline.  No GPU is needed."""

import glob
import os
import re

import bench


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // note\n/* block\n comment */ const char* s = "// not a comment";\n'
           "char c = '/';\n\n")
    out = bench.strip_comments(src)
    assert "note" not in out and "block" not in out
    assert '"// not a comment"' in out and "'/'" in out
    assert "int a = 1;" in out
    assert "\n\n" not in out


def test_a_comment_only_edit_keeps_the_stamp():
    path = os.path.join(bench.ROOT, "int8_kv_cache_02_gb300", "csrc", "decode_combine.cu")
    src = open(path).read()
    edited = src.replace("\n", "  // an added remark\n", 3) + "\n/* trailing */\n"
    assert bench.strip_comments(edited) == bench.strip_comments(src)
    changed = src.replace("kCombineWarps = 8", "kCombineWarps = 4", 1)
    assert changed != src
    assert bench.strip_comments(changed) != bench.strip_comments(src)


def test_every_profile_names_the_current_sources():
    """Each summary states the files its stamp covers; the stamp must be the hash of
    those files as they are now, or the summary describes other kernels."""
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")))
    assert paths
    for path in paths:
        txt = open(path).read()
        stamp = re.search(r"kernel source sha256: (\w+)", txt)
        files = re.search(r"The stamp covers `csrc/` (.*)\.", txt)
        assert stamp and files, path
        names = re.findall(r"`([\w.]+)`", files.group(1))
        assert names, path
        assert bench.source_sha(names) == stamp.group(1), f"{path}: taken on other sources"


def test_traffic_comes_from_a_fresh_summary_only():
    traffic = bench.traffic_from_profiles(bench.decode_source_sha())
    assert traffic is not None and traffic >= 8_675_328   # at least the algorithmic bytes
    assert bench.traffic_from_profiles("0" * 16) is None


def test_host_info():
    h = bench.host_info()
    assert h["cpu"] and h["machine"]
    assert h["cores_available"] >= 1 and h["cores_used_by_the_oracle"] == 1
