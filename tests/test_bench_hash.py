"""The kernel-source hash that keys bench.py's recorded DRAM traffic.

A record stays valid across comment and layout edits of the kernel sources and goes
stale on any change of code.
"""
import importlib.util
import os
import shutil

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_for_hash", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _copy_sources(bench, dst):
    src_dir = os.path.join(ROOT, "paged_kv_cache_61_gb300", "csrc")
    out_dir = os.path.join(dst, "paged_kv_cache_61_gb300", "csrc")
    os.makedirs(out_dir)
    for names in bench.KERNEL_SOURCES.values():
        for name in names:
            shutil.copy(os.path.join(src_dir, name), out_dir)
    return out_dir


def test_comment_edits_keep_the_hash_code_edits_change_it(tmp_path):
    bench = _bench()
    bench.ROOT = str(tmp_path)
    csrc = _copy_sources(bench, str(tmp_path))
    before = {kind: bench.kernel_hash(kind) for kind in bench.KERNEL_SOURCES}
    path = os.path.join(csrc, "mla_rows.cu")
    with open(path) as f:
        text = f.read()
    # a comment line, a trailing comment, a block comment and re-indentation
    edited = ("// an added comment line\n" +
              text.replace("constexpr int kStages = 5;",
                           "constexpr  int kStages = 5;   // stages /* of the ring */"))
    with open(path, "w") as f:
        f.write(edited + "\n/* trailing\n   block comment */\n")
    assert {kind: bench.kernel_hash(kind) for kind in bench.KERNEL_SOURCES} == before
    with open(path, "w") as f:
        f.write(text.replace("constexpr int kStages = 5;", "constexpr int kStages = 4;"))
    after = {kind: bench.kernel_hash(kind) for kind in bench.KERNEL_SOURCES}
    assert after["mla_rows"] != before["mla_rows"]
    assert after["gqa"] == before["gqa"] and after["mla"] == before["mla"]
