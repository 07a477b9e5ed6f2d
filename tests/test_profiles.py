"""The committed ncu summaries that give a kernel's DRAM bytes per launch
(which bench.py attaches to its roofline as `traffic`) must describe the
current code of that kernel: their `code_sha256_16` line has to equal the
hash bench.py computes from the source (comments and blank lines removed)."""
import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = {"attn_fwd": "fwd_tcgen05.cu", "attn_merge": "merge.cu"}


def test_profiles_with_traffic_match_the_current_kernel_code():
    seen = 0
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.txt")):
        name = os.path.basename(path)[:-4]
        kernel = next((k for k in SOURCES if name.startswith(k + "_")), None)
        if kernel is None or "dram_bytes_per_launch:" not in open(path).read():
            continue
        workload = name[len(kernel) + 1:]
        src = os.path.join(ROOT, "block_sparse_attention_slice_gb300", "csrc", SOURCES[kernel])
        assert bench.profile_traffic(kernel, workload, src) is not None, name
        seen += 1
    assert seen >= 3


def test_code_hash_ignores_comments_only(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    a.write_text('int f(int x) {  // one\n  return x + 1;\n}\n')
    b.write_text('// a new comment\nint f(int x) {\n\n  return x + 1;  // two\n}\n')
    assert bench.code_sha16(str(a)) == bench.code_sha16(str(b))
    b.write_text('int f(int x) {\n  return x + 2;\n}\n')
    assert bench.code_sha16(str(a)) != bench.code_sha16(str(b))
