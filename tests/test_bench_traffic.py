"""The benchmark's DRAM-traffic bookkeeping on CPU: the ncu byte counts are
keyed by a hash of the measured kernel's code (its translation unit and
every header it includes), so a comment edit keeps them and a code change
anywhere in the include closure drops them (the benchmark then reports null
instead of a stale figure).  No GPU is used."""
import os
import shutil

import pytest

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = "int a = 1;  // trailing\n\n/* block\n   comment */\nint b = 2;\n   \n// whole line\nint c;\n"
    assert bench._code_only(src) == "int a = 1;\nint b = 2;\nint c;"


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "sparse_attention_top_idx_gb300", "csrc"),
                    root / "sparse_attention_top_idx_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "include"), root / "include")
    return root


def _append(path, text):
    with open(path, "a") as f:
        f.write(text)


@pytest.mark.parametrize("tu, header", [("decode.cu", "segsel.cuh"), ("decode.cu", "topk.cuh"),
                                        ("prefill.cu", "topk.cuh"), ("decode.cu", "common.cuh")])
def test_hash_follows_code_of_included_headers_not_comments(tmp_path, monkeypatch, tu, header):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash(tu)
    assert h0 == bench.kernel_source_hash(tu)            # deterministic
    hdr = root / "sparse_attention_top_idx_gb300" / "csrc" / header
    _append(hdr, "\n// a comment only\n/* and a block\n   comment */\n\n")
    assert bench.kernel_source_hash(tu) == h0            # comments and blank lines do not count
    _append(hdr, "\nstatic_assert(true, \"a code change\");\n")
    assert bench.kernel_source_hash(tu) != h0            # code in an included header does


def test_hash_ignores_files_outside_the_include_closure(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash("prefill.cu")
    # the decode kernel's own header is not part of the prefill translation unit
    _append(root / "sparse_attention_top_idx_gb300" / "csrc" / "decode_kernel.cuh", "\nint unrelated;\n")
    assert bench.kernel_source_hash("prefill.cu") == h0


def test_traffic_table_shape():
    for (workload, digest), nbytes in bench.NCU_TRAFFIC.items():
        assert workload in bench.KERNEL_TU
        assert len(digest) == 16 and all(c in "0123456789abcdef" for c in digest)
        assert isinstance(nbytes, int) and nbytes > 0
    # a stale hash reports no traffic rather than an old number
    assert bench.NCU_TRAFFIC.get(("decode", "0" * 16)) is None
