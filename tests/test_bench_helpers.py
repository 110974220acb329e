"""Host-side helpers of bench.py: staging buffers of the end-to-end steps, the bit-exact
comparison of read-back results, and the rule that keys a committed DRAM-traffic record
to the kernel's code and workload."""
import os

import pytest
import torch

import bench


@pytest.fixture
def no_pinning(monkeypatch):
    # no driver here: plain host memory stands in for pinned memory
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)


def test_staging_layout(no_pinning):
    a = torch.randn(3, 5, 7).to(torch.bfloat16)     # 210 B: padded to 256
    b = torch.randn(3, 5)                            # 60 B
    bufs, views = bench.staging([a, b], "cpu", sets=2)
    assert len(bufs) == 2 and all(buf.numel() == 512 for buf in bufs)
    for v in views:
        assert v[0].shape == a.shape and v[0].dtype == a.dtype and v[0].is_contiguous()
        assert v[1].shape == b.shape and v[1].dtype == b.dtype
        assert v[1].data_ptr() - v[0].data_ptr() == 256
    assert views[0][0].data_ptr() != views[1][0].data_ptr()


def test_staged_equal(no_pinning):
    a = torch.randn(4, 2, 8).to(torch.bfloat16)
    b = torch.randn(4, 2)
    bufs, views = bench.staging([a, b], "cpu", sets=1)
    views[0][0].copy_(a)
    views[0][1].copy_(b)
    assert bench.staged_equal(bufs[0], (a, b))
    b2 = b.clone()
    b2[3, 1] = torch.nextafter(b2[3, 1], torch.tensor(float("inf")))   # one ulp off
    assert not bench.staged_equal(bufs[0], (a, b2))


def test_code_hash_ignores_comments_only():
    src = "int f(int x) {  // doubles\n  return 2 * x;\n}\n"
    assert bench.code_sha256(src) == bench.code_sha256("/* header */\n" + src.replace("// doubles", "// twice"))
    assert bench.code_sha256(src) == bench.code_sha256(src + "\n\n// trailing note\n")
    assert bench.code_sha256(src) != bench.code_sha256(src.replace("2 * x", "3 * x"))


def test_traffic_record_keyed_on_code_and_workload(tmp_path, monkeypatch):
    csrc = tmp_path / "segmented_kv_attention_msa_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    code, plan = "__global__ void k() {}\n", "int plan() { return 1; }\n"
    (csrc / "k.cu").write_text(code)
    (csrc / "p.cpp").write_text(plan)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setitem(bench.TRAFFIC_SOURCES, "k", ("k.cu", "p.cpp"))
    (tmp_path / "profiles" / "k_traffic.txt").write_text(
        f"applies_to: wl_a\ncode_sha256: {bench.sources_sha256('k')}\ndram_bytes_per_launch: 1234\n")
    assert bench.kernel_traffic("k", "wl_a") == 1234.0
    assert bench.kernel_traffic("k", "wl_b") is None              # another workload
    (tmp_path / "profiles" / "k_traffic_wl_b.txt").write_text(    # its own file
        f"applies_to: wl_b\ncode_sha256: {bench.sources_sha256('k')}\ndram_bytes_per_launch: 99\n")
    assert bench.kernel_traffic("k", "wl_b") == 99.0
    assert bench.kernel_traffic("k", "wl_a") == 1234.0
    (csrc / "k.cu").write_text("// a comment\n" + code)
    assert bench.kernel_traffic("k", "wl_a") == 1234.0            # comment-only edit
    (csrc / "p.cpp").write_text("int plan() { return 2; }\n")
    assert bench.kernel_traffic("k", "wl_a") is None              # the planner changed
    (csrc / "p.cpp").write_text(plan)
    (csrc / "k.cu").write_text("__global__ void k() { int x = 1; (void)x; }\n")
    assert bench.kernel_traffic("k", "wl_a") is None              # the kernel changed
    assert bench.kernel_traffic("k", "wl_b") is None
