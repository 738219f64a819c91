"""Host logic of bench.py that needs no GPU.

- The algorithmic bytes of the long causal workload (q, k, v read and o
  written once, bf16), the numerator of the bench's roofline figure.
- A DRAM traffic figure recorded from an ncu capture is reported only while
  the causal kernel's source files are byte-for-byte the ones it was captured
  on: any change to them makes the bench report `traffic: null`.
"""
import json

import bench


def test_alg_bytes_of_the_long_workload():
    w = bench.WORKLOADS["long"]
    assert (w.B, w.H, w.N, w.D, w.dtype) == (2, 8, 65536, 64, "bf16")
    assert bench.alg_bytes(w) == 2 * 8 * 65536 * (3 * 64 + 64) * 2 == 536_870_912


def _fake_tree(root):
    csrc = root / "linear_attention_elu_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    for name in bench.CAUSAL_SOURCES:
        (csrc / name).write_text(f"// {name}\n")
    (root / "profiles").mkdir(exist_ok=True)
    return csrc


def test_recorded_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    csrc = _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.csrc_digest()
    record = {"causal:long": {"bytes_per_launch": 767_000_000, "csrc_digest": digest}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(record))
    assert bench.recorded_traffic("causal:long") == 767_000_000
    assert bench.recorded_traffic("causal:image") is None          # never captured
    # Any edit to a file that compiles into the kernel invalidates the figure.
    (csrc / "tc_common.cuh").write_text("// tc_common.cuh, edited\n")
    assert bench.csrc_digest() != digest
    assert bench.recorded_traffic("causal:long") is None


def test_recorded_traffic_without_a_record_file(tmp_path, monkeypatch):
    _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("causal:long") is None


def test_digest_covers_exactly_the_kernel_sources(tmp_path, monkeypatch):
    csrc = _fake_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.csrc_digest()
    # A file outside the causal kernel's sources does not move the digest.
    (csrc / "decode.cu").write_text("// another kernel\n")
    assert bench.csrc_digest() == digest
