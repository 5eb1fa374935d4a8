"""Host-side pieces of bench.py: the algorithmic byte count and the recorded DRAM traffic."""
import json


import bench
from dsa_sparse_attention_mla_gb300 import workloads as W


def test_algorithmic_bytes_fp8_decode():
    # valid rows x 264-byte packed rows + q + out + index list + block table
    wl = W.config(3)
    w = bench.algorithmic_work(wl)
    n_valid = int((wl.indices >= 0).sum())
    expect = n_valid * 264 + wl.T * 64 * 256 * 2 * 2 + wl.indices.size * 4 + wl.block_table.size * 4
    assert w["bytes"] == expect
    assert w["flops"] == 2.0 * 64 * n_valid * (256 + 256)


def test_recorded_traffic_tracks_kernel_sources(tmp_path, monkeypatch):
    # a record whose hash matches the sources is reported; any change to them voids it
    root = tmp_path
    src = root / "dsa_sparse_attention_mla_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    import hashlib

    h = hashlib.sha256()
    h.update(b"k.cu")
    h.update(b"kernel v1")
    rec = {"csrc_sha256": h.hexdigest(), "workloads": {"w": {"traffic": 1234}}}
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench._recorded_traffic("w") == 1234
    assert bench._recorded_traffic("other") is None
    (src / "k.cu").write_text("kernel v2")
    assert bench._recorded_traffic("w") is None


def test_recorded_traffic_follows_only_the_listed_sources(tmp_path, monkeypatch):
    # a record that lists its kernels' files ignores the other files and voids on a listed one
    root = tmp_path
    src = root / "dsa_sparse_attention_mla_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "a.cu").write_text("measured v1")
    (src / "b.cu").write_text("other v1")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    import hashlib

    h = hashlib.sha256()
    h.update(b"a.cu")
    h.update(b"measured v1")
    rec = {"csrc_sha256": h.hexdigest(), "sources": ["a.cu"], "workloads": {"w": {"traffic": 99}}}
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench._recorded_traffic("w") == 99
    (src / "b.cu").write_text("other v2")
    assert bench._recorded_traffic("w") == 99
    (src / "a.cu").write_text("measured v2")
    assert bench._recorded_traffic("w") is None
    (src / "a.cu").unlink()
    assert bench._recorded_traffic("w") is None


def test_kernels_per_call_follows_the_launch_rule():
    # decode T=256 x 17 windows on 152 SMs: 28 units per CTA, one launch; causal prefill
    # T=8192 x 16 windows: 862 units per CTA, split pre-pass + attention; 512+64: one launch
    assert bench.kernels_per_call(W.config(3), 152) == 1
    assert bench.kernels_per_call(W.config(4), 152) == 3
    assert bench.kernels_per_call(W.config(5), 152) == 1


def test_roofline_bound_follows_the_stricter_term():
    # decode gathers distinct rows of a 2.2 GB table: memory-bound, and every gathered byte is
    # unique; causal prefill re-gathers a 4 MB table: the tensor term is the slower one
    w3 = bench.algorithmic_work(W.config(3))
    assert w3["unique_bytes"] == w3["bytes"]
    r3 = bench.roofline(w3, 100e-6, 6759.9, 1905.3)
    assert r3["bound"] == "hbm" and r3["unit"] == "GB/s"
    assert abs(r3["achieved"] - w3["bytes"] / 100e-6 / 1e9) < 1e-6 * r3["achieved"]
    w4 = bench.algorithmic_work(W.config(4))
    assert w4["unique_bytes"] == 8192 * 512 + 8192 * 64 * 256 * 2 * 2 + W.config(4).indices.size * 4
    r4 = bench.roofline(w4, 1.6e-3, 6759.9, 1905.3)
    assert r4["bound"] == "tensor" and r4["unit"] == "TFLOP/s"
    assert abs(r4["frac"] - w4["flops"] / 1.6e-3 / 1e12 / 1905.3) < 1e-12
