"""The bench's description of the layer workload (host only): the constants both arms
print agree with the oracle's layout and the layer's shapes."""
import bench
from oracle import layout as L
from param_buffers_gb300 import workloads as W
from test_oracle_layout import cfg_of, specs


def test_layer_buffer_numel_is_the_oracle_layout():
    bw = W.layer_buffer()
    lay = L.compute_layout(specs(bw.params), cfg_of(bw))
    assert bench.LAYER_BUFFER_NUMEL == lay.buffers[0].numel == 30_412_800


def test_layer_config_counts():
    c = bench.layer_config(W, 1, 152)
    M, mb = W.LAYER_M, W.LAYER_MICROBATCHES
    # 3 GEMMs of 2 M N K FLOPs per linear and microbatch: QKV 1536x2048, O 2048x1024,
    # fc1 8192x2048, fc2 2048x4096
    per_mb = 3 * 2 * M * (1536 * 2048 + 2048 * 1024 + 8192 * 2048 + 2048 * 4096)
    assert abs(c["gemm_tflop_per_step"] - mb * per_mb / 1e12) < 1e-9
    assert c["M"] == 8192 and c["microbatches"] == 8 and c["flat_buffer_elems"] == 30_412_800
    # bf16 X [M, K] and dY [M, N] of every linear, fresh each microbatch
    assert "3.02 GB" in c["l2"]
    assert c == bench.layer_config(W, 1, 152)             # one description for both arms


def test_traffic_records_follow_the_source_hash(tmp_path, monkeypatch):
    """A recorded DRAM-traffic figure is used only while the kernel sources it was taken
    from are unchanged; another hash, a missing row or a missing file give None."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "aaaa")
    monkeypatch.setattr(bench, "sweep_source_hash", lambda: "bbbb")
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    assert bench.traffic_from_profiles("overlap.fc1+proj") is None           # no file
    (prof / "traffic.txt").write_text("# kernel hash bytes\noverlap.fc1+proj aaaa 584628480\n"
                                      "fprop.fc1 cccc 1.0\n")
    assert bench.traffic_from_profiles("overlap.fc1+proj") == 584628480.0
    assert bench.traffic_from_profiles("fprop.fc1") is None                   # stale hash
    assert bench.traffic_from_profiles("dgrad.fc1") is None                   # no row
    (prof / "traffic_sweep.txt").write_text("adam_flat bbbb 33.84\n")
    assert bench.sweep_traffic_per_elem() == 33.84
    (prof / "traffic_sweep.txt").write_text("adam_flat dddd 33.84\n")
    assert bench.sweep_traffic_per_elem() is None


def test_committed_traffic_records_match_the_sources():
    """The committed records are the current sources' (a GEMM or sweep change without a new
    capture would leave the bench line without traffic)."""
    rows = {}
    for line in (bench.ROOT / "profiles" / "traffic.txt").read_text().splitlines():
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#"):
            rows[parts[0]] = parts[1]
    assert rows["overlap.fc1+proj"] == bench.gemm_source_hash()
    assert bench.sweep_traffic_per_elem() is not None
