"""Host-side measurement logic of bench.py, on CPU: the roofline arithmetic
(the slower of the HBM and tensor bounds), the algorithmic work per selected
row, and the reading of the committed ncu traffic record, which is valid only
while the attention kernel's sources hash to the value it was taken on."""
import bench


def test_algorithmic_work_per_selected_row():
    # one selected row: its 512 latent + 64 rotary bf16 values; every head's
    # score (K = 576) and PV (N = 512) multiply-adds
    assert bench.ROW_BYTES == (512 + 64) * 2 == 1152
    assert bench.FLOP_PER_ROW == 128 * (576 + 512) * 2
    # the headline workload: 64 sequences x 2048 selected rows
    assert 64 * 2048 * bench.ROW_BYTES == 150_994_944


def test_roofline_takes_the_slower_bound():
    # HBM-bound: 151 MB at 6,500 GB/s is 23.2 us; its FLOPs at 1,750 TFLOP/s 20.9 us
    rows = 64 * 2048
    r = bench.roofline(rows * bench.ROW_BYTES, rows * bench.FLOP_PER_ROW, 0.05, 6500.0, 1750.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["ideal_ms"] - rows * 1152 / 6500e9 * 1e3) < 1e-12
    assert abs(r["achieved"] - rows * 1152 / 50e-6 / 1e9) < 1e-6
    assert abs(r["frac"] - r["ideal_ms"] / 0.05) < 1e-12
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert r["other_bound_ms"] < r["ideal_ms"]
    # the same work against a slow tensor peak is tensor-bound
    t = bench.roofline(rows * bench.ROW_BYTES, rows * bench.FLOP_PER_ROW, 0.05, 6500.0, 100.0)
    assert t["bound"] == "tensor" and t["unit"] == "TFLOP/s"
    assert abs(t["frac"] - t["achieved"] / t["peak"]) < 1e-12
    assert t["other_bound_ms"] < t["ideal_ms"]


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    digest = bench.kernel_source_digest()
    good = tmp_path / "good.md"
    good.write_text(f"kernel_source_sha256: {digest}\ndram_bytes_per_launch: 164303104\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(good))
    assert bench.traffic_record() == 164303104.0
    # a summary taken on other sources is not used
    stale = tmp_path / "stale.md"
    stale.write_text("kernel_source_sha256: " + "0" * 64 + "\ndram_bytes_per_launch: 1\n")
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(stale))
    assert bench.traffic_record() is None
    # nor a missing one
    monkeypatch.setattr(bench, "TRAFFIC_SUMMARY", str(tmp_path / "absent.md"))
    assert bench.traffic_record() is None

