"""Host-side pieces of bench.py (no GPU): the workloads match the configurations
they are named for, the byte accounting matches the format, the weight
rotation keeps two uses of one copy apart, and the committed DRAM-traffic
figures are only reported for the kernel source they were captured on."""
import os

import bench


def test_decode_layer_workload():
    g = bench.workload("decode_layer", None)
    assert len(g) == 20
    assert {(K, N) for _, _, K, N, _, _ in g} == {(4096, 6144), (4096, 4096), (4096, 28672),
                                                  (14336, 4096)}
    assert sorted({B for _, B, _, _, _, _ in g}) == [1, 2, 4, 8, 16]
    assert not any(zp for *_, zp, _ in g)


def test_decode_step_workload_is_32_layers_and_lm_head():
    g = bench.workload("decode_step", 4)
    assert len(g) == 32 * 4 + 1
    assert g[-1][2:4] == (4096, 128256)
    b, f = bench.step_bytes_flops(g)
    # 7 504 658 432 streamed weights at 4.125 bits, plus x and y of every GEMM
    xy = sum(B * K * 2 + B * N * 2 for _, B, K, N, _, _ in g)
    assert b == 7504658432 * 4.125 / 8 + xy
    assert f == 2 * 4 * 7504658432


def test_zero_point_and_prefill_workloads():
    g = bench.workload("zp70b", 64)
    assert all(zp for *_, zp, _ in g) and {B for _, B, *_ in g} == {64}
    p = bench.workload("prefill", None)
    assert all(B == 2048 and outl == 0.01 for _, B, _, _, _, outl in p)


def test_copy_rotation_spacing():
    g = bench.workload("decode_layer", None)
    uses = {}
    for _, B, K, N, zp, _ in g:
        uses[(K, N, zp)] = uses.get((K, N, zp), 0) + 1
    n_copies = 6
    pick = bench.copy_index(g, uses, n_copies)
    # every (K, N) is used 5 times per step; consecutive uses of a layer take
    # consecutive copies, so one copy is reused only n_copies uses later
    seq = [pick(k, i, (K, N, zp)) for k in range(3) for i, (_, _, K, N, zp, _) in enumerate(g)
           if (K, N) == (4096, 4096)]
    assert seq == [j % n_copies for j in range(len(seq))]


def test_traffic_is_tied_to_the_kernel_source(tmp_path, monkeypatch):
    want = bench.kernel_source_hash(bench.KERNEL_FILES["skinny"])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        f"# comment\nskinny decode_layer {want} 123\nskinny decode_layer 0000000000000000 999\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names: want)
    assert bench.traffic_from_profiles("skinny", "decode_layer") == 123.0
    assert bench.traffic_from_profiles("skinny", "moe") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names: "ffffffffffffffff")
    assert bench.traffic_from_profiles("skinny", "decode_layer") is None


def test_committed_traffic_file_parses():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    lines = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert lines and all(len(p) == 4 and p[3].isdigit() for p in lines)


def test_sweep_is_config_three():
    """The default workload: the full decode step (32 layers + lm_head) at every
    batch of the crossover sweep."""
    layers = bench.sweep_layers()
    assert len(layers) == 129 and layers[-1][1:] == (4096, 128256)
    assert sum(K * N for _, K, N in layers) == 7504658432
    assert bench.SWEEP_BATCHES == (1, 4, 16, 64, 128, 256, 270, 384, 512, 1024)


def test_sweep_roofline_bound_and_excess():
    # memory-bound: 1 GB at 1000 GB/s = 1 ms; 1 TFLOP at 1000 TFLOP/s = 1 ms
    r = bench.sweep_roofline(1e9, 0.5e12, 2e-3, 1000.0, 1000.0)
    assert r["bound"] == "hbm" and abs(r["frac"] - 0.5) < 1e-12
    assert abs(r["above_roofline_us"] - 1000.0) < 1e-6
    r = bench.sweep_roofline(0.5e9, 1e12, 4e-3, 1000.0, 1000.0)
    assert r["bound"] == "tensor" and abs(r["frac"] - 0.25) < 1e-12
    assert abs(r["achieved"] - 250.0) < 1e-9 and abs(r["above_roofline_us"] - 3000.0) < 1e-6
