"""The dense NVFP4 tensor-core probe (nvmoe_fp4_mma_probe) runs every
variant to completion: one CTA and CTA pairs (cta_group::2), N = 256 and
128, with no scale copies, with the per-MMA 32x128b.warpx4 copies and with
per-stage 128x256b copies.  Status 0, a positive cycle count on every
issuing CTA, and a throughput below the datasheet's dense FP4 figure with
headroom (the probe cannot beat the hardware)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 8, 9])
def test_probe_variants_complete(nb, variant):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    r = nb.fp4_mma_probe(variant, iters=4096, grid=n_sm - (n_sm & 1), repeats=2)
    assert r["status"] == 0
    assert r["cycles_per_mma"] is not None and r["cycles_per_mma"] > 0
    assert 0 < r["tflops"] < 30000
    print(f"variant {variant}: {r['tflops']:.0f} TFLOP/s, {r['cycles_per_mma']:.1f} cycles/MMA")


def test_probe_rejects_bad_arguments(nb):
    cyc = torch.zeros(8, dtype=torch.int64, device="cuda")
    ws = nb._workspace(256, "cuda")
    lib = nb.lib()
    s = nb._stream()
    assert lib.nvmoe_fp4_mma_probe(12, 16, 8, nb._ptr(cyc), nb._ptr(ws), 256, s) == 1
    assert lib.nvmoe_fp4_mma_probe(1, 16, 7, nb._ptr(cyc), nb._ptr(ws), 256, s) == 1
    assert lib.nvmoe_fp4_mma_probe(0, 0, 8, nb._ptr(cyc), nb._ptr(ws), 256, s) == 1
    assert lib.nvmoe_fp4_mma_probe(0, 16, 8, nb._ptr(cyc), nb._ptr(ws), 16, s) == 4
