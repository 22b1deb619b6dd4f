"""The tensor-core rate probe (domino_tensor_peak) on the GB300: paired tcgen05 MMAs
alone.  Its three readings -- event time, the kernel's own cycle count and the
kernel's own nanosecond count -- must tell one consistent story, and the per-SM
rate per clock must lie in the range that the GPU's nominal dense bf16 peak
allows."""
import pytest
import torch

from communication_overlap_domino_gb300 import binding as b

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_probe_is_self_consistent():
    ws = torch.zeros(b.TENSOR_PEAK_WS_BYTES, dtype=torch.uint8, device="cuda")
    b.tensor_peak(1 << 14, workspace=ws)  # warm-up
    r = b.tensor_peak(1 << 19, workspace=ws)
    assert b.query_device_status(ws) == 0
    assert r["num_sms"] == torch.cuda.get_device_properties(0).multi_processor_count
    # every 2-CTA cluster on its own pair of SMs, at most one CTA per SM
    assert r["num_sms"] // 2 - 8 <= r["clusters"] <= r["num_sms"] // 2
    assert 500.0 <= r["sm_mhz"] <= 2300.0
    # 2.25 PFLOP/s nominal over 152 SMs needs >= 6,400 flops per clock per SM at <= 2.3 GHz;
    # a rate above twice that would mean MMAs were not executed
    assert 4096.0 <= r["flops_per_clk_sm"] <= 16384.0
    # the event-timed rate is what the clusters' cycle counts predict (all clusters run together)
    predicted = r["clusters"] * 2 * r["flops_per_clk_sm"] * r["sm_mhz"] * 1e6 / 1e12
    assert 0.85 * predicted <= r["tflops"] <= 1.02 * predicted
    assert r["flops"] == 2.0 * 256 * 256 * 16 * (1 << 19) * r["clusters"]


def test_probe_scales_with_clusters_and_rejects_too_many():
    full = b.tensor_peak(1 << 17)
    one = b.tensor_peak(1 << 17, clusters=1)
    assert one["clusters"] == 1
    # one cluster runs at the same per-SM rate per clock as all of them
    assert one["flops_per_clk_sm"] == pytest.approx(full["flops_per_clk_sm"], rel=0.05)
    with pytest.raises(b.DominoError) as e:
        b.tensor_peak(1 << 10, clusters=full["clusters"] + 1)
    assert e.value.status == 2
