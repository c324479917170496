"""The bench's roofline bookkeeping on the CPU (no GPU): a decode record's
whole-step HBM roofline divides the step's algorithmic bytes by the timed
step (not by the sum of eager stage times), and a tensor record reports its
longest stage against the burst peak, or the sustained one when the timed
region is long."""
import pytest

import bench

PEAKS = {"hbm_gbs": 6500.0, "bf16_tflops": 1750.0, "bf16_tflops_sustained": 1350.0,
         "source": "test"}


class _Step:
    """Stands in for a decode workload: only its algorithmic bytes matter."""

    def work(self):
        return {"step_bytes": 2.6e9, "attn_flop": 1.0}


@pytest.mark.parametrize("cls", [bench.Decode, bench.DecodeIncremental])
def test_decode_rooflines_use_the_timed_step(cls):
    # eager stage times that sum to more than the timed (graph-replayed) step
    r = cls.roofline(_Step(), [0.50, 0.05], PEAKS, 5.2, 0.52)
    assert r["bound"] == "hbm"
    assert r["achieved"] == pytest.approx(2.6e9 / 0.52e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"])
    assert r["algorithmic_bytes"] == 2.6e9


def test_tensor_roofline_reports_the_longest_stage():
    stages = ["compress", "index", "attn"]
    flops = {"index": 1.0e12, "attn": 3.0e12}
    r = bench.tensor_roofline(stages, [0.1, 1.0, 2.0], flops, PEAKS, 35.0)
    assert r["kernel"] == "attn"
    assert r["achieved"] == pytest.approx(3.0e12 / 2.0e-3 / 1e12)
    assert r["peak"] == PEAKS["bf16_tflops"]
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"])
    # a timed region over a second is held to the sustained peak
    r = bench.tensor_roofline(stages, [0.1, 3.0, 2.0], flops, PEAKS, 2000.0)
    assert r["kernel"] == "index"
    assert r["peak"] == PEAKS["bf16_tflops_sustained"]
