"""Host-side arithmetic of the bench line and the seeded inputs (CPU only)."""

import torch

import bench
from causal_convolution_gb300 import inputs


def test_real_taps_counts_the_taps_that_read_a_real_frame():
    # temporal offsets 0, 1, 2 read frames t-2, t-1, t; frames before 0 are zeros
    assert bench.real_taps(1, 9) == 9
    assert bench.real_taps(2, 9) == 9 + 18
    assert bench.real_taps(4, 9) == 9 + 18 + 27 + 27
    brute = sum(sum(1 for kt in range(3) if t + kt - 2 >= 0) for t in range(8)) * 4
    assert bench.real_taps(8, 4) == brute == 84


def test_algorithmic_work_of_the_convolutions():
    work = bench.algorithmic_work(rescale_bytes=123.0)
    cv, rs = inputs.CONFIGS["mid_conv"], inputs.CONFIGS["resampler"]
    plane = cv.h * cv.w
    # 4 frames: 9 + 18 + 27 + 27 taps of 1024 x 1024 multiply-adds per position
    assert work["conv3d_causal"] == ("tensor", 2.0 * plane * 1024 * 1024 * 81, "flop")
    assert abs(work["conv3d_causal"][1] / 0.583e12 - 1) < 1e-3
    # the resampler: 4 phases x 4 spatial taps x (1 + 2 + 3 x 6) temporal taps per low-res position
    low = rs.h * rs.w
    assert work["resample_up2_fused"][1] == 2.0 * 4 * low * 512 * 512 * 4 * 21
    assert work["resample_up2_fused"] == work["resample_phase_conv"]
    assert work["attn_exp_rescale"] == ("hbm", 123.0, "byte")
    assert work["attn_scores_exp"] == work["attn_scores"] == work["attn_pv_exp"]


def test_history_frames_are_seeded_and_shaped():
    a = inputs.history_frames(1, 64, 3, 5, seed=7)
    b = inputs.history_frames(1, 64, 3, 5, seed=7)
    c = inputs.history_frames(1, 64, 3, 5, seed=8)
    assert a.shape == (1, 2, 3, 5, 64) and a.dtype == torch.bfloat16 and a.is_contiguous()
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_clock_summary_reads_clocks_power_and_reasons():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.samples = [["1900", "2070", "1350.5", "Not Active", "Not Active", "Not Active", "Active"],
                 ["2070", "2070", "1200.0", "Not Active", "Not Active", "Not Active", "Not Active"],
                 ["[N/A]", "2070", "[N/A]", "", "", "", ""]]
    s = c.summary()
    assert s["sm_mhz"] == 1985.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 2
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_median"] == 1275.2 and s["power_w_max"] == 1350.5
    c.samples = []
    assert c.summary()["reasons"] == ["unavailable"]


def test_every_bench_kernel_has_work_sources_and_a_stage():
    work = bench.algorithmic_work(rescale_bytes=1.0)
    for name in bench.KERNELS + bench.ROW_KERNELS:
        assert name in work and name in bench.KERNEL_SOURCES and name in bench.Workload.STAGE_OF, name
        assert len(bench.kernel_source_hash(name)) == 64
    assert len(set(bench.KERNELS + bench.ROW_KERNELS)) == len(bench.KERNELS) + len(bench.ROW_KERNELS)


def test_algorithmic_work_of_the_fused_kernels():
    work = bench.algorithmic_work(rescale_bytes=0.0)
    hd, at = inputs.CONFIGS["head"], inputs.CONFIGS["attention"]
    positions = hd.n * hd.d * hd.h * hd.w
    # the fused head reads x once and writes the 12-channel output once
    assert work["head_out_fused"] == ("hbm", positions * (256 + 12) * 2.0, "byte")
    assert abs(work["head_out_fused"][1] / 1.884e9 - 1) < 1e-3
    # its multiply-adds: the 12-channel conv over real frames (45 of 48
    # temporal taps at 16 frames); the MMAs run 112 columns over 32-column
    # blocks of 30 interior columns (21 per 624-column row) and 89 4-row
    # blocks per strip
    useful, executed = bench.head_tensor_work()
    assert useful == 2.0 * hd.h * hd.w * 12 * 9 * (3 * hd.d - 3) * hd.c
    assert executed == 2.0 * (21 * 32) * (89 * 4) * 112 * (3 * hd.d - 3) * hd.c
    assert 1.12 < executed / useful < 1.14
    # the fused attention is credited with the attention's own products only
    assert work["attn_frame_fused"] == ("tensor", 2 * work["attn_scores"][1], "flop")
    assert work["attn_frame_fused"][1] == 4.0 * at.d * at.hw * at.hw * at.c


def test_profile_kernel_accepts_only_bench_kernels():
    import pytest
    with pytest.raises(SystemExit):
        bench.main(["--profile-kernel", "not_a_kernel"])
