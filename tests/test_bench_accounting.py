"""The benchmark's algorithmic byte counts -- the numerators of every roofline fraction it
reports -- against counts worked out by hand from the model shapes.

A decode token moves every weight byte it needs once (int8 weight + one fp16 scale per 32:
1.0625 bytes per parameter; a MoE token only the router and its top-k experts), the one
embedding row of its token, and the fp16 K and V rows of every position it attends.
"""
import numpy as np

import bench
import synth


def test_dense_8b_token_bytes():
    # per block: QKV (32 + 2 * 8) * 128 = 6144 rows x 4096 = 25,165,824; O 4096 x 4096 =
    # 16,777,216; gate, up, down 3 x 14336 x 4096 = 176,160,768 -> 218,103,808 parameters;
    # 32 blocks = 6,979,321,856, + readout 32000 x 4096 = 131,072,000 -> 7,110,393,856
    params = 7_110_393_856
    w, kv = bench.bytes_per_token(synth.CONFIGS[1], 2048)
    assert w == params * 1.0625 + 4096 * 1.0625
    # K and V: 32 blocks x 2 x 8 heads x 2048 positions x 128 dims x 2 bytes
    assert kv == 268_435_456


def test_moe_token_bytes():
    # per block: QKV (32 + 2 * 4) * 128 = 5120 rows x 2048 = 10,485,760; O 2048 x 4096 =
    # 8,388,608; router 128 x 2048 = 262,144; 8 experts x 3 x 768 x 2048 = 37,748,736
    # -> 56,885,248; 40 blocks = 2,275,409,920, + readout 151936 x 2048 = 311,164,928
    params = 2_586_574_848
    w, kv = bench.bytes_per_token(synth.CONFIGS[2], 4096)
    assert w == params * 1.0625 + 2048 * 1.0625
    # K and V: 40 blocks x 2 x 4 heads x 4096 positions x 128 dims x 2 bytes
    assert kv == 335_544_320


def test_batched_70b_workload_recipe():
    lens = bench.batched_lens(64)
    assert lens.shape == (64,) and lens.min() >= 128 and lens.max() <= 4096
    assert np.array_equal(lens, bench.batched_lens(64))  # seeded
    m = synth.CONFIGS[4]
    # per block: QKV (64 + 2 * 8) * 128 = 10240 rows x 8192 = 83,886,080; O 8192 x 8192 =
    # 67,108,864; gate, up, down 3 x 28672 x 8192 = 704,643,072 -> 855,638,016; 80 blocks =
    # 68,451,041,280, + readout 128256 x 8192 = 1,050,673,152 -> 69,501,714,432
    H = m.hidden
    per = (m.q_dim + 2 * m.kv_dim) * H + H * m.q_dim + 3 * m.ffn * H
    assert per == 855_638_016
    assert per * m.n_layers + m.vocab * H == 69_501_714_432


def test_clock_record_from_sampled_rows():
    """The clocks record of a timed region from nvidia-smi rows (sm, max sm, then the
    hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown and sw_power_cap states): the median
    SM clock under load, the highest max clock, every reason seen Active (never 'Not Active'),
    and rows with unreadable numbers skipped."""
    import bench
    cs = bench.ClockSampler()
    cs.samples = [["2070", "2070", "Not Active", "Not Active", "Not Active", "Not Active"],
                  ["1965", "2070", "Not Active", "Not Active", "Not Active", "Active"],
                  ["2055", "2070", "Not Active", "Not Active", "Not Active", "Not Active"],
                  ["[N/A]", "[N/A]", "Not Active", "Active", "Not Active", "Not Active"]]
    rec = cs.stop()
    assert rec["sm_mhz"] == 2055.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["samples"] == 4
    assert bench.ClockSampler().stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
