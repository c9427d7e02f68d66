"""The benchmark's byte / FLOP accounting reproduces the integers the pages
print (no GPU)."""
import bench


def test_io_formulas_match_printed_table():
    # "TileMaxSim" Sec. 2.3, table under Eqs. (3)-(5): Nq = 32, Nd = 128, d = 128, B = 10^4
    assert bench.io_naive_bytes(32, 128, 128, 10_000) == 655_368_192
    assert bench.io_fused_bytes(32, 128, 128, 10_000) == 328_968_192


def test_similarity_tensor_sizes():
    # "Flash-MaxSim" Sec. 1: 10^4 * 1024^2 * 2 bytes, about 21 GB in FP16 (42 GB in FP32)
    assert bench.similarity_bytes(10_000, 1024, 1024, 2) == 20_971_520_000
    assert bench.similarity_bytes(10_000, 1024, 1024, 4) == 41_943_040_000
    # design notes, "Problem": 128 * 128 * 128 * 1024 fp32 values = 8.6 GB
    assert round(bench.similarity_bytes(128 * 128, 128, 1024, 4) / 1e9, 1) == 8.6


def test_argmax_buffer_size():
    # design notes, "Backward": [Nq*Nd, Lq] int32 is 4 MB for Nq = Nd = 64, Lq = 256
    assert bench.argmax_bytes(64, 64, 256) == 4 * 1024 * 1024


def test_fused_arithmetic_intensity():
    # "TileMaxSim" Sec. 2.3: AI 32.0 FLOP/byte fused, 16.1 naive (FLOPs include
    # the max compare: B*Nq*Nd*(2d + 1))
    flops = 10_000 * 32 * 128 * (2 * 128 + 1)
    assert round(flops / bench.io_fused_bytes(32, 128, 128, 10_000), 1) == 32.0
    assert round(flops / bench.io_naive_bytes(32, 128, 128, 10_000), 1) == 16.1
    assert bench.maxsim_flops(32, 128, 128 * 10_000) == 2 * 32 * 128 * 128 * 10_000
