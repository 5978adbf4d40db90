"""Small and medium parity shapes: each spans several GEMM tiles and has
ragged tails (rows per expert not a multiple of 128, I or H not a multiple of
the tile widths, K not a multiple of 64)."""
from combine_warp_top_gb300 import synth

SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "ragged": synth.Workload("ragged", 300, 256, 8, 2, 384, 4),
    "wide": synth.Workload("wide", 257, 640, 16, 4, 200, 8),
    "odd_h": synth.Workload("odd_h", 150, 200, 6, 3, 136, 3),
    "k_eq_e": synth.Workload("k_eq_e", 40, 128, 8, 8, 128, 2),
    "one_rank": synth.Workload("one_rank", 100, 128, 8, 2, 128, 1),
    "rank_per_expert": synth.Workload("rank_per_expert", 100, 128, 8, 3, 128, 8),
    "e256": synth.Workload("e256", 200, 128, 256, 8, 128, 8),
    "deep_k": synth.Workload("deep_k", 96, 1024, 4, 2, 320, 2),
    # many experts per token: the combine loads a token's rows eight at a
    # time, so these put dedup rows across that boundary (12 over 6 ranks,
    # and the largest k the calls accept, 32 over 16 ranks)
    "k12": synth.Workload("k12", 70, 264, 24, 12, 128, 6),
    "k32": synth.Workload("k32", 40, 136, 64, 32, 128, 16),
}
