"""Reduced workloads that the fp64 oracle finishes in seconds.

Each keeps the structure of one of the five full workloads (dtypes, layout,
shared expert, replica map, router) at sizes that still span several 128-wide
tiles and leave a ragged tail."""
from moe_inputs import CONFIGS

SMALL = {
    "tiny": CONFIGS["tiny"],
    "bf16_masked": CONFIGS["mixtral_decode"].replace(
        name="bf16_masked", T=24, H=256, I=384, E=8, K=2, M_max=24),
    "e4m3_masked_shared": CONFIGS["dsv3_decode"].replace(
        name="e4m3_masked_shared", T=40, H=384, I=256, E=16, K=4, M_max=40),
    "e4m3_eplb_zipf": CONFIGS["skew_eplb"].replace(
        name="e4m3_eplb_zipf", T=48, H=256, I=384, E=16, K=4, M_max=48, redundant=4),
    "e4m3_contig": CONFIGS["prefill"].replace(
        name="e4m3_contig", T=64, H=256, I=256, E=32, K=4),
    # >= 64 expected rows per expert: the token-major GEMM orientation, experts
    # above 128 rows split into near-equal chunks
    "e4m3_contig_tm": CONFIGS["prefill"].replace(
        name="e4m3_contig_tm", T=320, H=384, I=256, E=5, K=2),
    "bf16_masked_tm": CONFIGS["mixtral_decode"].replace(
        name="bf16_masked_tm", T=200, H=256, I=384, E=4, K=2, M_max=200),
    # >= 128 expected rows per expert with H a multiple of 256: both GEMMs on SM pairs (256-row
    # tiles over two CTAs), slots above 256 rows split into near-equal chunks, ragged halves
    "e4m3_contig_pair": CONFIGS["prefill"].replace(
        name="e4m3_contig_pair", T=600, H=512, I=384, E=6, K=3),
    # FP4 (e2m1) experts: the decode shape with a shared expert, and a prefill-sized contiguous one
    "e2m1_masked_shared": CONFIGS["dsv4_fp4_decode"].replace(
        name="e2m1_masked_shared", T=40, H=384, I=256, E=16, K=3, M_max=40),
    "e2m1_contig_tm": CONFIGS["dsv4_fp4_decode"].replace(
        name="e2m1_contig_tm", T=320, H=384, I=256, E=5, K=2, shared=0, layout="contig", M_max=0),
    "e2m1_contig_pair": CONFIGS["dsv4_fp4_decode"].replace(
        name="e2m1_contig_pair", T=520, H=512, I=256, E=4, K=2, shared=0, layout="contig", M_max=0),
}
