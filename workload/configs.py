"""The five synthetic workloads of the Vegas hot path.

Shapes follow the attention layers the pages evaluate (Qwen3-8B: 32 query heads,
8 KV heads, head_dim 128; gpt-oss-20b: 64 query heads, 8 KV heads, head_dim 64)
at the pages' long-context range (32K-128K, LongBench-v2 96K-120K).  The values
are seeded synthetic stand-ins for real activations: no dataset or trained weight
is involved.
"""
from __future__ import annotations

from .gen import Workload

SEED_BASE = 0x5EED0000

TINY = Workload(
    name="tiny", layers=1, batch=1, hq=8, hkv=2, head_dim=64, gamma=4,
    ctx_lo=2048, ctx_hi=2048, heavy_pct=2.0, seed=SEED_BASE + 0, k_abs=128,
    shuffled=False, fp32_source=True,
    description="1 layer, batch 1, context 2048, Hq 8, Hkv 2, d 64, gamma 4, k 128")

QWEN3_8B_B1_32K = Workload(
    name="qwen3_8b_layer_b1_ctx32k", layers=1, batch=1, hq=32, hkv=8, head_dim=128,
    gamma=4, ctx_lo=32768, ctx_hi=32768, heavy_pct=2.0, seed=SEED_BASE + 1, k_pct=5,
    description="Qwen3-8B-shaped layer, batch 1, context 32768, gamma 4, k 5%")

QWEN3_8B_B8_48K_64K = Workload(
    name="qwen3_8b_layer_b8_ctx48k_64k", layers=1, batch=8, hq=32, hkv=8, head_dim=128,
    gamma=5, ctx_lo=49152, ctx_hi=65536, heavy_pct=2.0, seed=SEED_BASE + 2, k_pct=5,
    description="Qwen3-8B-shaped layer, batch 8, context U[48K,64K], gamma 5, k 5%")

GPTOSS_20B_B4_128K = Workload(
    name="gptoss_20b_layer_b4_ctx128k", layers=1, batch=4, hq=64, hkv=8, head_dim=64,
    gamma=6, ctx_lo=131072, ctx_hi=131072, heavy_pct=1.0, heavy_last=512,
    seed=SEED_BASE + 3, k_pct=3,
    description="gpt-oss-20b-shaped layer, batch 4, context 131072, gamma 6, k 3%")

QWEN3_8B_36L_B4_96K_120K = Workload(
    name="qwen3_8b_36layer_b4_ctx96k_120k", layers=36, batch=4, hq=32, hkv=8,
    head_dim=128, gamma=4, ctx_lo=98304, ctx_hi=122880, heavy_pct=2.0,
    seed=SEED_BASE + 4, k_pct=5,
    description="36-layer Qwen3-8B-shaped stack, batch 4, context U[96K,120K]; "
                "sweep gamma in {2,4,6,8} x k in {3,5,10}%")

STACK_SWEEP = [(g, r) for g in (2, 4, 6, 8) for r in (3, 5, 10)]

ALL = [TINY, QWEN3_8B_B1_32K, QWEN3_8B_B8_48K_64K, GPTOSS_20B_B4_128K,
       QWEN3_8B_36L_B4_96K_120K]
BY_NAME = {w.name: w for w in ALL}
