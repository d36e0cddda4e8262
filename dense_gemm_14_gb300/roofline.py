"""Roofline arithmetic for GEMM: FLOP count, algorithmic bytes, peaks.

The formulas are the pages' (gpu-hpc-book ch.06 "高级 cuda 特性 —— 从矩阵乘法(gemm)说起",
opening section and "显性的矩阵乘法性能分析"): a product of n x n matrices costs
2n^3 floating-point operations; with ideal reuse it moves 3n^2 elements (read A
and B once, write C once), operational intensity n/6 for fp32; with no reuse
every multiply-add loads two elements, 8n^3 bytes for fp32. Generalised here
to M x K times K x N with input element size `in_bytes` and output size
`out_bytes`.
"""
from __future__ import annotations

import json
import os


def flops(M: int, N: int, K: int) -> int:
    """2MNK: one multiply and one add per (i, j, k)."""
    return 2 * M * N * K


def ideal_bytes(M: int, N: int, K: int, in_bytes: int = 4, out_bytes: int = 4) -> int:
    """Bytes moved when A and B are read once and C written once."""
    return (M * K + K * N) * in_bytes + M * N * out_bytes


def no_reuse_bytes(M: int, N: int, K: int, in_bytes: int = 4) -> int:
    """Bytes moved when every multiply-add fetches its two operands from memory."""
    return 2 * M * N * K * in_bytes


def intensity(M, N, K, in_bytes=4, out_bytes=4) -> float:
    """Operational intensity (FLOP per byte) with ideal reuse."""
    return flops(M, N, K) / ideal_bytes(M, N, K, in_bytes, out_bytes)


# GB300 unit counts and clock (nominal): 152 SMs, 128 fp32 FMA lanes per SM,
# maximum SM clock 2070 MHz. FFMA counts two FLOPs.
GB300_SMS = 152
GB300_FP32_LANES_PER_SM = 128
GB300_SM_MAX_MHZ = 2070.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def fp32_alu_peak_tflops(sms: int = GB300_SMS, mhz: float = GB300_SM_MAX_MHZ) -> float:
    """FFMA peak: SMs x 128 lanes x 2 FLOP x clock."""
    return sms * GB300_FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12


def measured_peaks(path: str | None = None) -> dict:
    """Peaks for the roofline denominators: the measured file when present,
    else the fallback figures (marked by source='fallback')."""
    if path is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", GB300_SM_MAX_MHZ)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED,
                "sm_max_mhz": GB300_SM_MAX_MHZ, "source": "fallback"}
