"""Roofline arithmetic used by the benchmark.

* FLOPs of a GEMM = 2*M*N*K (one multiply and one add per MAC) and the bytes
  moved = each operand once plus the output once -- youngju.dev "GEMM to
  FlashAttention", the arithmetic-intensity helper and its two printed cases
  (4096^3: about 1370 FLOP/B; 1 x 4096 x 4096: about 1 FLOP/B).  Here the
  element sizes of A, B and C may differ (bf16 in, fp32 or bf16 out) and a
  bias vector is counted when present.
* Roofline: attainable = min(peak compute, intensity x bandwidth); the time
  bound of a kernel is the slower of its FLOPs at peak and its bytes at peak
  bandwidth -- CMU 15-418 "DNNs and ML accelerators" notes, sections 2.5 and 4.1.
* Three-block operational intensity OI(b) = 2b^3 / 3b^2 elements = b/6 FLOP/B
  for fp32 -- same notes, section 4.2.
* Tile counts with partial tiles rounded up (wave quantisation: 1792 -> 98
  tiles, 1793 -> 120 tiles of 256 x 128) -- devpress.csdn.net lecture notes,
  section 3.7.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def matmul_intensity(M: int, K: int, N: int, dtype_bytes: int = 2):
    """(flops, bytes, FLOP/B) of (M x K)(K x N) with one element size."""
    flops = 2 * M * K * N
    nbytes = (M * K + K * N + M * N) * dtype_bytes
    return flops, nbytes, flops / nbytes


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def gemm_bytes(M: int, N: int, K: int, a_bytes: int = 2, b_bytes: int = 2,
               c_bytes: int = 2, bias_bytes: int = 0) -> float:
    """Algorithmic bytes: A, B and C once each, plus the bias vector."""
    return float(M * K * a_bytes + K * N * b_bytes + M * N * c_bytes + N * bias_bytes)


def block_oi(b: int, elem_bytes: int = 4) -> float:
    """FLOP per byte when three b x b blocks are resident: 2b^3 / (3 b^2 elem_bytes)."""
    return 2.0 * b ** 3 / (3.0 * b * b * elem_bytes)


def tile_count(M: int, N: int, tile_m: int, tile_n: int) -> int:
    return math.ceil(M / tile_m) * math.ceil(N / tile_n)


def roofline_time(flops: float, nbytes: float, peak_flops: float, peak_bw: float) -> float:
    """Lower bound on run time: the slower of compute at peak and traffic at peak."""
    return max(flops / peak_flops, nbytes / peak_bw)


def load_peaks(path: str | Path | None = None):
    """Measured peaks of this GPU model (copy bandwidth, dense bf16 FLOP/s),
    or the fallback figures when no measurement file is present.
    Returns (dict, source) with source "measured" or "fallback"."""
    p = Path(path) if path else Path(__file__).resolve().parent.parent / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        out = {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}
        return out, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"
