"""Helpers shared by the GPU parity tests: run a case through the C ABI with a
guard band around C, and compare with the oracle.

Comparison rules (per element):
* integer inputs: every product and partial sum is an exact integer below
  2^24, so the fp32 accumulator is exact in any order; the output must equal
  the oracle exactly (after one round-to-nearest-even for a 16-bit output);
* float inputs: |C - C_ref| <= 1e-3 * sum_k |A_ik B_kj| + 1e-6, plus one ulp
  of the output type at |C_ref| for a 16-bit output.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G

OUT_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CANARY_BITS = {torch.float32: 0x7FC0DEAD, torch.bfloat16: 0x7FDE, torch.float16: 0x7E5A}


def out_dtype_of(case) -> torch.dtype:
    if case.out == "f32":
        return torch.float32
    return torch.bfloat16 if case.in_dtype == "bf16" else torch.float16


def alloc_with_guard(M: int, N: int, dtype: torch.dtype, pad_cols: int = 8, pad_rows: int = 1,
                     ldc: int | None = None, device="cuda"):
    """C view of M x N inside a buffer filled with a NaN canary pattern."""
    ldc = ldc or (N + pad_cols)
    buf = torch.empty((M + 2 * pad_rows, ldc), dtype=dtype, device=device)
    int_view = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.float16: torch.int16}[dtype]
    bits = CANARY_BITS[dtype]
    if int_view == torch.int16 and bits >= 0x8000:
        bits -= 0x10000
    buf.view(int_view).fill_(bits)
    C = buf[pad_rows:pad_rows + M, :N]
    return buf, C, int_view, bits


def guard_intact(buf, M, N, int_view, bits, pad_rows=1) -> bool:
    raw = buf.view(int_view).cpu()
    mask = torch.ones_like(raw, dtype=torch.bool)
    mask[pad_rows:pad_rows + M, :N] = False
    return bool((raw[mask] == bits).all())


def oracle_full(case, A, B, bias):
    return oracle.gemm(A, B, bias=bias, relu=case.relu, b_nk=case.b_nk, with_mag=True)


def compare(case, C_gpu, C_ref, S):
    """Assert parity; returns the worst error/bound ratio (0 for exact cases)."""
    out16 = case.out != "f32"
    Cg = C_gpu.double().cpu().numpy() if isinstance(C_gpu, torch.Tensor) else C_gpu
    if case.integer:
        if case.out == "f32":
            expect = C_ref
        elif case.in_dtype == "bf16":
            expect = oracle.bf16_round(C_ref)
        else:
            expect = C_ref.astype(np.float16).astype(np.float64)   # exact integers < 2048; rounding RNE
        bad = np.argwhere(Cg != expect)
        assert bad.size == 0, f"{case.name}: {len(bad)} mismatches, first at {bad[0]}: {Cg[tuple(bad[0])]} vs {expect[tuple(bad[0])]}"
        return 0.0
    if out16 and case.in_dtype == "f16":
        # one fp16 ulp at |C_ref| for the fp16 output cast
        ulp = np.spacing(np.abs(C_ref).astype(np.float16)).astype(np.float64)
        bound = 1e-3 * S + 1e-6 + ulp
        err = np.abs(Cg - C_ref)
        ok = bool(np.all(err <= bound))
        worst = float((err / bound).max()) if err.size else 0.0
    else:
        ok, worst, idx = oracle.check_close(Cg, C_ref, S, out_bf16=out16)
    assert ok, f"{case.name}: worst error/bound ratio {worst:.3f}"
    return worst


def run_case(plan: G.Plan, case, device="cuda", guard=True, stream=None, kernel=None):
    """Generate the case, run it through the C ABI, return (A, B, bias, C_gpu on host)."""
    A, B, bias = case.tensors()
    Ad, Bd = A.to(device), B.to(device)
    bd = bias.to(device) if bias is not None else None
    od = out_dtype_of(case)
    if kernel is not None:
        plan.set_kernel(kernel)
    if guard:
        buf, C, iv, bits = alloc_with_guard(case.M, case.N, od, device=device)
    else:
        C = torch.empty((case.M, case.N), dtype=od, device=device)
    plan.run(Ad, Bd, C, bd, case.relu, stream=stream)
    st = plan.status()
    assert st == 0, f"device status {st}"
    if guard:
        assert guard_intact(buf, case.M, case.N, iv, bits), f"{case.name}: write outside C"
    return A, B, bias, C.cpu()


def sample_rows_cols(M, N, tile_m=256, tile_n=256, n_random=32, seed=0):
    """Tile-boundary rows/columns (multiples of 128/256 +-1, first, last) plus random ones."""
    rng = np.random.default_rng(seed)

    def pick(L, t):
        s = {0, L - 1}
        for b in range(0, L, t // 2):
            for d in (-1, 0, 1):
                if 0 <= b + d < L:
                    s.add(b + d)
        s.update(rng.integers(0, L, size=min(n_random, L)).tolist())
        return np.array(sorted(s), dtype=np.int64)

    rows = pick(M, tile_m)
    cols = pick(N, tile_n)
    if len(rows) > 160:
        rows = np.unique(np.concatenate([rows[:: max(1, len(rows) // 120)], [0, M - 1]]))
    if len(cols) > 160:
        cols = np.unique(np.concatenate([cols[:: max(1, len(cols) // 120)], [0, N - 1]]))
    return rows, cols
