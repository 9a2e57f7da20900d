"""Host-side pieces of the benchmark: whole-job throughput over replicas, the
max-over-ranks timing on a real 2-rank process group (gloo, CPU), the
reference arm's rank handling, and the map from every benchmarked workload to
the GPU parity tests that run it at its own size.  No GPU needed."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def test_job_throughput_counts_every_replica():
    flops = 2.0 * 8192 ** 3
    one = bench.job_throughput(flops, 10, 1, 7.0)
    assert abs(one - flops * 10 / 7e-3 / 1e12) < 1e-9
    # four replicas doing the same work in the same (slowest) time: four times the throughput
    assert abs(bench.job_throughput(flops, 10, 4, 7.0) - 4 * one) < 1e-9


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks(3.5) == 3.5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 5.0 + 2.0 * rank              # rank 1 is the slow one
        m = bench.max_over_ranks(local_ms)
        q.put((rank, m, bench.job_throughput(1e12, 3, world, m)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, tput in got:
        assert m == 7.0                           # both ranks see the slowest rank's time
        assert abs(tput - 2 * 1e12 * 3 / 7e-3 / 1e12) < 1e-9


def test_reference_arm_non_zero_rank_does_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, steps, warmup, cpu_seconds = "square8192_bf16", 1, 3, 1.0

    assert bench.run_reference(Args()) is None


def test_attention_workload_shapes_and_flops():
    assert bench.attn_shape("attention_b4h32s4096d128") == (4, 32, 4096, 128)
    assert bench.attn_shape("attention_causal_b4h32s4096d128") == (4, 32, 4096, 128)
    assert bench.attn_shape("attention_b4h32s4096d64") == (4, 32, 4096, 64)
    B, H, S, D = 4, 32, 4096, 128
    # two products of 2 D FLOPs per (query, key) pair: every pair, or the
    # S (S + 1) / 2 pairs on and below the diagonal under the causal mask
    assert bench.attention_flops("attention_b4h32s4096d128") == 4.0 * B * H * S * S * D
    assert bench.attention_flops("attention_causal_b4h32s4096d128") == 4.0 * B * H * D * S * (S + 1) / 2
    # the oracle's unit of work is one head, and the heads add up to the workload
    per, total, _ = bench.oracle_unit("attention_causal_b4h32s4096d128")
    assert total == B * H and per * total == bench.attention_flops("attention_causal_b4h32s4096d128")


def test_gemm_oracle_unit_and_operand_types():
    import torch
    per, total, _ = bench.oracle_unit("square8192_bf16")
    assert total == 8192 and per == 2.0 * 8192 * 8192          # one row of C
    assert bench.fp8_dtype("square8192_e4m3") == torch.float8_e4m3fn
    assert bench.fp8_dtype("square8192_e5m2") == torch.float8_e5m2
    assert bench.fp8_dtype("square8192_tf32") == torch.float32
    assert bench.fp8_dtype("square8192_bf16") is None
    # nominal dense rates relative to bf16: fp8 2x, tf32 1.1 / 2.25
    assert bench.PEAK_RATIO["e4m3"] == bench.PEAK_RATIO["e5m2"] == 2.0
    assert abs(bench.PEAK_RATIO["tf32"] - 1.1 / 2.25) < 1e-12
    for name, (M, N, K, lay, *_rest) in bench.WORKLOADS.items():
        assert M > 0 and N > 0 and K > 0 and lay in ("kn", "nk"), name


# Every benchmarked workload and the GPU parity tests that run it at its own
# size (test file, test function): the benchmark publishes no number for a
# configuration that no parity test covers.
WORKLOAD_TESTS = {
    "square8192_bf16": [("test_fullsize_gpu.py", "test_square_8192_bf16"),
                        ("test_fullsize_gpu.py", "test_square_8192_integer_exact_whole_matrix")],
    "square4096_bf16": [("test_fullsize_gpu.py", "test_square_sweep_integer_exact"),
                        ("test_fullsize_gpu.py", "test_square_sweep_float_sampled")],
    "square2048_bf16": [("test_fullsize_gpu.py", "test_square_sweep_integer_exact")],
    "square1024_bf16": [("test_fullsize_gpu.py", "test_square_sweep_integer_exact")],
    "square512_f32": [("test_gemm_gpu.py", "test_config_512_f32_out")],
    "square8192_nk_bf16": [("test_fullsize_gpu.py", "test_square_nk_weight_layout")],
    "square4096_nk_bf16": [("test_fullsize_gpu.py", "test_square_nk_weight_layout")],
    "qkv_8192x4096x12288": [("test_fullsize_gpu.py", "test_transformer_layers")],
    "ffn_up_8192x4096x14336": [("test_fullsize_gpu.py", "test_transformer_layers")],
    "ffn_down_8192x14336x4096": [("test_fullsize_gpu.py", "test_transformer_layers")],
    "conv_im2col_100352x2304x256": [("test_conv_gpu.py", "test_full_conv_config_sampled")],
    "conv_implicit_32x56x56x256_3x3": [("test_conv_gpu.py", "test_full_conv_config_implicit_sampled")],
    "conv_pool_32x56x56x256_3x3": [("test_fullsize_gpu.py", "test_pooled_conv_full_size_every_output")],
    "odd_3000x5000x2048": [("test_fullsize_gpu.py", "test_odd_shapes")],
    "attention_b4h32s4096d128": [("test_fullsize_gpu.py", "test_attention_full_size_sampled_heads")],
    "attention_causal_b4h32s4096d128": [("test_fullsize_gpu.py", "test_attention_full_size_sampled_heads")],
    "attention_b4h32s4096d64": [("test_fullsize_gpu.py", "test_attention_d64_full_size_sampled_heads")],
    "square8192_e4m3": [("test_fullsize_gpu.py", "test_square_8192_fp8")],
    "square8192_e5m2": [("test_fullsize_gpu.py", "test_square_8192_fp8")],
    "square8192_tf32": [("test_fullsize_gpu.py", "test_square_8192_tf32")],
    "square8192_transa_bf16": [("test_fullsize_gpu.py", "test_square_8192_transposed_a")],
    "odd_4095": [("test_fullsize_gpu.py", "test_odd_shapes")],
    "odd_1000": [("test_fullsize_gpu.py", "test_odd_shapes")],
    "linear_m1_4096x14336": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m16_4096x14336": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m128_4096x14336": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m1_4096x4096": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m2_4096x14336": [("test_warp_mma_gpu.py", "test_warp_mma_decode_layers_every_output")],
    "linear_m4_4096x14336": [("test_fullsize_gpu.py", "test_decode_linear_layers_m4_every_output"),
                             ("test_warp_mma_gpu.py", "test_warp_mma_decode_layers_every_output")],
    "linear_m8_4096x14336": [("test_warp_mma_gpu.py", "test_warp_mma_decode_layers_every_output")],
    "linear_m4_4096x4096": [("test_fullsize_gpu.py", "test_decode_linear_layers_m4_every_output")],
    "linear_m16_4096x4096": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m128_4096x4096": [("test_fullsize_gpu.py", "test_decode_linear_layers_every_output")],
    "linear_m1_4096x14336_e4m3": [("test_fullsize_gpu.py", "test_decode_fp8_layers_every_output")],
    "linear_m4_4096x14336_e4m3": [("test_fullsize_gpu.py", "test_decode_fp8_layers_every_output")],
    "linear_m16_4096x14336_e4m3": [("test_fullsize_gpu.py", "test_decode_fp8_layers_every_output")],
    "linear_m128_4096x14336_e4m3": [("test_fullsize_gpu.py", "test_decode_fp8_layers_every_output")],
}


def test_every_benchmarked_workload_has_a_parity_test_at_its_size():
    import ast
    from pathlib import Path
    here = Path(__file__).resolve().parent
    assert set(WORKLOAD_TESTS) == set(bench.WORKLOADS), "workload list and parity map disagree"
    defined = {}
    for f in {f for tests in WORKLOAD_TESTS.values() for f, _ in tests}:
        tree = ast.parse((here / f).read_text())
        defined[f] = {n.name for n in tree.body if isinstance(n, ast.FunctionDef)}
    for name, tests in WORKLOAD_TESTS.items():
        for f, fn in tests:
            assert fn in defined[f], f"{name}: {f}::{fn} does not exist"
