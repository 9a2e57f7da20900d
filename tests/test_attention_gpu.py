"""Fused attention forward (gemm_attention) against the float64 oracle.

Bound: the kernel rounds the probabilities p = 2^(s - m) to the input type
before they multiply V, while the row sum l uses the unrounded values, so each
output moves by at most u * sum_j p_j |V_jd| / l <= u * max_j |V_jd| with u the
unit roundoff of the input type (2^-9 bf16, 2^-12 fp16); the scores, the
exponentials and the fp32 sums add far less.  The test allows 2 u max_j |V_jd|
+ 1e-5, plus one ulp of the output type for a 16-bit output.
"""
import numpy as np
import pytest
import torch

import oracle
from dnn_linear_layers_gb300 import gemm as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from dnn_linear_layers_gb300 import build
    build.build()
    p = G.Plan(0, "nk")
    yield p
    p.close()


def run(plan, B, H, Sq, Sk, D, causal, in_dtype=torch.bfloat16, out_dtype=torch.float32, seed=0, scale=0.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, D, generator=g).to(in_dtype)
    k = torch.randn(B, H, Sk, D, generator=g).to(in_dtype)
    v = torch.randn(B, H, Sk, D, generator=g).to(in_dtype)
    o = torch.full((B, H, Sq, D), float("nan"), dtype=out_dtype, device="cuda")
    plan.attention(q.cuda(), k.cuda(), v.cuda(), o, scale=scale, causal=causal)
    assert plan.status() == 0
    ref = oracle.attention(q, k, v, scale=None if scale <= 0 else scale, causal=causal)
    got = o.double().cpu().numpy()
    u = 2.0 ** -9 if in_dtype == torch.bfloat16 else 2.0 ** -12
    vmax = np.abs(oracle._f64(v)).max(axis=-2, keepdims=True)          # per (b, h, d)
    bound = 2 * u * vmax + 1e-5
    if out_dtype == torch.bfloat16:
        bound = bound + oracle.ulp_bf16(ref)
    elif out_dtype == torch.float16:
        bound = bound + np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    worst = float((err / bound).max()) if err.size else 0.0
    assert np.all(err <= bound), f"worst err/bound {worst:.3f}"
    return worst


@pytest.mark.parametrize("shape", [(1, 2, 128, 128, 64), (1, 1, 300, 300, 128), (2, 3, 257, 513, 64),
                                   (1, 1, 64, 1000, 128), (1, 2, 513, 200, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_matches_oracle(plan, shape, causal):
    B, H, Sq, Sk, D = shape
    run(plan, B, H, Sq, Sk, D, causal, seed=sum(shape) + causal)


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_attention_fp16_and_bf16_outputs(plan, out):
    run(plan, 1, 2, 200, 300, 64, False, in_dtype=torch.float16, out_dtype=torch.float16 if out == torch.bfloat16 else out, seed=3)
    run(plan, 2, 1, 130, 130, 128, True, in_dtype=torch.bfloat16, out_dtype=out, seed=4)


def test_attention_scale_and_empty_rows(plan):
    run(plan, 1, 1, 256, 256, 64, False, seed=5, scale=0.05)
    # causal with more queries than keys: the first Sq - Sk queries see nothing -> zeros
    B, H, Sq, Sk, D = 1, 1, 300, 100, 64
    q = torch.randn(B, H, Sq, D).bfloat16().cuda()
    k = torch.randn(B, H, Sk, D).bfloat16().cuda()
    v = torch.randn(B, H, Sk, D).bfloat16().cuda()
    o = torch.full((B, H, Sq, D), float("nan"), device="cuda")
    plan.attention(q, k, v, o, causal=True)
    assert plan.status() == 0
    assert torch.all(o[:, :, :Sq - Sk] == 0)
    # no keys at all
    o2 = torch.full((1, 1, 10, 64), float("nan"), device="cuda")
    plan.attention(q[:, :, :10], k[:, :, :0], v[:, :, :0], o2)
    assert torch.all(o2 == 0)


def test_attention_rejects_bad_head_dim(plan):
    q = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(G.GemmError) as e:
        plan.attention(q, q, q, torch.zeros(1, 1, 8, 96, device="cuda"))
    assert e.value.code == G.ERR_UNSUPPORTED


@pytest.mark.parametrize("causal", [False, True])
def test_attention_persistent_many_items_per_cta(plan, causal):
    # 160 heads x 3 query blocks = 480 items: every CTA walks several items (in
    # pairs under the causal mask), so barrier phases carry across items
    run(plan, 2, 80, 300, 260, 64, causal, seed=40 + causal)


def test_attention_persistent_with_empty_items(plan):
    # causal with twice as many queries as keys: the first query blocks of every
    # head see no key (items with no key block) between items that do
    run(plan, 1, 160, 600, 300, 64, True, seed=42)


def test_attention_persistent_d128_bf16_out(plan):
    run(plan, 1, 64, 640, 512, 128, True, out_dtype=torch.bfloat16, seed=43)


def test_attention_bounded_wait_reports_timeout_and_context_survives():
    """Fault injection on the host's request: the PV issuer withholds the first
    'product done' signal, a softmax wait runs out, every role leaves through
    its bounded waits, the run reports GEMM_ERR_DEVICE_TIMEOUT, and the next
    run on the same context matches the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    with G.Plan(0, "nk") as p:
        p.set_timeout_ns(20_000_000)          # 20 ms
        g = torch.Generator().manual_seed(50)
        q = torch.randn(1, 2, 512, 64, generator=g).bfloat16()
        k = torch.randn(1, 2, 512, 64, generator=g).bfloat16()
        v = torch.randn(1, 2, 512, 64, generator=g).bfloat16()
        o = torch.zeros(1, 2, 512, 64, device="cuda")
        p.set_debug(1)
        p.attention(q.cuda(), k.cuda(), v.cuda(), o)
        assert p.status() == G.ERR_DEVICE_TIMEOUT
        p.set_debug(0)
        p.attention(q.cuda(), k.cuda(), v.cuda(), o)
        assert p.status() == 0
        ref = oracle.attention(q, k, v)
        vmax = np.abs(oracle._f64(v)).max(axis=-2, keepdims=True)
        assert np.all(np.abs(o.double().cpu().numpy() - ref) <= 2 * 2.0 ** -9 * vmax + 1e-5)


def test_attention_module_function():
    # gemm.attention allocates the output (the input dtype unless told otherwise)
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    g = torch.Generator().manual_seed(70)
    q = torch.randn(2, 3, 200, 64, generator=g).bfloat16()
    k = torch.randn(2, 3, 260, 64, generator=g).bfloat16()
    v = torch.randn(2, 3, 260, 64, generator=g).bfloat16()
    o = G.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.float32)
    assert o.dtype == torch.float32 and tuple(o.shape) == (2, 3, 200, 64)
    ref = oracle.attention(q, k, v, causal=True)
    vmax = np.abs(oracle._f64(v)).max(axis=-2, keepdims=True)
    assert np.all(np.abs(o.double().cpu().numpy() - ref) <= 2 * 2.0 ** -9 * vmax + 1e-5)

