"""GPU parity of the attention forward pass (flash_attn_fwd through the C ABI)
against the fp64 oracle, element by element.

"TileLang: a tile language one level below Triton", section "FlashAttention:
online softmax as tile code": O = softmax(scale * Q K^T, causal mask) V on
[batch, seq, heads, dim] arrays. Criterion (per element):
    |o - ref| <= 1e-2 * sum_j p_j |V[j][d]| + 1e-3.

Shapes span several 128-query and 128-key tiles with ragged tails (seq not a
multiple of 128), both head dims (64, 128), both storage types, causal and not;
the full-size workloads are checked on sampled query rows, which the oracle
computes one by one.
"""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
import dense_tiled_gemm_03_gb300 as gt
from dense_tiled_gemm_03_gb300.workloads import ATTN_WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    from _parity import require_gpu
    require_gpu()


def run_flash(q_cpu, k_cpu, v_cpu, causal=True, scale=None):
    """Copy Q, K, V to cuda:0, run flash_attn (O pre-filled with NaN so every
    element must be written), return O on the CPU and the status word."""
    dev = torch.device("cuda", 0)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gt.flash_attn(q, k, v, causal=causal, scale=scale, out=out, status=status)
    torch.cuda.synchronize()
    return out.cpu(), int(status.item())


def assert_attn_parity(o, q, k, v, causal, scale=None, rows=None, label=""):
    ref, bound = oracle.attention_reference(q, k, v, causal=causal, scale=scale, rows=rows)
    got = o if rows is None else o[:, torch.as_tensor(rows, dtype=torch.long)]
    rep = oracle.parity_report(got, ref, bound)
    print(f"{label}: {rep}")
    assert rep.ok, f"{label}: {rep}"
    return rep


SHAPES = [(1, 1, 1), (1, 2, 1), (2, 63, 3), (1, 127, 2), (1, 128, 2), (2, 129, 1), (1, 255, 2), (1, 256, 1),
          (3, 300, 2), (1, 517, 3), (2, 1000, 1)]


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
@pytest.mark.parametrize("bsh", SHAPES, ids=lambda s: "b{}s{}h{}".format(*s))
def test_parity_odd_shapes(bsh, causal, dim, dtype):
    b, s, h = bsh
    q, k, v = make_qkv(b, s, h, dim, dtype, seed=b * 1000 + s * 10 + h + dim)
    o, st = run_flash(q, k, v, causal)
    assert st == 0
    assert_attn_parity(o, q, k, v, causal, label=f"{bsh} d{dim} {dtype} causal={causal}")


def test_the_sections_own_call_full():
    """flash_attn(1, 8, 1024, 64) of the section, fp16, causal: every element."""
    w = ATTN_WORKLOADS["attn_fp16_b1_s1024_h8_d64_causal"]
    q, k, v = make_qkv(w.batch, w.seq, w.heads, w.dim, w.dtype, seed=w.seed)
    o, st = run_flash(q, k, v, w.causal)
    assert st == 0
    assert_attn_parity(o, q, k, v, w.causal, label=w.name)


def _sample_rows(seq: int, n: int = 40, seed: int = 0) -> list[int]:
    """Tile edges, the first and last rows, and random rows."""
    g = np.random.Generator(np.random.PCG64(seed))
    rows = {0, 1, seq - 1, seq // 2}
    for t in range(0, seq, 128 * max(1, seq // (128 * 8))):
        rows.update({t, min(seq - 1, t + 127)})
    rows.update(int(x) for x in g.integers(0, seq, size=n))
    return sorted(r for r in rows if 0 <= r < seq)


@pytest.mark.parametrize("name", [n for n in ATTN_WORKLOADS if n != "attn_fp16_b1_s1024_h8_d64_causal"])
def test_full_size_workloads_sampled(name):
    """The benchmark's workloads at full size, in the launch the benchmark
    times: every batch, head and dim of ~60 sampled query rows."""
    w = ATTN_WORKLOADS[name]
    q, k, v = make_qkv(w.batch, w.seq, w.heads, w.dim, w.dtype, seed=w.seed)
    o, st = run_flash(q, k, v, w.causal)
    assert st == 0
    assert torch.isfinite(o.float()).all()
    assert_attn_parity(o, q, k, v, w.causal, rows=_sample_rows(w.seq, seed=w.seed), label=w.name)


@pytest.mark.parametrize("dim", [64, 128])
def test_explicit_scale(dim):
    q, k, v = make_qkv(2, 333, 2, dim, "bf16", seed=7)
    for scale in (0.05, 0.3):
        o, st = run_flash(q, k, v, True, scale=scale)
        assert st == 0
        assert_attn_parity(o, q, k, v, True, scale=scale, label=f"scale {scale}")


def test_large_scores_stress_the_rescaling():
    """Scores spread over a wide range (scaled-up Q), growing along the keys,
    so the row maximum moves by more than 2^8 several times per row and the
    output rescaling runs."""
    b, s, h, d = 1, 1024, 2, 64
    q, k, v = make_qkv(b, s, h, d, "fp16", seed=11)
    ramp = torch.linspace(0.2, 3.0, s).reshape(1, s, 1, 1)
    q = (q.float() * 4.0).to(torch.float16)
    k = (k.float() * ramp).to(torch.float16)
    for causal in (True, False):
        o, st = run_flash(q, k, v, causal)
        assert st == 0
        assert_attn_parity(o, q, k, v, causal, label=f"wide scores causal={causal}")


def test_closed_forms_on_the_gpu():
    """Zero queries give the mean of the visible values; constant values come
    back (to the output rounding)."""
    b, s, h, d = 2, 300, 2, 128
    _, k, v = make_qkv(b, s, h, d, "bf16", seed=12)
    q = torch.zeros_like(k)
    o, st = run_flash(q, k, v, True)
    assert st == 0
    counts = torch.arange(1, s + 1, dtype=torch.float64).reshape(1, s, 1, 1)
    mean = torch.cumsum(v.double(), dim=1) / counts
    assert (o.double() - mean).abs().max().item() < 1e-2
    c = torch.full_like(v, 0.8125)   # exact in bf16
    o, st = run_flash(q + k, k, c, False)
    assert st == 0
    # the weights sum to one up to the rounding of P (2^-9 relative) and of O
    assert (o.double() - 0.8125).abs().max().item() <= 0.8125 * 2.0 ** -7


def test_repeated_launches_are_bit_identical():
    q, k, v = make_qkv(2, 777, 4, 128, "bf16", seed=13)
    o1, _ = run_flash(q, k, v, True)
    o2, _ = run_flash(q, k, v, True)
    assert torch.equal(o1, o2)


def test_empty_sizes_are_no_ops_and_errors_raise():
    dev = torch.device("cuda", 0)
    q = torch.zeros((0, 16, 2, 64), dtype=torch.float16, device=dev)
    assert gt.flash_attn(q, q, q).shape == q.shape
    q = torch.randn((1, 16, 2, 96), device=dev).to(torch.float16)
    with pytest.raises(gt.GemmTnError, match="INVALID_VALUE"):
        gt.flash_attn(q, q, q)
    x = torch.randn((1, 64 * 2 * 64 + 8), device=dev).to(torch.float16)
    mis = x[0, 8:8 + 64 * 2 * 64].view(1, 64, 2, 64)   # 16-byte aligned + 16: fine
    assert gt.flash_attn(mis, mis, mis).shape == mis.shape
    mis = x[0, 1:1 + 64 * 2 * 64].view(1, 64, 2, 64)   # 2-byte offset
    with pytest.raises(gt.GemmTnError, match="MISALIGNED"):
        gt.flash_attn(mis, mis, mis)
    torch.cuda.synchronize()


def test_watchdog_reports_timeout_and_context_survives():
    """The first CTA's producer skips one K load (test hook), so the MMA
    issuer's bounded wait expires: TIMEOUT must reach the status word within
    the budget, and the next call must be correct."""
    from _parity import env_var
    dev = torch.device("cuda", 0)
    q_cpu, k_cpu, v_cpu = make_qkv(1, 1024, 2, 128, "bf16", seed=14)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    with env_var("GEMM_TN_WATCHDOG_MS", "200"), env_var("GEMM_TN_TEST_DROP_LOAD", "3"):
        gt.flash_attn(q, k, v, causal=True, status=status)
        torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == gt.GEMM_TN_ERR_TIMEOUT
    assert elapsed < 5.0, f"watchdog took {elapsed:.1f} s"
    o, st = run_flash(q_cpu, k_cpu, v_cpu, True)
    assert st == 0
    assert_attn_parity(o, q_cpu, k_cpu, v_cpu, True, label="after watchdog")


def test_runs_on_the_callers_stream_and_in_a_graph():
    q_cpu, k_cpu, v_cpu = make_qkv(1, 640, 4, 64, "fp16", seed=15)
    dev = torch.device("cuda", 0)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gt.flash_attn(q, k, v, out=out)   # warm-up outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gt.flash_attn(q, k, v, out=out)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert_attn_parity(out.cpu(), q_cpu, k_cpu, v_cpu, True, label="graph replay")


def test_long_sequence_sampled():
    """seq = 32768 (256 key tiles, 128 query units per head), one head group;
    checked on sampled rows, including the last ones (they walk every key)."""
    b, s, h, d = 1, 32768, 2, 128
    q, k, v = make_qkv(b, s, h, d, "bf16", seed=16)
    o, st = run_flash(q, k, v, True)
    assert st == 0
    rows = sorted({0, 127, 128, 255, 256, 16383, 16384, s - 129, s - 128, s - 2, s - 1} |
                  set(np.random.Generator(np.random.PCG64(16)).integers(0, s, size=12).tolist()))
    assert_attn_parity(o, q, k, v, True, rows=rows, label="seq 32768")


def test_concurrent_with_a_gemm_on_another_stream():
    """Attention and a GEMM launched on two streams at once (both kernels use
    all of an SM's tensor memory); both results are correct."""
    from dense_tiled_gemm_03_gb300.workloads import make_operands
    dev = torch.device("cuda", 0)
    q_cpu, k_cpu, v_cpu = make_qkv(2, 2048, 4, 128, "bf16", seed=17)
    a_cpu, b_cpu = make_operands(1536, 2560, 1024, "bf16", "uniform", seed=17)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    a, b_ = a_cpu.to(dev), b_cpu.to(dev)
    o = torch.full_like(q, float("nan"))
    c = torch.full((1536, 2560), float("nan"), dtype=torch.bfloat16, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            gt.flash_attn(q, k, v, causal=True, out=o)
        with torch.cuda.stream(s2):
            gt.mm_tn(a, b_, out=c)
    torch.cuda.synchronize()
    assert_attn_parity(o.cpu(), q_cpu, k_cpu, v_cpu, True,
                       rows=list(range(0, 2048, 97)) + [2047], label="concurrent attention")
    ref, bound = oracle.gemm_tn_reference(a_cpu, b_cpu)
    rep = oracle.parity_report(c.cpu(), ref, bound)
    assert rep.ok, rep


def test_dependent_launch_chain():
    """The attention kernel is launched as a programmatic dependent of the
    previous kernel in its stream. A pass whose queries are the previous
    pass's output (pre-filled with NaN just before it), then a GEMM reading
    that output, all back to back with no synchronisation, 10 times: every
    result equals the one computed with synchronisations in between."""
    dev = torch.device("cuda", 0)
    q_cpu, k_cpu, v_cpu = make_qkv(2, 700, 4, 64, "bf16", seed=21)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    o1 = torch.empty_like(q)
    o2 = torch.empty_like(q)
    w = torch.randn(320, 4 * 64, device=dev).to(torch.bfloat16)
    g = torch.empty((2 * 700, 320), dtype=torch.bfloat16, device=dev)

    def chain(sync):
        gt.flash_attn(q, k, v, causal=True, out=o1)
        if sync:
            torch.cuda.synchronize()
        gt.flash_attn(o1, k, v, causal=True, out=o2)
        if sync:
            torch.cuda.synchronize()
        gt.mm_tn(o2.view(2 * 700, 4 * 64), w, out=g)

    chain(True)
    torch.cuda.synchronize()
    expected_o2, expected_g = o2.clone(), g.clone()
    assert torch.isfinite(expected_g.float()).all()
    outs = []
    for _ in range(10):
        o1.fill_(float("nan"))
        o2.fill_(float("nan"))
        chain(False)
        outs.append((o2.clone(), g.clone()))
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(outs):
        assert torch.equal(a, expected_o2), f"iteration {i}: attention read its input early"
        assert torch.equal(b, expected_g), f"iteration {i}: the GEMM read the attention output early"
