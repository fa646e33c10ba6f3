"""GPU parity of the sm_103a GEMM against the fp64 oracle, through the C ABI.

Pass criterion for every element: |c - ref| <= 1e-2 * sum_k |a_ik * b_jk| + 1e-3,
no NaN/Inf (C is pre-filled with NaN, so every element must be written).
Exactness where the arithmetic is exact: small-integer operands, identity and
permutation matrices. Edge cases: empty and ragged shapes, K = 0, padded and
misaligned strides, misaligned base pointers, repeated launches.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dense_tiled_gemm_03_gb300 as gt
from dense_tiled_gemm_03_gb300.workloads import WORKLOADS, make_operands, workload_operands

from _parity import (assert_parity, assert_sampled_parity, edge_indices, epilogue_mode, forced_config, gpu_gemm,
                     require_gpu)

pytestmark = pytest.mark.gpu

CONFIGS = ["1cta_n256", "1cta_n128", "1cta_n64", "2cta_n128", "2cta_n256", "2cta_n256_mc", "1cta_n128_splitk",
           "1cta_decode_splitk"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    from dense_tiled_gemm_03_gb300 import build as native_build
    native_build.build()
    torch.cuda.init()


# ------------------------------------------------------------ small and odd shapes

ODD_SHAPES = [(1, 1, 1), (1, 1, 64), (7, 13, 17), (128, 256, 64), (129, 257, 65), (255, 511, 130),
              (300, 200, 1000), (64, 1024, 8), (513, 129, 200), (1000, 1000, 64)]


@pytest.mark.parametrize("epilogue", ["auto", "direct"])
@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("mnk", ODD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_odd_shapes(mnk, dtype, config, epilogue):
    m, n, k = mnk
    a, b = make_operands(m, n, k, dtype, "uniform", seed=m * 131 + n * 7 + k)
    c, status = gpu_gemm(a, b, config, epilogue=epilogue)
    assert status == 0
    assert_parity(c, a, b, f"{mnk} {dtype} {config} {epilogue}")


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("mn", [(257, 250), (1000, 1003), (129, 40), (300, 1000), (1001, 264)])
def test_ragged_output_with_aligned_pitch(mn, config):
    """Ragged M and N but a C pitch that is a multiple of 8: the epilogue goes
    through TMA stores whose boxes are clipped at M and N; the pad columns of
    C must stay untouched."""
    m, n = mn
    k = 320
    ldc = (n + 7) // 8 * 8 + 8
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=m + n)
    c_big = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device=dev)
    c = c_big[:, :n]
    with forced_config(config):
        gt.mm_tn(a_cpu.to(dev), b_cpu.to(dev), out=c)
    torch.cuda.synchronize()
    assert_parity(c.cpu(), a_cpu, b_cpu, f"{mn} {config}")
    assert torch.isnan(c_big[:, n:].float()).all(), "wrote past N"


# ------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("name", ["fp16_256x256x256", "fp16_4096x4096x4096", "fp16_3001x5003x4097",
                                  "bf16_128x16384x16384", "bf16_8x4096x4096"])
def test_workload_full_parity(name):
    """Element-by-element parity over the whole output, default configuration."""
    a, b = workload_operands(name)
    c, status = gpu_gemm(a, b)
    assert status == 0
    assert_parity(c, a, b, name)


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("name", ["fp16_256x256x256", "fp16_3001x5003x4097"])
def test_workload_parity_every_config(name, config):
    a, b = workload_operands(name)
    c, status = gpu_gemm(a, b, config)
    assert status == 0
    assert_parity(c, a, b, f"{name} {config}")


@pytest.fixture(scope="module")
def headline_reference():
    """The bf16 8192^3 workload's operands with the oracle's ref and bound over
    the whole output, computed once for the module (about 25 s on 16 host
    cores): the plain, [K, N] and fused headline checks all compare with it."""
    import oracle
    w = WORKLOADS["bf16_8192x8192x8192"]
    a, b = workload_operands(w)
    ref, bound = oracle.gemm_tn_reference(a, b)
    return w, a, b, ref, bound


def test_headline_workload_full_parity(headline_reference):
    """bf16 8192^3 in the configuration the benchmark runs: every one of the
    67M output elements against the oracle."""
    import oracle
    w, a, b, ref, bound = headline_reference
    c, status = gpu_gemm(a, b)
    assert status == 0
    rep = oracle.parity_report(c, ref, bound)
    assert rep.ok, f"{w.name}: {rep}"


def test_multicast_guard_on_the_device():
    """The multicast configuration reads only this GPU's own memory: device
    tensors pass the check, pinned and pageable host memory do not, and a
    shape the selection sends to the multicast kernel runs it on device
    operands (with parity)."""
    dev = torch.device("cuda", 0)
    a = torch.empty(4096, dtype=torch.float16, device=dev)
    b = torch.empty(4096, dtype=torch.float16, device=dev)
    pinned = torch.empty(4096, dtype=torch.float16).pin_memory()
    pageable = torch.empty(4096, dtype=torch.float16)
    assert gt.gemm_tn_multicast_allowed(a.data_ptr(), b.data_ptr()) == 1
    assert gt.gemm_tn_multicast_allowed(pinned.data_ptr(), b.data_ptr()) == 0
    assert gt.gemm_tn_multicast_allowed(a.data_ptr(), pinned.data_ptr()) == 0
    assert gt.gemm_tn_multicast_allowed(pageable.data_ptr(), b.data_ptr()) == 0
    m, n, k = 2560, 2560, 1024
    assert gt.gemm_tn_config_name(gt.gemm_tn_select_config(gt.GEMM_TN_F16, m, n, k)) == "2cta_n256_mc"
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=17)
    c, status = gpu_gemm(a_cpu, b_cpu)
    assert gt.gemm_tn_config_name(gt.gemm_tn_last_config()) == "2cta_n256_mc"
    assert status == 0
    assert_parity(c, a_cpu, b_cpu, "multicast on device operands")


# ------------------------------------------------------------ exact cases

@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_small_integers_are_exact(dtype, config):
    # entries in {-2..2}, K = 64: |C| <= 256, exact in fp32 and in both 16-bit types
    m, n, k = 300, 400, 64
    a, b = make_operands(m, n, k, dtype, "int_small", seed=77)
    c, status = gpu_gemm(a, b, config)
    assert status == 0
    exact = (a.long() @ b.long().T)
    assert torch.equal(c.double(), exact.double()), "integer product not reproduced exactly"


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_identity_and_permutation_reproduce_a(dtype, config):
    m, k = 333, 256
    a, _ = make_operands(m, 1, k, dtype, "uniform", seed=5)
    eye = torch.eye(k, dtype=a.dtype)
    c, _ = gpu_gemm(a, eye, config)
    assert torch.equal(c, a)
    perm = torch.from_numpy(np.random.Generator(np.random.PCG64(3)).permutation(k))
    p = torch.zeros((k, k), dtype=a.dtype)
    p[torch.arange(k), perm] = 1
    c, _ = gpu_gemm(a, p, config)
    assert torch.equal(c, a[:, perm])


def test_all_ones_gives_k():
    for k in (256, 4096):
        a = torch.ones((200, k), dtype=torch.float16)
        b = torch.ones((300, k), dtype=torch.float16)
        c, _ = gpu_gemm(a, b)
        assert (c.double() == k).all()


# ------------------------------------------------------------ edge cases

def test_k_zero_writes_zeros():
    a = torch.empty((10, 0), dtype=torch.bfloat16)
    b = torch.empty((20, 0), dtype=torch.bfloat16)
    c, status = gpu_gemm(a, b)
    assert status == 0 and (c == 0).all()


def test_empty_m_or_n_is_noop():
    dev = torch.device("cuda", 0)
    a = torch.ones((0, 8), dtype=torch.float16, device=dev)
    b = torch.ones((5, 8), dtype=torch.float16, device=dev)
    out = gt.mm_tn(a, b)
    assert out.shape == (0, 5)
    out = gt.mm_tn(b, a)
    assert out.shape == (5, 0)


@pytest.mark.parametrize("pad", [(8, 8, 8), (3, 5, 7), (0, 0, 5), (1, 0, 0)])
def test_padded_and_misaligned_strides(pad):
    """Row pitches larger than the logical width: multiples of 8 use the TMA
    directly, others go through the repack workspace; any ldc is stored with
    predicated element stores."""
    pa, pb, pc = pad
    m, n, k = 300, 333, 200
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=sum(pad))
    a_big = torch.zeros((m, k + pa), dtype=torch.float16)
    a_big[:, :k] = a_cpu
    b_big = torch.zeros((n, k + pb), dtype=torch.float16)
    b_big[:, :k] = b_cpu
    a = a_big.to(dev)[:, :k]
    b = b_big.to(dev)[:, :k]
    c_big = torch.full((m, n + pc), float("nan"), dtype=torch.float16, device=dev)
    c = c_big[:, :n]
    gt.mm_tn(a, b, out=c)
    torch.cuda.synchronize()
    assert_parity(c.cpu(), a_cpu, b_cpu, f"pad {pad}")
    if pc:
        assert torch.isnan(c_big[:, n:].float()).all(), "wrote outside C"


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("k", [203, 1001, 65])
def test_k_tail_with_aligned_pitch_ignores_padding(k, config):
    """K not a multiple of 8 but row pitches that are (no repack): the pad
    columns past K hold NaN and must never reach the product."""
    m, n = 300, 264
    ld = (k + 7) // 8 * 8 + 8
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=k)
    a_big = torch.full((m, ld), float("nan"), dtype=torch.float16)
    a_big[:, :k] = a_cpu
    b_big = torch.full((n, ld), float("nan"), dtype=torch.float16)
    b_big[:, :k] = b_cpu
    c = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
    with forced_config(config):
        gt.mm_tn(a_big.to(dev)[:, :k], b_big.to(dev)[:, :k], out=c)
    torch.cuda.synchronize()
    assert_parity(c.cpu(), a_cpu, b_cpu, f"k={k} {config}")


def test_misaligned_base_pointers():
    """Operands starting 2 bytes past a 16-byte boundary (repack path) and an
    output starting 2 bytes past one (predicated stores)."""
    m, n, k = 257, 129, 4097
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=9)
    a_buf = torch.zeros(m * k + 1, dtype=torch.bfloat16, device=dev)
    a_buf[1:] = a_cpu.flatten().to(dev)
    b_buf = torch.zeros(n * k + 1, dtype=torch.bfloat16, device=dev)
    b_buf[1:] = b_cpu.flatten().to(dev)
    c_buf = torch.full((m * n + 1,), float("nan"), dtype=torch.bfloat16, device=dev)
    a = a_buf[1:].view(m, k)
    b = b_buf[1:].view(n, k)
    c = c_buf[1:].view(m, n)
    assert a.data_ptr() % 16 == 2
    gt.mm_tn(a, b, out=c)
    torch.cuda.synchronize()
    assert_parity(c.cpu(), a_cpu, b_cpu, "misaligned base")
    assert torch.isnan(c_buf[:1].float()).all()


@pytest.mark.parametrize("offset", [1, 3, 5, 7])
@pytest.mark.parametrize("k", [1, 7, 9, 63, 65, 200])
def test_repack_every_byte_offset(offset, k):
    """Operands starting 2, 6, 10 or 14 bytes past a 16-byte boundary with
    pitches that are not multiples of 8: the repack cuts every 16-byte chunk
    out of two aligned source blocks; NaN guards around the data must never
    reach C."""
    m, n = 131, 77
    ld = k + 3
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=offset * 100 + k)
    def planted(t):
        rows = t.shape[0]
        buf = torch.full((offset + rows * ld + 16,), float("nan"), dtype=t.dtype)
        view = buf[offset:offset + rows * ld].view(rows, ld)
        view[:, :k] = t
        return buf.to(dev), offset
    a_buf, _ = planted(a_cpu)
    b_buf, _ = planted(b_cpu)
    a = a_buf[offset:offset + m * ld].view(m, ld)[:, :k]
    b = b_buf[offset:offset + n * ld].view(n, ld)[:, :k]
    assert a.data_ptr() % 16 == 2 * offset
    c = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
    gt.mm_tn(a, b, out=c)
    torch.cuda.synchronize()
    assert_parity(c.cpu(), a_cpu, b_cpu, f"offset {offset} k {k}")


@pytest.mark.parametrize("epilogue", ["auto", "direct"])
@pytest.mark.parametrize("config", CONFIGS)
def test_repeated_launches_are_bit_identical(config, epilogue):
    """NaN canary + determinism: C is re-filled with NaN before each launch,
    every launch must overwrite all of it, and all launches agree bit for bit
    (a corrupted barrier shows up as sporadic NaNs or differences)."""
    m, n, k = 1000, 1200, 1024
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=31)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    first = None
    with forced_config(config), epilogue_mode(epilogue):
        for _ in range(20):
            out.fill_(float("nan"))
            gt.mm_tn(a, b, out=out)
            got = out.clone()
            if first is None:
                first = got
            else:
                assert torch.equal(got.view(torch.int16), first.view(torch.int16))
    torch.cuda.synchronize()
    assert not torch.isnan(first.float()).any()
    assert_parity(first.cpu(), a_cpu, b_cpu, config)


def test_plain_entry_point_and_host_entry_point_agree():
    """gemm_tn (device pointers, contiguous) and gemm_tn_host (host buffers,
    copies inside the call) give the same bits as gemm_tn_ex."""
    m, n, k = 640, 768, 512
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "normal_over_sqrt_k", seed=12)
    c_ex, _ = gpu_gemm(a_cpu, b_cpu)
    dev = torch.device("cuda", 0)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    c = torch.empty((m, n), dtype=torch.float16, device=dev)
    rc = gt.gemm_tn(gt.GEMM_TN_F16, m, n, k, a.data_ptr(), b.data_ptr(), c.data_ptr(),
                    torch.cuda.current_stream().cuda_stream)
    assert rc == gt.GEMM_TN_OK
    torch.cuda.synchronize()
    assert torch.equal(c.cpu(), c_ex)
    c_host = gt.mm_tn_host(a_cpu.pin_memory(), b_cpu.pin_memory())
    assert torch.equal(c_host, c_ex)
    c_host = gt.mm_tn_host(a_cpu, b_cpu)   # pageable
    assert torch.equal(c_host, c_ex)


# ------------------------------------------------------------ device watchdog

@pytest.mark.parametrize("config", ["1cta_n256", "2cta_n256", "1cta_n128_splitk", "1cta_decode_splitk"])
def test_watchdog_reports_timeout_and_context_survives(config):
    """A wait that can never complete (the producer skips one k-block's loads
    through the test hook) must end within the watchdog budget with
    GEMM_TN_ERR_TIMEOUT in the status word; afterwards the context is usable
    and a normal call is correct."""
    import time
    from _parity import env_var
    # the decode kernel runs only for M <= 32 (a forced decode configuration
    # with more rows runs the 128 x 128 split-K kernel instead)
    m = 8 if config == "1cta_decode_splitk" else 512
    n, k = 512, 1024
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=4)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    out = torch.zeros((m, n), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    # load 1 (counted from the start of each CTA's K range) exists for every
    # configuration: K = 1024 has 16 k-blocks, and the split-K kernels keep
    # at least 4 per CTA here (512 x 512 x 1024 at S = 4; 8 x 512 x 1024 at
    # S = 2 or 4), which they move in copies of two
    with forced_config(config), env_var("GEMM_TN_WATCHDOG_MS", "200"), env_var("GEMM_TN_TEST_DROP_LOAD", "1"):
        gt.mm_tn(a, b, out=out, status=status)
        ran = gt.gemm_tn_config_name(gt.gemm_tn_last_config())
        torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert ran == config, f"forced {config} but {ran} ran"
    assert int(status.item()) == gt.GEMM_TN_ERR_TIMEOUT
    assert elapsed < 5.0, f"watchdog took {elapsed:.1f} s"
    status.zero_()
    c, st = gpu_gemm(a_cpu, b_cpu, config)
    assert st == 0
    assert_parity(c, a_cpu, b_cpu, "after watchdog")


# ------------------------------------------------------------ stream-K tail

@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("mnk", [(256, 512, 8192), (300, 1000, 3000), (2000, 2100, 640), (2304, 4352, 1000),
                                 (128, 4096, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_stream_k_cut_tiles(mnk, config):
    """Shapes whose tiles do not fill whole waves: the last tiles are cut by
    k-block ranges across workers (up to ~16 contributors per tile when there
    are fewer tiles than workers; mode 3 cuts each partial-wave tile into equal
    parts, one per worker) and finished by the worker holding their first
    k-block. Parity with stream-K on in every mode, and with it off."""
    from _parity import env_var
    m, n, k = mnk
    a, b = make_operands(m, n, k, "bf16", "normal_over_sqrt_k", seed=m ^ n ^ k)
    for sk in ("1", "2", "3", "0"):
        with env_var("GEMM_TN_STREAMK", sk):
            c, status = gpu_gemm(a, b, config)
        assert status == 0
        assert_parity(c, a, b, f"{mnk} {config} streamk={sk}")


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("mnk", [(128, 4096, 4160), (100, 3000, 1000), (300, 1000, 3000), (8, 640, 64 * 37 + 5)],
                         ids=lambda s: "x".join(map(str, s)))
def test_k_rotation(mnk, config):
    """Tiles that start their K walk at a hashed k-block and wrap around (the
    default for one row of tiles, forced on here for every configuration and
    shape, with and without the stream-K tail, whose partial items keep the
    plain order): parity both ways, and repeated launches bit-identical."""
    from _parity import env_var
    m, n, k = mnk
    a, b = make_operands(m, n, k, "bf16", "uniform", seed=m + 3 * n + k)
    for sk in ("0", "1"):
        outs = []
        for rot in ("1", "0", "1"):
            with env_var("GEMM_TN_K_ROTATE", rot), env_var("GEMM_TN_STREAMK", sk):
                c, status = gpu_gemm(a, b, config)
            assert status == 0
            assert_parity(c, a, b, f"{mnk} {config} rotate={rot} streamk={sk}")
            outs.append(c)
        assert torch.equal(outs[0], outs[2]), "rotated launches differ"


@pytest.mark.parametrize("pad", [0, 1])
def test_dependent_launch_chain(pad):
    """Kernels are launched as programmatic dependents of the previous kernel
    in the stream: their set-up may overlap it, their memory accesses may not.
    Call 2 reads call 1's output (pre-filled with NaN just before call 1),
    back to back with no synchronisation, 20 times; with pad = 1 that output
    has an odd row pitch, so call 2 first repacks it (the repack kernel is a
    dependent of call 1, and call 2's GEMM of the repack). Every result must
    equal the one computed with a synchronisation between the calls."""
    dev = torch.device("cuda", 0)
    m, k1, k2, n2 = 1000, 640, 1536, 700
    a_cpu, b_cpu = make_operands(m, k2, k1, "fp16", "normal_over_sqrt_k", seed=31)
    _, d_cpu = make_operands(m, n2, k2, "fp16", "normal_over_sqrt_k", seed=32)
    a, b, d = a_cpu.to(dev), b_cpu.to(dev), d_cpu.to(dev)
    c1_big = torch.empty((m, k2 + pad), dtype=torch.float16, device=dev)
    c1 = c1_big[:, :k2]
    c2 = torch.empty((m, n2), dtype=torch.float16, device=dev)
    gt.mm_tn(a, b, out=c1)
    torch.cuda.synchronize()
    gt.mm_tn(c1, d, out=c2)
    torch.cuda.synchronize()
    expected = c2.clone()
    assert torch.isfinite(expected.float()).all()
    outs = []
    for _ in range(20):
        c1_big.fill_(float("nan"))
        c2.fill_(float("nan"))
        gt.mm_tn(a, b, out=c1)
        gt.mm_tn(c1, d, out=c2)
        outs.append(c2.clone())
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, expected), f"iteration {i}: a dependent call read its input before the previous call finished"


@pytest.mark.parametrize("splits", ["2", "4", "8"])
@pytest.mark.parametrize("mnk", [(128, 1024, 4096), (16, 4096, 2048), (300, 700, 1000), (129, 257, 513),
                                 (1, 1, 1024), (200, 390, 4097), (256, 384, 1216), (64, 300, 320)],
                         ids=lambda s: "x".join(map(str, s)))
def test_split_k_over_a_cluster(mnk, splits):
    """K cut over a cluster of 2, 4 or 8 CTAs per 128 x 128 tile, the fp32
    partials added through distributed shared memory in CTA order: parity for
    ragged M, N, K (K = 4097 also repacks A and B), an odd C pitch written
    only inside N, and bit-identical results on repeated launches. With K a
    multiple of 64 each copy moves two k-blocks (1216 = 19 x 64 leaves the
    last copy's second k-block past K; 320 = 5 x 64 has fewer pairs than CTAs
    at S = 4 and keeps one k-block per copy)."""
    from _parity import env_var
    m, n, k = mnk
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "normal_over_sqrt_k", seed=m + n + k + int(splits))
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    ldc = n + 3
    outs = []
    for _ in range(2):
        c_big = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device=dev)
        c = c_big[:, :n]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        with forced_config("1cta_n128_splitk"), env_var("GEMM_TN_SPLITK", splits):
            gt.mm_tn(a, b, out=c, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isnan(c_big[:, n:].float()).all(), "wrote past N"
        outs.append(c.cpu())
    assert_parity(outs[0], a_cpu, b_cpu, f"{mnk} split {splits}")
    assert torch.equal(outs[0], outs[1]), "split-K launches differ"


@pytest.mark.parametrize("splits", ["2", "4", "8"])
@pytest.mark.parametrize("mnk", [(1, 4096, 4096), (8, 1000, 2048), (16, 300, 1000), (17, 640, 4097), (32, 129, 512),
                                 (33, 4000, 8192), (64, 2048, 1024), (8, 512, 4160), (24, 384, 1472), (5, 700, 576)],
                         ids=lambda s: "x".join(map(str, s)))
def test_decode_split_k(mnk, splits):
    """At most 32 rows of A: B's rows on the MMA's M side and A's rows
    (zero-filled to 16 or 32) on its N side (a forced decode configuration
    with more rows runs the 128 x 128 split-K kernel), K split over a cluster, C
    stored column by column: parity, nothing written past N into C's padded
    pitch, and bit-identical results on repeated launches. With K a multiple
    of 64 each copy moves two k-blocks (an odd count leaves the last copy's
    second k-block past K: 4160 = 65 x 64, 1472 = 23 x 64, 576 = 9 x 64; with
    fewer pairs than CTAs, 576 at S = 8, one k-block per copy instead)."""
    from _parity import env_var
    m, n, k = mnk
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "normal_over_sqrt_k", seed=m * 7 + n + k + int(splits))
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    ldc = n + 5
    outs = []
    for _ in range(2):
        c_big = torch.full((m, ldc), float("nan"), dtype=torch.float16, device=dev)
        c = c_big[:, :n]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        with forced_config("1cta_decode_splitk"), env_var("GEMM_TN_SPLITK", splits):
            gt.mm_tn(a, b, out=c, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isnan(c_big[:, n:].float()).all(), "wrote past N"
        outs.append(c.cpu())
    assert_parity(outs[0], a_cpu, b_cpu, f"{mnk} decode split {splits}")
    assert torch.equal(outs[0], outs[1]), "decode launches differ"


@pytest.mark.parametrize("config", ["1cta_n64", "1cta_n128"])
@pytest.mark.parametrize("mnk", [(256, 256, 192), (300, 520, 1216), (1000, 700, 64), (129, 1000, 4032)],
                         ids=lambda s: "x".join(map(str, s)))
def test_single_cta_two_k_blocks_per_copy(mnk, config):
    """128 x 64 and 128 x 128 tiles with K a multiple of 64 move two k-blocks
    per copy: an odd k-block count (3, 19, 63) leaves the last copy's second
    k-block past K, and K = 64 has only that one; ragged M and N. Parity in
    both dtypes and bit-identical repeated launches."""
    m, n, k = mnk
    for dtype in ("fp16", "bf16"):
        a_cpu, b_cpu = make_operands(m, n, k, dtype, "normal_over_sqrt_k", seed=m + 3 * n + k)
        outs = []
        for _ in range(2):
            c, st = gpu_gemm(a_cpu, b_cpu, config)
            assert st == 0
            assert gt.gemm_tn_config_name(gt.gemm_tn_last_config()) == config
            outs.append(c)
        assert_parity(outs[0], a_cpu, b_cpu, f"{mnk} {config} {dtype}")
        assert torch.equal(outs[0], outs[1]), "launches differ"


@pytest.mark.parametrize("mnk", [(8, 4096, 4096), (32, 2048, 4160), (3, 1000, 2048)], ids=lambda s: "x".join(map(str, s)))
def test_decode_bf16_default_choice(mnk):
    """bf16 decode-like shapes through the default selection (the decode
    kernel with two k-blocks per copy, K a multiple of 64, odd k-block count
    included): parity, and bit-identical repeated launches."""
    m, n, k = mnk
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "normal_over_sqrt_k", seed=m + n + k)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    outs = []
    for _ in range(2):
        c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        gt.mm_tn(a, b, out=c, status=status)
        assert gt.gemm_tn_config_name(gt.gemm_tn_last_config()) == "1cta_decode_splitk"
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(c.cpu())
    assert_parity(outs[0], a_cpu, b_cpu, f"{mnk} bf16 decode")
    assert torch.equal(outs[0], outs[1]), "decode launches differ"


def test_split_k_is_chosen_for_few_tiles_and_matches_whole_tiles():
    """The default choice for 128 x 4096 x 4096 is the split-K cluster; its
    result is within the criterion of the whole-K single-CTA tiles'."""
    m, n, k = 128, 4096, 4096
    a, b = make_operands(m, n, k, "fp16", "normal_over_sqrt_k", seed=5)
    assert gt.gemm_tn_config_name(gt.gemm_tn_select_config(gt.GEMM_TN_F16, m, n, k)) == "1cta_n128_splitk"
    c_split, st1 = gpu_gemm(a, b)
    c_whole, st2 = gpu_gemm(a, b, "1cta_n128")
    assert st1 == 0 and st2 == 0
    assert_parity(c_split, a, b, "split-K default")
    assert_parity(c_whole, a, b, "whole tiles")


def test_launch_counter():
    """gemm_tn_launch_count counts this library's kernel launches: one for an
    aligned GEMM without a cut tail, one more for a repack of misaligned
    operands, one per attention pass, none for the K = 0 memset."""
    dev = torch.device("cuda", 0)
    a, b = (t.to(dev) for t in make_operands(512, 512, 512, "fp16", "uniform", seed=3))
    n0 = gt.gemm_tn_launch_count()
    gt.mm_tn(a, b)
    assert gt.gemm_tn_launch_count() - n0 == 1
    ar, br = (t.to(dev) for t in make_operands(300, 200, 100, "fp16", "uniform", seed=4))   # K = 100: repack
    n0 = gt.gemm_tn_launch_count()
    gt.mm_tn(ar, br)
    assert gt.gemm_tn_launch_count() - n0 == 2
    az, bz = torch.empty((64, 0), dtype=torch.float16, device=dev), torch.empty((32, 0), dtype=torch.float16, device=dev)
    n0 = gt.gemm_tn_launch_count()
    gt.mm_tn(az, bz)
    assert gt.gemm_tn_launch_count() - n0 == 0
    torch.cuda.synchronize()


def test_stream_k_is_deterministic():
    m, n, k = 300, 1000, 3000
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "uniform", seed=99)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    outs = []
    for _ in range(5):
        out = torch.full((m, n), float("nan"), dtype=torch.float16, device=dev)
        gt.mm_tn(a, b, out=out)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


# ------------------------------------------------------------ streams, threads, graphs

def test_cuda_graph_capture_and_replay():
    """The default path (TMA-aligned operands) issues only stream-ordered work,
    so a call can be captured into a CUDA graph and replayed; after a warm-up
    call has filled the per-device caches."""
    m, n, k = 1024, 1536, 2048
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=21)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        gt.mm_tn(a, b, out=out)            # warm-up: attribute and occupancy caches
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gt.mm_tn(a, b, out=out)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert_parity(out.cpu(), a_cpu, b_cpu, "graph replay")
    # new operand values in the same buffers are picked up by the replay
    a.copy_(b_cpu[:m].to(dev) if n >= m else a)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert_parity(out.cpu(), a.cpu(), b_cpu, "graph replay after operand update")


@pytest.mark.parametrize("mnk", [(128, 4096, 4096), (8, 4096, 4096), (256, 256, 256), (2048, 2048, 2048),
                                 (2304, 4352, 1000), (1000, 1003, 1001)],
                         ids=["splitk", "decode", "one_round_128", "one_round_128x256", "stream_k", "repack"])
def test_cuda_graph_chain_of_each_kernel_kind(mnk):
    """Three dependent calls of one kernel kind (cluster split-K, decode,
    single-CTA tiles, a stream-K tail, misaligned operands that are copied
    first) captured into a CUDA graph, where their programmatic dependent
    launches become graph edges and their workspaces (stream-K partials,
    padded copies) allocations of the graph: C1 = A B^T, C2 = C1' ...,
    replayed twice with the intermediate pre-filled with NaN; the results
    equal the ones computed call by call with synchronisations."""
    m, n, k = mnk
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "normal_over_sqrt_k", seed=m + n)
    a, b = a_cpu.to(dev), b_cpu.to(dev)
    w = torch.randn(n, n, device=dev).to(torch.bfloat16) / n ** 0.5     # second GEMM: C2 = C1 W^T
    c1 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    c2 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    gt.mm_tn(a, b, out=c1)
    torch.cuda.synchronize()
    gt.mm_tn(c1, w, out=c2)
    torch.cuda.synchronize()
    expected = c2.clone()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c1.fill_(float("nan"))
        gt.mm_tn(a, b, out=c1)
        gt.mm_tn(c1, w, out=c2)
    for _ in range(2):
        c2.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(c2, expected), f"{mnk}: graph replay differs"


def test_concurrent_calls_from_two_threads_on_two_streams():
    import threading
    dev = torch.device("cuda", 0)
    shapes = [(700, 900, 1100), (513, 1030, 777)]
    data = [make_operands(m, n, k, "fp16", "uniform", seed=i) for i, (m, n, k) in enumerate(shapes)]
    results = [None, None]
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(dev)
            a, b = data[i][0].to(dev), data[i][1].to(dev)
            with torch.cuda.stream(s):
                outs = [gt.mm_tn(a, b) for _ in range(10)]
            s.synchronize()
            results[i] = [o.cpu() for o in outs]
        except Exception as exc:  # pragma: no cover - reported below
            errors.append(exc)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        for o in results[i][1:]:
            assert torch.equal(o, results[i][0])
        assert_parity(results[i][0], data[i][0], data[i][1], f"thread {i}")


def test_host_entry_point_chunked_with_ragged_pitches():
    """gemm_tn_host on a problem it splits into several row chunks, with K and
    N whose host row pitches are not multiples of 16 bytes (the device staging
    rows are padded by 2-D copies); pinned and pageable buffers."""
    m, n, k = 5000, 1003, 4097
    a_cpu, b_cpu = make_operands(m, n, k, "fp16", "normal_over_sqrt_k", seed=77)
    c_pinned = gt.mm_tn_host(a_cpu.pin_memory(), b_cpu.pin_memory())
    c_pageable = gt.mm_tn_host(a_cpu, b_cpu)
    assert torch.equal(c_pinned, c_pageable)
    rng = np.random.Generator(np.random.PCG64(5))
    rows = edge_indices(m, 2560, rng, 24)
    cols = edge_indices(n, 256, rng, 24)
    assert_sampled_parity(c_pinned, a_cpu, b_cpu, rows, cols, "host path")


def test_host_entry_point_large_ragged():
    """gemm_tn_host on a larger bf16 problem that it copies in two row chunks
    of A and C (the last one ragged), with a padded K (2049) and B of 37 MB;
    pinned and pageable buffers."""
    m, n, k = 9000, 9000, 2049
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "normal_over_sqrt_k", seed=78)
    c_pinned = gt.mm_tn_host(a_cpu.pin_memory(), b_cpu.pin_memory())
    c_pageable = gt.mm_tn_host(a_cpu, b_cpu)
    assert torch.equal(c_pinned, c_pageable)
    rng = np.random.Generator(np.random.PCG64(6))
    rows = edge_indices(m, 4608, rng, 24)
    cols = edge_indices(n, 4608, rng, 24)
    assert_sampled_parity(c_pinned, a_cpu, b_cpu, rows, cols, "host path, large ragged")


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("mnk", [(1000, 1000, 640), (2304, 4352, 1000), (3001, 5003, 577), (4096, 4096, 512),
                                 (300, 2000, 700)], ids=lambda s: "x".join(map(str, s)))
def test_tail_split_sub_tiles(mnk, config):
    """The last, partial wave of tiles is cut into 2 or 4 sub-tiles along N
    (runtime MMA N, narrower B boxes); parity with the cut on and off."""
    from _parity import env_var
    m, n, k = mnk
    a, b = make_operands(m, n, k, "bf16", "uniform", seed=m + 3 * n + 7 * k)
    for on in (None, "0"):
        with env_var("GEMM_TN_TAIL_SPLIT", on):
            c, status = gpu_gemm(a, b, config)
        assert status == 0
        assert_parity(c, a, b, f"{mnk} {config} tail_split={'off' if on else 'on'}")



# ------------------------------------------------------------ B stored [K, N] (gemm_nn)

def _nn_parity(m, n, k, dtype, config, seed, ldb_pad=0, epilogue="auto"):
    import oracle
    from _parity import env_var
    dev = torch.device("cuda", 0)
    a_cpu, bt_cpu = make_operands(m, n, k, dtype, "uniform", seed=seed)   # bt: [N, K]
    b_cpu = bt_cpu.T.contiguous()                                          # [K, N]
    b_big = torch.zeros((k, n + ldb_pad), dtype=b_cpu.dtype)
    b_big[:, :n] = b_cpu
    b = b_big.to(dev)[:, :n]
    c = torch.full((m, n), float("nan"), dtype=a_cpu.dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with forced_config(config), epilogue_mode(epilogue):
        gt.mm_nn(a_cpu.to(dev), b, out=c, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, bound = oracle.gemm_nn_reference(a_cpu, b_cpu)
    rep = oracle.parity_report(c.cpu(), ref, bound)
    assert rep.ok, f"nn {m}x{n}x{k} {dtype} {config}: {rep}"


@pytest.mark.parametrize("config", CONFIGS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("mnk", [(1, 1, 1), (7, 13, 17), (128, 256, 64), (129, 257, 65), (300, 200, 1000),
                                 (513, 640, 200), (1000, 1000, 64), (2304, 4352, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
def test_nn_parity(mnk, dtype, config):
    _nn_parity(*mnk, dtype, config, seed=sum(mnk))


@pytest.mark.parametrize("ldb_pad", [3, 8])
def test_nn_padded_and_misaligned_b(ldb_pad):
    _nn_parity(300, 333, 200, "fp16", None, seed=ldb_pad, ldb_pad=ldb_pad)


@pytest.mark.parametrize("config", CONFIGS)
def test_nn_small_integers_are_exact(config):
    m, n, k = 300, 400, 64
    a, bt = make_operands(m, n, k, "bf16", "int_small", seed=78)
    b = bt.T.contiguous()
    dev = torch.device("cuda", 0)
    with forced_config(config):
        c = gt.mm_nn(a.to(dev), b.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(c.cpu().double(), (a.long() @ b.long()).double())


def test_nn_headline_full_parity(headline_reference):
    """bf16 8192^3 with B stored [K, N] (the headline's B transposed, so the
    product is the headline's): every output element against the oracle."""
    import oracle
    w, a_cpu, bt_cpu, ref, bound = headline_reference
    b_cpu = bt_cpu.T.contiguous()
    dev = torch.device("cuda", 0)
    c = torch.full((w.m, w.n), float("nan"), dtype=a_cpu.dtype, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gt.mm_nn(a_cpu.to(dev), b_cpu.to(dev), out=c, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rep = oracle.parity_report(c.cpu(), ref, bound)
    assert rep.ok, f"nn headline: {rep}"



# ------------------------------------------------------------ fused epilogue (gemm_tn_fused)

def _fused_case(m, n, k, dtype, activation, out_fp32, alpha, beta, with_bias, seed, ldc_pad=0):
    import oracle
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, dtype, "uniform", seed=seed)
    g = torch.Generator().manual_seed(seed)
    bias = (torch.rand(n, generator=g) * 4 - 2).float() if with_bias else None
    out_dtype = torch.float32 if out_fp32 else a_cpu.dtype
    c_in = (torch.rand((m, n), generator=g) * 2 - 1).to(out_dtype)
    c_big = torch.full((m, n + ldc_pad), float("nan"), dtype=out_dtype)
    c_big[:, :n] = c_in
    c_big = c_big.to(dev)
    c = c_big[:, :n]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gt.mm_tn_fused(a_cpu.to(dev), b_cpu.to(dev), out=c, alpha=alpha, beta=beta,
                   bias=bias.to(dev) if bias is not None else None, activation=activation, out_fp32=out_fp32,
                   status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    act = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu": oracle.ACT_GELU}[activation]
    d_ref, pre_bound = oracle.fused_reference(a_cpu, b_cpu, alpha, beta, c_in, bias, act)
    rep = oracle.fused_parity_report(c.cpu(), d_ref, pre_bound, act)
    assert rep.ok, f"fused {m}x{n}x{k} {dtype} {activation} f32={out_fp32} a={alpha} b={beta}: {rep}"
    if ldc_pad:
        assert torch.isnan(c_big[:, n:].float()).all(), "wrote outside C"


@pytest.mark.parametrize("activation", ["none", "relu", "gelu"])
@pytest.mark.parametrize("out_fp32", [False, True])
@pytest.mark.parametrize("mnk", [(129, 257, 65), (300, 1000, 640), (64, 640, 512), (1000, 1003, 200)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_epilogue_parity(mnk, activation, out_fp32):
    m, n, k = mnk
    _fused_case(m, n, k, "bf16", activation, out_fp32, alpha=0.75, beta=0.5, with_bias=True, seed=m + n + k)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("beta,with_bias", [(0.0, False), (1.0, False), (0.0, True)])
def test_fused_epilogue_terms(dtype, beta, with_bias):
    _fused_case(777, 900, 333, dtype, "relu", False, alpha=1.5, beta=beta, with_bias=with_bias, seed=9, ldc_pad=5)


@pytest.mark.parametrize("out_fp32", [False, True])
def test_fused_epilogue_k_zero(out_fp32):
    _fused_case(100, 70, 0, "fp16", "gelu", out_fp32, alpha=2.0, beta=0.5, with_bias=True, seed=3)


def _fused_e4m3_case(m, n, k, dtype, activation, alpha, beta, with_bias, seed, ldc_pad=0):
    """gemm_tn_fused with the fp8 e4m3 output, against the oracle's fp64 D and
    the e4m3 criterion (rounding and saturation carried through)."""
    import oracle
    from oracle import fp8
    dev = torch.device("cuda", 0)
    a_cpu, b_cpu = make_operands(m, n, k, dtype, "uniform", seed=seed)
    g = torch.Generator().manual_seed(seed)
    bias = (torch.rand(n, generator=g) * 8 - 4).float() if with_bias else None
    # C's previous contents: random finite e4m3 codes; the padding holds NaN (0x7F)
    codes_in = torch.randint(0, 256, (m, n), generator=g, dtype=torch.int32).to(torch.uint8)
    codes_in[(codes_in & 0x7F) == 0x7F] = 0x3A
    c_big = torch.full((m, n + ldc_pad), 0x7F, dtype=torch.uint8)
    c_big[:, :n] = codes_in
    c_big = c_big.to(dev).view(torch.float8_e4m3fn)
    c = c_big[:, :n]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gt.mm_tn_fused(a_cpu.to(dev), b_cpu.to(dev), out=c, alpha=alpha, beta=beta,
                   bias=bias.to(dev) if bias is not None else None, activation=activation,
                   out_dtype=torch.float8_e4m3fn, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    act = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu": oracle.ACT_GELU}[activation]
    d_ref, pre_bound = oracle.fused_reference(a_cpu, b_cpu, alpha, beta, fp8.e4m3_decode(codes_in), bias, act)
    rep = oracle.fused_e4m3_parity_report(c.cpu(), d_ref, pre_bound, act)
    assert rep.ok, f"fused e4m3 {m}x{n}x{k} {dtype} {activation} a={alpha} b={beta}: {rep}"
    if ldc_pad:
        assert (c_big[:, n:].cpu().view(torch.uint8) == 0x7F).all(), "wrote outside C"


@pytest.mark.parametrize("activation", ["none", "gelu"])
@pytest.mark.parametrize("mnk,ldc_pad", [((129, 257, 65), 3), ((64, 640, 512), 0), ((1000, 1003, 200), 0),
                                         ((300, 1024, 640), 0), ((77, 333, 128), 5)],
                         ids=lambda s: "x".join(map(str, s)) if isinstance(s, tuple) else f"pad{s}")
def test_fused_e4m3_parity(mnk, ldc_pad, activation):
    m, n, k = mnk
    # alpha as the quantisation scale: |D| reaches the top binades of e4m3
    _fused_e4m3_case(m, n, k, "bf16", activation, alpha=8.0, beta=0.25, with_bias=True, seed=m * n + k,
                     ldc_pad=ldc_pad)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fused_e4m3_saturates(dtype):
    """alpha far above the range: most outputs clamp to +-448 exactly."""
    _fused_e4m3_case(260, 300, 256, dtype, "none", alpha=500.0, beta=0.0, with_bias=False, seed=4)


def test_fused_e4m3_k_zero():
    _fused_e4m3_case(100, 70, 0, "fp16", "relu", alpha=2.0, beta=0.5, with_bias=True, seed=3)


@pytest.mark.parametrize("m", [100, 300])
def test_fused_e4m3_exact_integers(m):
    """Entries in {-1, 0, 1} and K = 16: every product sum is an integer in
    [-16, 16], and times alpha = 16 still exact in e4m3 (at most 3 mantissa
    bits), so the stored codes equal the oracle's encoding bit for bit (zero's
    sign aside: +0 and -0 are the same value)."""
    import oracle
    from oracle import fp8
    dev = torch.device("cuda", 0)
    n, k = 520, 16
    g = torch.Generator().manual_seed(m)
    a_cpu = torch.randint(-1, 2, (m, k), generator=g).to(torch.bfloat16)
    b_cpu = torch.randint(-1, 2, (n, k), generator=g).to(torch.bfloat16)
    c = gt.mm_tn_fused(a_cpu.to(dev), b_cpu.to(dev), alpha=16.0, out_dtype=torch.float8_e4m3fn)
    torch.cuda.synchronize()
    d_ref, _ = oracle.fused_reference(a_cpu, b_cpu, alpha=16.0)
    want = fp8.e4m3_encode(d_ref)
    got = c.cpu().view(torch.uint8).numpy()
    zero_sign = np.uint8(0x80)
    assert np.array_equal(np.where(got == zero_sign, 0, got), np.where(want == zero_sign, 0, want))


def test_fused_headline_full_parity(headline_reference):
    """bf16 8192^3 with bias + GELU and fp32 output: every output element
    against the oracle's epilogue applied to the headline product."""
    import oracle
    w, a_cpu, b_cpu, ref, bound = headline_reference
    dev = torch.device("cuda", 0)
    bias = torch.linspace(-1, 1, w.n, dtype=torch.float32)
    c = gt.mm_tn_fused(a_cpu.to(dev), b_cpu.to(dev), bias=bias.to(dev), activation="gelu", out_fp32=True).cpu()
    d_ref, pb = oracle.fused_reference(a_cpu, b_cpu, bias=bias, activation=oracle.ACT_GELU, product=(ref, bound))
    rep = oracle.fused_parity_report(c, d_ref, pb, oracle.ACT_GELU)
    assert rep.ok, rep


def test_workspace_pool_keeps_memory_between_calls():
    """A call with a stream-K tail takes its fp32 partials from the library's
    workspace pool. After a synchronisation the pool still holds that memory
    (the next call reuses it without mapping memory again), trimming returns
    it, and a call after the trim is still correct."""
    import ctypes
    m, n, k = 2304, 4352, 1000
    a_cpu, b_cpu = make_operands(m, n, k, "bf16", "uniform", seed=23)
    cuda = ctypes.CDLL("libcuda.so.1")
    pool = ctypes.c_void_p(gt.gemm_tn_workspace_pool())
    assert pool.value

    def attr(code):   # CU_MEMPOOL_ATTR_RESERVED_MEM_CURRENT = 5, USED_MEM_HIGH = 8
        v = ctypes.c_uint64()
        assert cuda.cuMemPoolGetAttribute(pool, code, ctypes.byref(v)) == 0
        return v.value

    zero = ctypes.c_uint64(0)
    assert cuda.cuMemPoolSetAttribute(pool, 8, ctypes.byref(zero)) == 0
    c, status = gpu_gemm(a_cpu, b_cpu)
    assert status == 0
    assert attr(8) > 0, "the stream-K tail took no workspace"
    assert attr(5) > 0, "the pool gave its memory back at the synchronisation"
    assert_parity(c, a_cpu, b_cpu, "stream-K tail from the pool")
    assert gt.gemm_tn_trim_workspace() == gt.GEMM_TN_OK
    assert attr(5) == 0
    c2, status = gpu_gemm(a_cpu, b_cpu)
    assert status == 0 and torch.equal(c, c2)


def test_fused_gelu_accuracy_on_a_grid():
    """The epilogue's GELU, x * Phi(x) with erf from Abramowitz and Stegun
    7.1.26 (absolute error <= 1.5e-7), evaluated through the K = 0 fused call
    (D = act(beta * C)) on a grid of x in [-12, 12] and the fp32 extremes of
    its range, against the oracle's fp64 GELU: |d - gelu(x)| <= 1e-6 * |x|
    (erf's bound plus the fp32 reciprocal and exponential)."""
    import oracle
    dev = torch.device("cuda", 0)
    grid = np.concatenate([np.linspace(-12.0, 12.0, 48001), [0.0, -0.0, 1e-30, -1e-30, 1e-5, -1e-5, 40.0, -40.0]])
    x = torch.tensor(grid, dtype=torch.float32).reshape(1, -1)
    n = x.shape[1]
    c = x.to(dev).clone()
    empty = torch.empty((1, 0), dtype=torch.bfloat16, device=dev)
    b = torch.empty((n, 0), dtype=torch.bfloat16, device=dev)
    gt.mm_tn_fused(empty, b, out=c, alpha=1.0, beta=1.0, activation="gelu", out_dtype=torch.float32)
    torch.cuda.synchronize()
    want, _ = oracle.fused_reference(np.zeros((1, 0)), np.zeros((n, 0)), beta=1.0, c_in=x.double().numpy(),
                                     activation=oracle.ACT_GELU)
    got = c.cpu().double().numpy()
    xd = x.double().numpy()
    err = np.abs(got - want)
    assert np.isfinite(got).all()
    assert (err <= 1e-6 * np.abs(xd)).all(), f"max err/|x| {np.max(err / np.maximum(np.abs(xd), 1e-300)):.3e}"
