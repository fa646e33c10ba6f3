"""Pins for the fp64 attention oracle, against things other than itself.

The oracle computes, per batch and head, O = softmax(scale * Q K^T, causal
mask) V on [batch, seq, heads, dim] arrays ("TileLang: a tile language one level
below Triton", section "FlashAttention: online softmax as tile code"). Its pins:

* closed forms: zero queries weight every visible key equally, so each output
  row is the mean of the visible value rows (a cumulative sum under the causal
  mask); constant values come back unchanged (the weights sum to one); a single
  key returns its value row; one-hot queries and keys give scores that are zero
  except on one key per query, so the output has a two-term closed form in
  exp(scale * beta);
* a library routine: torch's scaled_dot_product_attention in fp64 on the CPU
  (an independent implementation of the same definition, causal and not);
* the section's own algorithm: the online softmax walked tile by tile (running
  maximum, rescaled accumulator and row sum, exp2 with log2(e) folded into the
  scale, the causal loop bound and the in-tile mask) in fp64 numpy reaches the
  same values;
* planted mistakes: deliberately wrong builds of the C loop (strict causal mask,
  scale ignored, no normalisation, Q and K exchanged, V read from head 0) each
  fail at least one of the pins above.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import build as oracle_build


def _normal(shape, seed, dtype=None):
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal(size=shape).astype(np.float32)
    if dtype is None:
        return x.astype(np.float64)
    return torch.from_numpy(x).to(dtype).to(torch.float64).numpy()


def _visible(i: int, seq: int, causal: bool) -> int:
    return i + 1 if causal else seq


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 1, 1, 8), (2, 9, 3, 16), (1, 70, 2, 64), (2, 131, 1, 128)])
def test_zero_queries_average_the_visible_values(shape, causal):
    B, S, H, D = shape
    q = np.zeros(shape)
    k = _normal(shape, 11)
    v = _normal(shape, 12, torch.float16)
    out, bound = oracle.attention_reference(q, k, v, causal=causal)
    if causal:
        counts = np.arange(1, S + 1, dtype=np.float64).reshape(1, S, 1, 1)
        want = np.cumsum(v, axis=1) / counts
        want_bound = np.cumsum(np.abs(v), axis=1) / counts
    else:
        want = np.broadcast_to(v.mean(axis=1, keepdims=True), shape)
        want_bound = np.broadcast_to(np.abs(v).mean(axis=1, keepdims=True), shape)
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(bound, want_bound, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("causal", [True, False])
def test_constant_values_come_back_unchanged(causal):
    B, S, H, D = 2, 45, 3, 32
    q = _normal((B, S, H, D), 21) * 3.0
    k = _normal((B, S, H, D), 22) * 3.0
    c = _normal((1, 1, H, D), 23, torch.bfloat16)   # one constant row per head
    v = np.broadcast_to(c, (B, S, H, D)).copy()
    out, bound = oracle.attention_reference(q, k, v, causal=causal)
    np.testing.assert_allclose(out, v, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(bound, np.abs(v), rtol=1e-14, atol=1e-15)


def test_single_key_returns_its_value_row():
    shape = (3, 1, 2, 64)
    q, k = _normal(shape, 31), _normal(shape, 32)
    v = _normal(shape, 33, torch.float16)
    for causal in (True, False):
        out, _ = oracle.attention_reference(q, k, v, causal=causal)
        assert np.array_equal(out, v)


@pytest.mark.parametrize("causal", [True, False])
def test_one_hot_scores_closed_form(causal):
    # keys are unit vectors e_j, query i is beta * e_t(i): the only non-zero
    # score of row i is scale * beta at key t(i) (t(i) <= i keeps it visible)
    S, D, H, beta = 24, 32, 2, 5.0
    scale = 1.0 / math.sqrt(D)
    g = np.random.Generator(np.random.PCG64(41))
    target = np.array([g.integers(0, i + 1) for i in range(S)])
    k = np.zeros((1, S, H, D))
    q = np.zeros((1, S, H, D))
    for j in range(S):
        k[0, j, :, j] = 1.0
        q[0, j, :, target[j]] = beta
    v = _normal((1, S, H, D), 42, torch.float16)
    out, _ = oracle.attention_reference(q, k, v, causal=causal)
    w = math.exp(scale * beta)
    for i in range(S):
        n = _visible(i, S, causal)
        rest = v[0, :n].sum(axis=0) - v[0, target[i]]
        want = (w * v[0, target[i]] + rest) / (w + n - 1)
        np.testing.assert_allclose(out[0, i], want, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- a library routine

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (2, 63, 3, 64), (1, 129, 4, 128), (3, 200, 2, 16)])
def test_agrees_with_torch_sdpa_in_fp64(shape, causal):
    q = _normal(shape, 51, torch.float16)
    k = _normal(shape, 52, torch.float16)
    v = _normal(shape, 53, torch.float16)
    out, _ = oracle.attention_reference(q, k, v, causal=causal)
    qt, kt, vt = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    lib = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
    np.testing.assert_allclose(out, lib.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-13)


def test_explicit_scale_is_used():
    shape = (1, 40, 2, 64)
    q, k, v = _normal(shape, 61), _normal(shape, 62), _normal(shape, 63)
    out, _ = oracle.attention_reference(q, k, v, causal=True, scale=0.3)
    qt, kt, vt = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    lib = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.3)
    np.testing.assert_allclose(out, lib.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- the section's online algorithm

def _online_softmax_tiles(q, k, v, causal, block_m=64, block_n=64):
    """The tile walk of the FlashAttention section in fp64: per query tile, the
    running row maximum and row sum, the accumulator rescaled by exp2 of the
    change of maximum, probabilities exp2(score * scale * log2 e - max), one
    division by the row sum at the end. Keys past the end of the sequence (a
    ragged last tile) are masked like the causal ones."""
    B, S, H, D = q.shape
    c = (1.0 / math.sqrt(D)) * math.log2(math.e)
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            for q0 in range(0, S, block_m):
                qi = q[b, q0:q0 + block_m, h]                     # [bm, D]
                rows = np.arange(q0, q0 + qi.shape[0])
                acc = np.zeros((qi.shape[0], D))
                row_max = np.full(qi.shape[0], -np.inf)
                row_sum = np.zeros(qi.shape[0])
                n_tiles = -(-min(S, q0 + block_m) // block_n) if causal else -(-S // block_n)
                for t in range(n_tiles):
                    kj = k[b, t * block_n:(t + 1) * block_n, h]
                    vj = v[b, t * block_n:(t + 1) * block_n, h]
                    cols = np.arange(t * block_n, t * block_n + kj.shape[0])
                    s = (qi @ kj.T) * c
                    keep = np.ones_like(s, dtype=bool) if not causal else rows[:, None] >= cols[None, :]
                    s = np.where(keep, s, -np.inf)
                    prev = row_max
                    row_max = np.maximum(prev, s.max(axis=1))
                    rescale = np.exp2(prev - row_max)
                    p = np.exp2(s - row_max[:, None])
                    acc = acc * rescale[:, None] + p @ vj
                    row_sum = row_sum * rescale + p.sum(axis=1)
                out[b, q0:q0 + block_m, h] = acc / row_sum[:, None]
    return out


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 128, 2, 64), (2, 200, 1, 64), (1, 257, 2, 32)])
def test_online_softmax_tile_walk_reaches_the_definition(shape, causal):
    q = _normal(shape, 71, torch.float16) * 2.0
    k = _normal(shape, 72, torch.float16)
    v = _normal(shape, 73, torch.float16)
    out, _ = oracle.attention_reference(q, k, v, causal=causal)
    np.testing.assert_allclose(out, _online_softmax_tiles(q, k, v, causal), rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- host logic of the wrapper

def test_row_subset_and_thread_count_do_not_change_values():
    shape = (2, 150, 3, 64)
    q, k, v = _normal(shape, 81), _normal(shape, 82), _normal(shape, 83)
    full, fb = oracle.attention_reference(q, k, v, causal=True, nthreads=1)
    full8, _ = oracle.attention_reference(q, k, v, causal=True, nthreads=8)
    assert np.array_equal(full, full8)
    rows = [149, 0, 63, 64, 127, 128]
    sub, sb = oracle.attention_reference(q, k, v, causal=True, rows=rows)
    assert np.array_equal(sub, full[:, rows])
    assert np.array_equal(sb, fb[:, rows])


def test_empty_shapes_and_bad_rows():
    for shape in [(0, 5, 2, 8), (1, 0, 2, 8), (1, 5, 0, 8), (1, 5, 2, 0)]:
        out, bound = oracle.attention_reference(np.zeros(shape), np.zeros(shape), np.zeros(shape))
        assert out.shape == shape and bound.shape == shape
    with pytest.raises(RuntimeError):
        oracle.attention_reference(np.zeros((1, 4, 1, 8)), np.zeros((1, 4, 1, 8)), np.zeros((1, 4, 1, 8)),
                                   rows=[4])
    with pytest.raises(ValueError):
        oracle.attention_reference(np.zeros((1, 4, 1, 8)), np.zeros((1, 5, 1, 8)), np.zeros((1, 4, 1, 8)))


def test_criterion_accepts_rounded_oracle_and_rejects_a_moved_element():
    shape = (1, 100, 2, 64)
    q, k, v = (_normal(shape, s, torch.bfloat16) for s in (91, 92, 93))
    out, bound = oracle.attention_reference(q, k, v, causal=True)
    rounded = torch.from_numpy(out).to(torch.bfloat16)
    rep = oracle.parity_report(rounded, out, bound)
    assert rep.ok and rep.max_ratio < 0.5, rep
    moved = out.copy()
    moved[0, 37, 1, 5] += 2.0 * (oracle.ALLOW_REL * bound[0, 37, 1, 5] + oracle.ALLOW_ABS)
    assert not oracle.parity_report(moved, out, bound).ok


# ---------------------------------------------------------------- planted mistakes

def _pins_failed(lib) -> list[str]:
    """A compact version of the pins above against a given build; returns the
    names of those that fail."""
    failed = []
    shape = (1, 20, 2, 16)
    v = _normal(shape, 101, torch.float16)
    with np.errstate(all="ignore"):
        out, _ = oracle.attention_reference(np.zeros(shape), _normal(shape, 102), v, causal=True, lib=lib)
        counts = np.arange(1, 21, dtype=np.float64).reshape(1, 20, 1, 1)
        if not np.allclose(out, np.cumsum(v, axis=1) / counts, rtol=1e-12, atol=1e-14):
            failed.append("zero_queries")
        c = np.broadcast_to(_normal((1, 1, 2, 16), 103), shape).copy()
        out, _ = oracle.attention_reference(_normal(shape, 104), _normal(shape, 105), c, causal=False, lib=lib)
        if not np.allclose(out, c, rtol=1e-12, atol=1e-14):
            failed.append("constant_values")
        # one-hot scores: key j = e_j, query i = 4 e_t(i) with t(i) = i // 2
        S1, D1 = 12, 16
        k1 = np.zeros((1, S1, 1, D1))
        q1 = np.zeros((1, S1, 1, D1))
        for j in range(S1):
            k1[0, j, 0, j] = 1.0
            q1[0, j, 0, j // 2] = 4.0
        v1 = _normal((1, S1, 1, D1), 109)
        out, _ = oracle.attention_reference(q1, k1, v1, causal=True, lib=lib)
        w = math.exp(4.0 / math.sqrt(D1))
        want = np.stack([(w * v1[0, i // 2, 0] + v1[0, :i + 1, 0].sum(axis=0) - v1[0, i // 2, 0]) / (w + i)
                         for i in range(S1)])
        if not np.allclose(out[0, :, 0], want, rtol=1e-12, atol=1e-14):
            failed.append("one_hot")
        q, k, vv = (_normal((1, 33, 3, 16), s) for s in (106, 107, 108))
        out, _ = oracle.attention_reference(q, k, vv, causal=True, lib=lib)
        qt, kt, vt = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, vv))
        want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
        if not np.allclose(out, want.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12):
            failed.append("library_sdpa")
    return failed


def test_real_build_passes_compact_pins():
    assert _pins_failed(oracle.load_library()) == []


@pytest.mark.parametrize("plant", [11, 12, 13, 14, 15])
def test_each_planted_mistake_is_caught(plant, tmp_path):
    lib = oracle.load_library(plant=plant, out_dir=tmp_path)
    assert _pins_failed(lib), f"planted mistake {plant} went unnoticed"
    assert oracle_build.library_path(plant, tmp_path).exists()
