"""Pins for the oracle's sparse MLA decode and number formats (CPU only).

* all 256 e4m3 codes and random bf16 patterns decode as torch's own dtypes do;
* with every token selected, sparse MLA equals dense MLA attention computed in
  float64 by torch (softmax and matmul as library routines), including the MTP
  causal rule (query token t sits at position L - T + t);
* closed forms: q = 0 gives the mean of V and lse = ln n; one valid row gives
  V and lse = s; no valid row gives 0 and -inf;
* the order of the top-K list does not change the result;
* FP8 rows with per-row scales equal dense attention over torch's own
  dequantisation.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

D, NOPE = 576, 512


def test_e4m3_all_codes(oracle_lib):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    got = np.array([oracle_lib.e4m3_to_double(int(c)) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_patterns(oracle_lib):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle_lib.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(ref, got)


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rows_bf16(rng_t, n):
    x = torch.randn((n, D), generator=rng_t).to(torch.bfloat16)
    return x, x.view(torch.uint8).numpy().reshape(n, 2 * D)


def _dense(q, k, L, T, scale):
    """Dense MLA decode over all L positions in float64: q [T][H][576],
    k [L][576]; token t sees positions <= L - T + t."""
    qd, kd = q.double(), k.double()
    s = torch.einsum("thd,jd->thj", qd, kd) * scale
    pos = torch.arange(L)
    for t in range(T):
        s[t, :, pos > L - T + t] = -math.inf
    p = torch.softmax(s, dim=-1)
    out = p @ kd[:, :NOPE]
    lse = torch.logsumexp(s, dim=-1)
    return out, lse


@pytest.mark.parametrize("T,H,L", [(1, 4, 37), (3, 2, 64), (4, 3, 130)])
def test_all_selected_equals_dense(oracle_lib, T, H, L):
    g = torch.Generator().manual_seed(T * 100 + L)
    k, kb = _rows_bf16(g, L)
    q = torch.randn((1, T, H, D), generator=g).to(torch.bfloat16)
    perm = torch.randperm(L, generator=g).numpy().astype(np.int32)
    topk = perm[None]                       # every position, shuffled
    gathered = kb[perm][None]
    resolved = np.arange(L, dtype=np.int32)[None]
    scale = 1 / math.sqrt(D)
    out, lse = oracle_lib.sparse_mla_decode(_bf16_bits(q), gathered, None, resolved, topk,
                                            np.array([L]), scale)
    ref_o, ref_l = _dense(q[0], k, L, T, scale)
    np.testing.assert_allclose(out, ref_o.reshape(-1, NOPE).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l.reshape(-1).numpy(), rtol=1e-12, atol=1e-12)


def test_fp8_rows_equal_dense_on_torch_dequant(oracle_lib):
    g = torch.Generator().manual_seed(9)
    L, T, H = 70, 2, 3
    x = torch.randn((L, D), generator=g)
    s = x.abs().amax(dim=1) / 448.0
    codes = (x / s[:, None]).to(torch.float8_e4m3fn)
    k = codes.to(torch.float64) * s.double()[:, None]
    q = torch.randn((1, T, H, D), generator=g).to(torch.bfloat16)
    topk = np.arange(L, dtype=np.int32)[None]
    out, lse = oracle_lib.sparse_mla_decode(
        _bf16_bits(q), codes.view(torch.uint8).numpy()[None], s.numpy()[None], topk.copy(),
        topk, np.array([L]), 0.05)
    ref_o, ref_l = _dense(q[0], k, L, T, 0.05)
    np.testing.assert_allclose(out, ref_o.reshape(-1, NOPE).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l.reshape(-1).numpy(), rtol=1e-12)


def test_closed_forms(oracle_lib):
    g = torch.Generator().manual_seed(3)
    K = 9
    k, kb = _rows_bf16(g, K)
    topk = np.arange(K, dtype=np.int32)[None]
    resolved = topk.copy()
    # q = 0: uniform weights
    q0 = torch.zeros((1, 1, 2, D), dtype=torch.bfloat16)
    out, lse = oracle_lib.sparse_mla_decode(_bf16_bits(q0), kb[None], None, resolved, topk,
                                            np.array([K]), 0.1)
    np.testing.assert_allclose(out[0], k.double()[:, :NOPE].mean(0).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, [math.log(K)] * 2, rtol=1e-14)
    # one valid row (others unresolved): out = V_j, lse = s_j
    q = torch.randn((1, 1, 1, D), generator=g).to(torch.bfloat16)
    res1 = np.full((1, K), -1, np.int32)
    res1[0, 4] = 4
    out, lse = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb[None], None, res1, topk,
                                            np.array([K]), 0.3)
    np.testing.assert_array_equal(out[0], k[4, :NOPE].double().numpy())
    s4 = 0.3 * float((q[0, 0, 0].double() * k[4].double()).sum())
    assert lse[0] == pytest.approx(s4, rel=1e-13)
    # nothing valid: causal rule excludes every position
    topk_late = np.full((1, K), 1000, np.int32)
    out, lse = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb[None], None, resolved, topk_late,
                                            np.array([K]), 0.3)
    assert not out.any() and lse[0] == -math.inf


def test_list_order_does_not_matter(oracle_lib):
    g = torch.Generator().manual_seed(11)
    K, T, H, L = 40, 2, 2, 64
    _, kb = _rows_bf16(g, K)
    q = torch.randn((1, T, H, D), generator=g).to(torch.bfloat16)
    topk = (torch.randperm(L, generator=g)[:K]).numpy().astype(np.int32)[None]
    resolved = np.arange(K, dtype=np.int32)[None]
    resolved[0, 3] = -1
    a = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb[None], None, resolved, topk,
                                     np.array([L]), 0.07)
    p = np.random.default_rng(2).permutation(K)
    b = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb[p][None], None, resolved[:, p],
                                     topk[:, p], np.array([L]), 0.07)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13)


def test_selected_rows_match_full(oracle_lib):
    g = torch.Generator().manual_seed(4)
    B, T, H, K, L = 2, 2, 3, 16, 40
    kb = np.stack([_rows_bf16(g, K)[1] for _ in range(B)])
    q = torch.randn((B, T, H, D), generator=g).to(torch.bfloat16)
    topk = np.stack([np.random.default_rng(b).permutation(L)[:K] for b in range(B)]).astype(np.int32)
    res = np.tile(np.arange(K, dtype=np.int32), (B, 1))
    full = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb, None, res, topk, np.array([L, L - 3]), 0.1)
    sel = np.array([[1, 1, 2], [0, 0, 0], [1, 0, 1]], np.int32)
    part = oracle_lib.sparse_mla_decode(_bf16_bits(q), kb, None, res, topk, np.array([L, L - 3]),
                                        0.1, sel=sel)
    idx = [(b * T + t) * H + h for b, t, h in sel]
    np.testing.assert_array_equal(part[0], full[0][idx])
    np.testing.assert_array_equal(part[1], full[1][idx])


def test_per_token_layout_equals_shared_list_decode():
    """One list per query token, each attended as a one-token entry whose
    context ends at its position L - T + t, equals the T-token decode when
    every token has the same list (the causal rule of the shared-list form)."""
    import oracle
    rng = np.random.default_rng(9)
    B, T, H, K, L = 2, 4, 3, 40, 300
    q = rng.integers(0, 1 << 16, size=(B, T, H, 576), dtype=np.uint16)
    q = (q & 0x3FFF).astype(np.uint16)  # finite, moderate bf16 values
    rows = rng.standard_normal((B, K, 576)).astype(np.float32)
    gat = rows.view(np.uint32).astype(np.uint64)
    gat = ((gat + 0x7FFF + ((gat >> 16) & 1)) >> 16).astype(np.uint16).view(np.uint8)
    gat = gat.reshape(B, K, 1152)
    topk = np.stack([rng.choice(L, size=K, replace=False) for _ in range(B)]).astype(np.int32)
    topk[:, :3] = [L - 1, L - 2, L - 4]       # positions some tokens cannot see
    res = np.arange(B * K, dtype=np.int32).reshape(B, K)
    res[:, 5] = -1
    o1, l1 = oracle.sparse_mla_decode(q, gat, None, res, topk, np.full(B, L, np.int32), 0.05)
    rep = lambda a: np.repeat(a, T, axis=0)
    L1 = (L - T + 1 + np.tile(np.arange(T), B)).astype(np.int32)
    o2, l2 = oracle.sparse_mla_decode(q.reshape(B * T, 1, H, 576), rep(gat), None, rep(res),
                                      rep(topk), L1, 0.05)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
