"""GPU parity of sparse MLA decode where attention is peaked or the query is
far from unit scale.

Attention over the selected rows ("vLLM Hybrid HiSparse：稀疏MLA破解长上下文显存瓶颈",
section 稀疏MLA的核心思想) is exercised here outside the N(0,1) regime of the
other decode tests, whose logits have a standard deviation near 1 so that the
softmax is almost uniform over 2048 keys. Cases:

  * q scaled by 8 and 32 (logits with a spread of tens; many near-ties among
    the largest scores);
  * a "needle": head h of every query token is c_h times the dequantised
    latent row of one selected key, plus N(0, 0.25) noise, with c_h from
    0.05 to 2 (the needle's logit runs from about 1 to about 50);
  * |q| in the thousands (q x 1024) and tiny q (q x 2^-20, sm_scale x 2^20,
    so the logits are those of the unscaled case).

Each case runs on BF16 and FP8 rows, with rows gathered by the resolve and
read in place, with one KV split and with several, and with one shared list
or one list per query token. Tolerances are the decode tests' own:
  ||out - out_ref||_2 / max(||out_ref||_2, 1e-6) <= 2e-2 (BF16 rows), 5e-2 (FP8),
  |lse - lse_ref| <= 1e-2,
against the float64 oracle on the same seeded inputs. The largest and mean
errors of every case are printed (pytest -s shows them).
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "fp8": 5e-2}
LSE_TOL = 1e-2
NEEDLE_C = (0.05, 0.1, 0.2, 0.35, 0.5, 0.75, 1.0, 2.0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


def _bits(q):
    return q.cpu().view(torch.int16).numpy().view(np.uint16)


def _needle_rows(gw):
    """Per request: a position every query token sees (L - T - 1, inside the
    always-selected tail) and its dequantised latent row, read from the pool
    as the input generator filled it (resident rows never change)."""
    w, lay = gw.w, gw.lay
    pos = w.ctx - w.T - 1
    rows = gw.pool.gpu_rows()
    scales = gw.pool.gpu_scales()
    out = []
    for b in range(w.B):
        blk = int(lay.page_gpu[b, pos // 64])
        assert blk >= 0, "the needle position must be GPU-resident"
        rid = blk * 64 + pos % 64
        r = rows[rid]
        if w.dtype == "bf16":
            k = r.view(torch.bfloat16).float()
        else:
            k = r.view(torch.float8_e4m3fn).float() * scales[rid].float()
        out.append(k)
    return pos, torch.stack(out)  # [B][576] float32 on the device


def _make_q(gw, kind, step):
    """(q bf16 [B][T][H][576] on cuda, sm_scale)"""
    w = gw.w
    base = W.make_q(w, step, device="cuda").float()
    sc = w.sm_scale
    if kind == "x8":
        q = base * 8.0
    elif kind == "x32":
        q = base * 32.0
    elif kind == "x1024":
        q = base * 1024.0
    elif kind == "tiny":
        q = base * 2.0 ** -20
        sc = w.sm_scale * 2.0 ** 20
    elif kind == "needle":
        _, k = _needle_rows(gw)
        c = torch.tensor(NEEDLE_C, device="cuda")[torch.arange(w.H, device="cuda") % len(NEEDLE_C)]
        q = c[None, None, :, None] * k[:, None, None, :] + 0.5 * base
    else:
        raise ValueError(kind)
    return q.to(torch.bfloat16), sc


def _run(w, kind, in_place=False, per_token=False, steps=1, sample_rows=None, nthreads=8):
    import oracle
    from harness import GpuWorkload
    from _mirror import attention_errors, oracle_mirror
    gw = GpuWorkload(w, in_place=in_place, per_token=per_token)
    ot = oracle_mirror(gw)
    B, T, H, K = w.B, w.T, w.H, w.K
    worst, means = (0.0, 0.0), []
    for s in range(steps):
        q, sc = _make_q(gw, kind, s)
        gw.resolve(s)
        gw.decode(s, q, sm_scale=sc)
        torch.cuda.synchronize()
        assert gw.pool.get_error() == 0
        lists = gw.topk_host[s]
        sel = None
        if per_token:
            flat = np.ascontiguousarray(lists.reshape(B, T * K))
            res, gat, gsc, _, err = ot.resolve(np.arange(B), flat, nthreads=nthreads, union=True)
            L1 = (w.ctx - T + 1 + np.tile(np.arange(T), B)).astype(np.int32)
            o_ref, l_ref = oracle.sparse_mla_decode(
                _bits(q).reshape(B * T, 1, H, -1), gat.reshape(B * T, K, -1),
                None if gsc is None else gsc.reshape(B * T, K), res.reshape(B * T, K),
                lists.reshape(B * T, K), L1, sc, nthreads=nthreads)
        else:
            res, gat, gsc, _, err = ot.resolve(np.arange(B), lists, nthreads=nthreads)
            if sample_rows is not None:
                rng = np.random.default_rng(300 + s)
                n = B * T * H
                idx = np.sort(rng.choice(n, size=min(sample_rows, n), replace=False))
                sel = np.stack([idx // (T * H), (idx // H) % T, idx % H], 1).astype(np.int32)
            o_ref, l_ref = oracle.sparse_mla_decode(_bits(q), gat, gsc, res, lists,
                                                    np.full(B, w.ctx, np.int32), sc, sel=sel,
                                                    nthreads=nthreads)
        assert err == 0
        out, lse = gw.out, gw.lse
        if sel is not None:
            out = gw.out[sel[:, 0], sel[:, 1], sel[:, 2]]
            lse = gw.lse[sel[:, 0], sel[:, 1], sel[:, 2]]
        rel, dl = attention_errors(out, lse, o_ref, l_ref)
        print(f"[{w.name} {w.dtype} {kind} in_place={in_place} per_token={per_token} K={K}] "
              f"step {s}: rel max {rel.max():.3e} mean {rel.mean():.3e}; "
              f"lse max {dl.max() if dl.size else 0:.3e}")
        assert np.isfinite(rel).all(), "non-finite output"
        assert rel.max() <= TOL[w.dtype], f"{kind} step {s}: max rel err {rel.max():.3e}"
        assert dl.size == 0 or dl.max() <= LSE_TOL, f"{kind} step {s}: max lse err {dl.max():.3e}"
        worst = (max(worst[0], rel.max()), max(worst[1], dl.max() if dl.size else 0.0))
        means.append(rel.mean())
    gw.pool.close()
    return worst


# Several KV splits (small batches spread one request's 2048 keys over many
# clusters) and one split (K = 128: two key tiles, one split).
SHAPES = {
    "bf16_splits": W.WORKLOADS["resident"].scaled(B=2, ctx=16384, H=64, steps=1),
    "bf16_one_split": W.WORKLOADS["resident"].scaled(B=3, ctx=16384, H=64, K=128, tail=64,
                                                     hot_rows=256, steps=1),
    "fp8_splits": W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=32,
                                               steps=1),
    "fp8_one_split": W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=32,
                                                  K=128, tail=64, hot_rows=256, steps=1),
}
KINDS = ["x8", "x32", "needle", "x1024", "tiny"]


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("in_place", [False, True])
def test_peaked_decode_parity(shape, kind, in_place):
    _run(SHAPES[shape], kind, in_place=in_place)


@pytest.mark.parametrize("kind", ["x32", "needle", "x1024", "tiny"])
@pytest.mark.parametrize("in_place", [False, True])
def test_peaked_decode_per_token_parity(kind, in_place):
    """One top-K list per query token, resolved as a union (FP8, 4 tokens)."""
    _run(SHAPES["fp8_splits"], kind, in_place=in_place, per_token=True)


@pytest.mark.parametrize("kind", ["x32", "needle"])
def test_peaked_decode_full_size_sampled(kind):
    """The fully resident workload at full size (32 requests, 128 heads,
    top-2048; the launch shape the benchmark times), sampled query rows."""
    _run(W.WORKLOADS["resident"], kind, sample_rows=256, nthreads=16)


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("scale", [1.0, 0.125, 3.0])
def test_fp8_codes_decode_exactly(in_place, scale):
    """A list with one valid entry gives out = that entry's value row exactly.
    The entry's row holds every finite e4m3 code (subnormals included, NaN
    codes replaced by 0) with row scale `scale`; each code times the scale is
    a BF16 value (scale 3 = 1.5 x 2 keeps three mantissa bits within BF16's
    eight), so out must equal torch's decoding of the codes exactly. (Values
    are compared, not bits: code 0x80 decodes to -0, and the tensor cores'
    sum of -0 with the +0 products of the other keys is +0.)"""
    from harness import GpuWorkload
    w = SHAPES["fp8_splits"].scaled(B=2, H=16)
    gw = GpuWorkload(w, in_place=in_place)
    pos, _ = _needle_rows(gw)
    codes = torch.arange(576, dtype=torch.int64) % 256
    codes[(codes == 0x7F) | (codes == 0xFF)] = 0
    codes = codes.to(torch.uint8)
    rows, scales = gw.pool.gpu_rows(), gw.pool.gpu_scales()
    lists = torch.full((w.B, w.K), -1, dtype=torch.int32)
    lists[:, 3] = pos
    for b in range(w.B):
        rid = int(gw.lay.page_gpu[b, pos // 64]) * 64 + pos % 64
        rows[rid] = codes.cuda()
        scales[rid] = scale
    torch.cuda.synchronize()
    t = lists.cuda()
    q = W.make_q(w, 0, device="cuda")
    gw.resolve(0, topk=t)
    gw.decode(0, q, topk=t)
    torch.cuda.synchronize()
    assert gw.pool.get_error() == 0
    want = (codes.view(torch.float8_e4m3fn).float() * scale)[:512].to(torch.bfloat16)
    got = gw.out.cpu().float()
    bad = (got != want.float().expand_as(got)).nonzero()
    assert bad.numel() == 0, f"decoded row differs at {bad[:8].tolist()}"
    k = codes.view(torch.float8_e4m3fn).double() * scale
    s_ref = (q.cpu().double() @ k) * w.sm_scale
    assert (gw.lse.cpu().double() - s_ref).abs().max().item() <= LSE_TOL
    gw.pool.close()
