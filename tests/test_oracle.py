"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: torch's own
float8/bfloat16 conversions, textbook values of the OCP E4M3 format, closed
forms of special cases, element-by-element brute force in pure Python on tiny
inputs, torch's scaled_dot_product_attention and scipy's logsumexp, and
invariants (page-table layout, K >= context == dense causal attention).
"""
import math

import numpy as np
import pytest
import torch

import dsa_workloads as W
from oracle import dsa_oracle as O


def small(name="decode_b1", seed=0, **over):
    base = dict(ctx=[200], K=16, H_I=4, D_I=32, H=4, d_latent=64, d_rope=16)
    if name == "decode_b4_long":
        base.update(d_latent=512, d_rope=64)
    base.update(over)
    return W.make(name, seed=seed, **base)


# --------------------------------------------------------------------------- formats

def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_table()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_textbook_values():
    t = O.e4m3_table()
    assert t[0x7E] == 448.0            # largest finite: 1.75 * 2^8
    assert t[0x01] == 2.0 ** -9        # smallest subnormal
    assert t[0x08] == 2.0 ** -6        # smallest normal
    assert t[0x38] == 1.0 and t[0xB8] == -1.0
    assert t[0x00] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0


def test_bf16_decode_matches_torch():
    x = torch.randn(10000, generator=torch.Generator().manual_seed(3)) * 100
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.decode_bf16(bits), ref)


def test_fp8_latent_row_decode():
    """656-byte row: latent = code * scale, rope = bf16 at byte 528."""
    wl = small("decode_b4_long", ctx=[64], B=1, K=8)
    row = wl.kv[5]
    scale = np.frombuffer(row[512:516].tobytes(), "<f4")[0]
    lat = torch.from_numpy(row[:512].copy()).view(torch.float8_e4m3fn).double().numpy() * scale
    rope = torch.from_numpy(row[528:656].copy()).view(torch.bfloat16).double().numpy()
    got = O.latent_rows(wl, np.array([5]))[0]
    assert np.array_equal(got[:512], lat) and np.array_equal(got[512:], rope)


# --------------------------------------------------------------------------- indexer

def brute_scores(wl, t):
    """Element-by-element definition, pure Python, decoding with torch."""
    def deq_q(h, i):
        if wl.idx_dtype == "e4m3":
            v = torch.tensor([wl.q_i[t, h, i]], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
            return v * float(wl.q_i_scale[t, h])
        if wl.idx_dtype == "mx_e4m3":   # block i // 32 carries the E8M0 exponent
            v = torch.tensor([wl.q_i[t, h, i]], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
            return v * 2.0 ** (int(wl.q_i_scale[t, h, i // 32]) - 127)
        return float(wl.q_i[t, h, i])

    def deq_k(row, i):
        if wl.idx_dtype == "e4m3":
            v = torch.tensor([wl.k_i[row, i]], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
            return v * float(wl.k_i_scale[row])
        if wl.idx_dtype == "mx_e4m3":
            v = torch.tensor([wl.k_i[row, i]], dtype=torch.uint8).view(torch.float8_e4m3fn).item()
            return v * 2.0 ** (int(wl.k_i_scale[row, i // 32]) - 127)
        return float(wl.k_i[row, i])

    b = wl.q_seq[t]
    out = []
    qd = [[deq_q(h, i) for i in range(wl.D_I)] for h in range(wl.H_I)]
    for s in range(int(wl.q_pos[t]) + 1):
        row = int(wl.block_table[b, s // wl.page_size]) * wl.page_size + s % wl.page_size
        kd = [deq_k(row, i) for i in range(wl.D_I)]
        acc = 0.0
        for h in range(wl.H_I):
            dot = 0.0
            for i in range(wl.D_I):
                dot += qd[h][i] * kd[i]
            acc += float(wl.w[t, h]) * (dot if dot > 0 else 0.0)
        out.append(acc)
    return np.array(out)


@pytest.mark.parametrize("name", ["tiny_fp32", "decode_b1", "decode_b64", "mx"])
def test_indexer_brute_force(name):
    over = dict(ctx=[70], K=8, H_I=3, D_I=8)
    if name == "decode_b64":
        over = dict(ctx=None, ctx_range=(65, 130), B=2, K=8, H_I=3, D_I=8)
    if name == "mx":   # MXFP8: blocks of 32 with their own power-of-two scales
        name, over = "decode_b64", dict(ctx=None, ctx_range=(40, 70), B=2, K=8, H_I=2, D_I=64,
                                        idx_dtype="mx_e4m3")
    wl = small(name, **over)
    for t in range(wl.T):
        ref = brute_scores(wl, t)
        got = O.indexer_scores_row(wl, t)
        assert got.dtype == np.float32 and got.shape == ref.shape
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())


def test_indexer_one_hot_closed_form():
    """H_I = 1, w = 1, q = e_i: I[s] = max(k_I[s, i] * q_scale, 0)."""
    wl = small(ctx=[130], H_I=1, D_I=32)
    i = 7
    wl.q_i[:] = 0
    wl.q_i[0, 0, i] = 0x38            # e4m3 code of 1.0
    wl.q_i_scale[0, 0] = 0.5
    wl.w[0, 0] = 1.0
    got = O.indexer_scores_row(wl, 0)
    kcode = torch.from_numpy(wl.k_i[:, i].copy()).view(torch.float8_e4m3fn).double().numpy()
    expect = np.maximum(kcode * wl.k_i_scale * 0.5, 0.0)[:130]
    np.testing.assert_allclose(got, expect.astype(np.float32), rtol=0, atol=0)


def test_indexer_zero_weight_negative_dots_and_sign():
    wl = small(ctx=[100])
    t = 0
    base = O.indexer_scores_row(wl, t).astype(np.float64)
    wl2 = small(ctx=[100]); wl2.w[:] = 0
    assert np.all(O.indexer_scores_row(wl2, t) == 0)
    # flipping every key's sign... make all dots negative: q and k of opposite sign
    wl3 = small(ctx=[100]); wl3.idx_dtype = "f32"
    wl3.q_i = np.abs(np.random.default_rng(0).standard_normal((1, wl3.H_I, wl3.D_I))).astype(np.float32)
    wl3.k_i = -np.abs(np.random.default_rng(1).standard_normal((wl3.cache_rows, wl3.D_I))).astype(np.float32)
    wl3.q_i_scale[:] = 1; wl3.k_i_scale[:] = 1
    assert np.all(O.indexer_scores_row(wl3, t) == 0)
    # negating all head weights negates the score (linearity in w)
    wl4 = small(ctx=[100]); wl4.w *= -1
    np.testing.assert_array_equal(O.indexer_scores_row(wl4, t), -base.astype(np.float32))
    # scaling w by 3 scales the score by 3 (within one fp32 rounding)
    wl5 = small(ctx=[100]); wl5.w *= 3
    np.testing.assert_allclose(O.indexer_scores_row(wl5, t), 3 * base, rtol=1e-6, atol=1e-6)


def test_indexer_page_table_invariance():
    """Shuffled physical pages give the same logical scores as contiguous ones."""
    a = small("decode_b64", ctx=None, ctx_range=(150, 400), B=3, K=16)
    b = small("decode_b64", ctx=None, ctx_range=(150, 400), B=3, K=16)
    # rebuild b with an identity page table: move every page to its logical slot
    P = a.page_size
    order = []
    for bb in range(a.B):
        npg = (a.seq_lens[bb] + P - 1) // P
        order += list(a.block_table[bb, :npg])
    rows = np.concatenate([np.arange(p * P, p * P + P) for p in order])
    b.k_i = a.k_i[rows]; b.k_i_scale = a.k_i_scale[rows]; b.kv = a.kv[rows]
    off = 0
    for bb in range(a.B):
        npg = (a.seq_lens[bb] + P - 1) // P
        b.block_table[bb, :npg] = np.arange(off, off + npg)
        off += npg
    assert not np.array_equal(a.block_table, b.block_table)
    np.testing.assert_array_equal(O.indexer_scores(a), O.indexer_scores(b))
    idx = O.topk(O.indexer_scores(a), a.q_pos, a.K)
    oa, la = O.sparse_mla_attn(a, idx)
    ob, lb = O.sparse_mla_attn(b, idx)
    np.testing.assert_array_equal(oa, ob); np.testing.assert_array_equal(la, lb)


def test_indexer_causal_extent():
    wl = small("tiny_fp32")
    s = O.indexer_scores(wl)
    for t in range(wl.T):
        n = wl.q_pos[t] + 1
        assert np.all(np.isfinite(s[t, :n])) and np.all(np.isneginf(s[t, n:]))
    # the query's own position is part of its history
    assert wl.q_pos[-1] + 1 == wl.max_ctx


# --------------------------------------------------------------------------- top-k

def brute_topk(vals, n, K):
    """Repeatedly take the largest remaining value, lowest index first."""
    remaining = list(range(n))
    chosen = []
    for _ in range(min(K, n)):
        best = remaining[0]
        for j in remaining[1:]:
            if vals[j] > vals[best]:
                best = j
        chosen.append(best)
        remaining.remove(best)
    return sorted(chosen)


def as_set(row):
    return sorted(int(x) for x in row if x >= 0)


@pytest.mark.parametrize("seed", range(5))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 120))
    K = int(rng.integers(1, 40))
    vals = rng.integers(-5, 6, size=n).astype(np.float32)   # many ties
    got = O.topk_row(vals, n, K)
    assert as_set(got) == brute_topk(vals, n, K)
    assert np.all(got[min(K, n):] == -1)


def test_topk_special_cases():
    n, K = 50, 10
    assert as_set(O.topk_row(np.zeros(n, np.float32), n, K)) == list(range(K))
    inc = np.arange(n, dtype=np.float32)
    assert as_set(O.topk_row(inc, n, K)) == list(range(n - K, n))
    assert as_set(O.topk_row(inc[::-1].copy(), n, K)) == list(range(K))
    assert as_set(O.topk_row(inc, n, 80)) == list(range(n))
    # ties straddling the K-th value go to the lower indices
    v = np.array([5, 3, 3, 3, 1], np.float32)
    assert as_set(O.topk_row(v, 5, 2)) == [0, 1]
    assert as_set(O.topk_row(v, 5, 3)) == [0, 1, 2]
    # -0.0 and +0.0 are equal values
    z = np.array([1.0, -0.0, 0.0, -1.0], np.float32)
    assert as_set(O.topk_row(z, 4, 2)) == [0, 1]
    # only the causal prefix counts
    big = np.array([0, 0, 0, 9, 9], np.float32)
    assert as_set(O.topk_row(big, 3, 2)) == [0, 1]


# --------------------------------------------------------------------------- attention

def sdpa_dense(wl, t):
    """Dense causal attention of query t with torch's SDPA (float64), MQA form."""
    b = wl.q_seq[t]
    n = int(wl.q_pos[t]) + 1
    rows = np.array([int(wl.block_table[b, s // wl.page_size]) * wl.page_size + s % wl.page_size
                     for s in range(n)])
    if wl.mla_dtype == "bf16":
        kv = torch.from_numpy(wl.kv[rows].view(np.int16)).view(torch.bfloat16).double()
        q = torch.from_numpy(wl.q[t].view(np.int16)).view(torch.bfloat16).double()
    elif wl.mla_dtype == "f32":
        kv = torch.from_numpy(wl.kv[rows]).double(); q = torch.from_numpy(wl.q[t]).double()
    else:
        raw = wl.kv[rows]
        sc = torch.from_numpy(raw[:, 512:516].copy().view("<f4")).double()
        lat = torch.from_numpy(raw[:, :512].copy()).view(torch.float8_e4m3fn).double() * sc
        rope = torch.from_numpy(raw[:, 528:].copy()).view(torch.bfloat16).double()
        kv = torch.cat([lat, rope], 1)
        q = torch.from_numpy(wl.q[t].view(np.int16)).view(torch.bfloat16).double()
    H = wl.H
    qq = q.view(1, H, 1, -1)
    kk = kv.view(1, 1, n, -1).expand(1, H, n, -1)
    vv = kv[:, :wl.d_v].reshape(1, 1, n, -1).expand(1, H, n, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=wl.softmax_scale)
    logits = (q @ kv.T) * wl.softmax_scale
    return out.view(H, -1).numpy(), torch.logsumexp(logits, dim=1).numpy()


@pytest.mark.parametrize("name", ["tiny_fp32", "decode_b1", "decode_b4_long"])
def test_attention_k_ge_ctx_equals_dense(name):
    """Top-K with K >= context selects everything: sparse == dense causal attention."""
    over = dict(ctx=[90], K=128)
    if name == "tiny_fp32":
        over = {}
        wl = W.make(name, K=256)
    else:
        wl = small(name, **over)
    _, idx, out, lse = O.decode_step(wl)
    for t in range(wl.T):
        assert as_set(idx[t]) == list(range(wl.q_pos[t] + 1))
        ro, rl = sdpa_dense(wl, t)
        np.testing.assert_allclose(out[t], ro, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[t], rl, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms():
    from scipy.special import logsumexp
    wl = small(ctx=[128], K=32)
    rows_all = O.latent_rows(wl, np.arange(128))
    q = O.mla_query(wl, 0)
    # one selected row: out = its value part, lse = its logit
    idx = np.full(32, -1, np.int32); idx[0] = 17
    out, lse = O.sparse_mla_attn_row(wl, 0, idx)
    np.testing.assert_array_equal(out, np.broadcast_to(rows_all[17, :wl.d_v], out.shape))
    np.testing.assert_allclose(lse, wl.softmax_scale * q @ rows_all[17], rtol=1e-12)
    # q = 0: uniform weights -> mean of the selected value rows, lse = log m
    sel = np.array([3, 9, 10, 64, 100], np.int32)
    idx = np.full(32, -1, np.int32); idx[:5] = sel
    wl0 = small(ctx=[128], K=32); wl0.q[:] = 0
    out, lse = O.sparse_mla_attn_row(wl0, 0, idx)
    np.testing.assert_allclose(out, np.broadcast_to(rows_all[sel, :wl.d_v].mean(0), out.shape), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(5))
    # lse against scipy's logsumexp; -1 entries anywhere are skipped
    idx = np.array([5, -1, 40, 7, -1, 90] + [-1] * 26, np.int32)
    out, lse = O.sparse_mla_attn_row(wl, 0, idx)
    logits = wl.softmax_scale * q @ rows_all[[5, 40, 7, 90]].T
    np.testing.assert_allclose(lse, logsumexp(logits, axis=1), rtol=1e-12)
    out2, _ = O.sparse_mla_attn_row(wl, 0, np.array([5, 40, 7, 90], np.int32))
    np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-15)
    # softmax weights sum to 1: out of all-equal value rows equals that row
    wl1 = small(ctx=[128], K=32); wl1.idx_dtype = wl.idx_dtype
    wl1.kv[:, :wl.d_v] = wl1.kv[0, :wl.d_v]
    out, _ = O.sparse_mla_attn_row(wl1, 0, np.arange(32, dtype=np.int32))
    np.testing.assert_allclose(out, np.broadcast_to(O.latent_rows(wl1, [0])[0, :wl.d_v], out.shape), rtol=1e-12)
    # empty selection
    out, lse = O.sparse_mla_attn_row(wl, 0, np.full(32, -1, np.int32))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_decode_step_composition_and_order():
    wl = small("decode_b64", ctx=None, ctx_range=(100, 300), B=3, K=40)
    scores, idx, out, lse = O.decode_step(wl)
    for t in range(wl.T):
        n = wl.q_pos[t] + 1
        s = idx[t][idx[t] >= 0]
        assert len(s) == min(40, n) and np.all(np.diff(s) > 0)
        kth = np.sort(scores[t, :n])[::-1][min(40, n) - 1]
        assert np.all(scores[t, s] >= kth)
    # the subset of queries path equals the full path
    s2, i2, o2, l2 = O.decode_step(wl, ts=[2, 0])
    np.testing.assert_array_equal(i2, idx[[2, 0]])
    np.testing.assert_array_equal(o2, out[[2, 0]])


def test_workload_recipes_small():
    """Shapes and storage of each named recipe (scaled down)."""
    wl = W.make("tiny_fp32")
    assert (wl.T, wl.K, wl.H_I, wl.D_I, wl.H, wl.d_qk, wl.d_v) == (8, 32, 4, 32, 4, 80, 64)
    assert list(wl.q_pos) == list(range(248, 256))
    wl = small("decode_b64", ctx=None, ctx_range=(2048, 2100), B=5, K=16)
    assert np.all((wl.seq_lens >= 2048) & (wl.seq_lens <= 2100))
    used = np.sort(wl.block_table[wl.block_table >= 0])
    assert np.array_equal(used, np.arange(wl.cache_rows // 64))
    wl = small("decode_b4_long", ctx=[100, 64], B=2, K=8)
    assert wl.kv.shape == (wl.cache_rows, 656) and wl.row_bytes == 656
    assert np.all(wl.kv[:, 516:528] == 0)


def test_hand_worked_golden_example():
    from tests.fixtures import hand_example
    wl, exp = hand_example()
    scores, idx, out, lse = O.decode_step(wl)
    np.testing.assert_array_equal(scores[0], np.array(exp["scores"], np.float32))
    assert as_set(idx[0]) == exp["topk_set"]
    # ln 3 is stored as an fp32 cache value (relative rounding <= 2^-24), so the
    # closed form holds to ~1e-7 relative
    np.testing.assert_allclose(out[0, 0], exp["out"], rtol=1e-7)
    np.testing.assert_allclose(lse[0, 0], exp["lse"], rtol=1e-7)


# --------------------------------------------------------------------------- cache writers (step 0)

def test_e4m3_encode_matches_torch_cast_within_range():
    """torch's float8_e4m3fn cast (a library routine: round to nearest, ties to
    even) agrees with the encoder wherever it does not overflow (|x| <= 464),
    including every tie between adjacent codes, subnormals and signed zero."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    vals = O.e4m3_table()[:127]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)     # exact ties
    x = np.concatenate([rng.uniform(-464, 464, 50000).astype(np.float32),
                        rng.normal(0, 0.01, 5000).astype(np.float32), vals.astype(np.float32),
                        mids, -mids, np.array([0.0, -0.0, 464.0, -464.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_e4m3_encode_round_trip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = O.decode_e4m3(codes).astype(np.float32)
    got = O.e4m3_encode(vals)
    assert np.array_equal(O.decode_e4m3(got), vals.astype(np.float64))   # +-0 both decode to 0
    sat = O.e4m3_encode(np.array([465.0, 500.0, 1e30, -465.0, -1e30], np.float32))
    assert sat.tolist() == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]                # +-448, never NaN


def test_quantize_row_rule():
    rng = np.random.default_rng(22)
    x = rng.normal(0, 3, 128).astype(np.float32)
    codes, scale = O.quantize_e4m3_row(x)
    amax = np.float32(np.abs(x).max())
    assert scale == np.float32(amax / np.float32(448.0))
    k = int(np.argmax(np.abs(x)))
    assert O.decode_e4m3(codes[k:k + 1])[0] == np.sign(x[k]) * 448.0       # the largest element maps to +-448
    deq = O.decode_e4m3(codes) * np.float64(scale)
    # nearest-value rounding: within half a step of E4M3 (2**-4 relative for normals,
    # 2**-10 * scale absolute in the subnormal range)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(scale)) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)
    zc, zs = O.quantize_e4m3_row(np.zeros(64, np.float32))
    assert zs == np.float32(1.0) and not zc.any()


def test_cache_append_oracle_layout_and_untouched_rows():
    """Rows other than the targets keep their bytes; the FP8 row holds codes,
    the float32 scale (little endian), 12 zero bytes and the rope bits."""
    rng = np.random.default_rng(23)
    page, pages = 64, 6
    block_table = np.array([[4, 1, 5], [0, 3, 2]], dtype=np.int32)
    q_seq = np.array([0, 1, 1], dtype=np.int32)
    q_pos = np.array([130, 5, 64], dtype=np.int32)
    rows = [5 * 64 + 2, 0 * 64 + 5, 3 * 64 + 0]
    k_new = rng.normal(0, 1, (3, 128)).astype(np.float32)
    kc0 = rng.integers(0, 256, (pages * page, 128)).astype(np.uint8)
    ks0 = rng.normal(0, 1, pages * page).astype(np.float32)
    kc, ks = O.index_cache_append(block_table, page, q_seq, q_pos, k_new, kc0, ks0)
    other = np.setdiff1d(np.arange(pages * page), rows)
    assert np.array_equal(kc[other], kc0[other]) and np.array_equal(ks[other], ks0[other])
    for t, r in enumerate(rows):
        codes, scale = O.quantize_e4m3_row(k_new[t])
        assert np.array_equal(kc[r], codes) and ks[r] == scale
    bits = (rng.normal(0, 1, (3, 576)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cache0 = rng.integers(0, 256, (pages * page, 656)).astype(np.uint8)
    cache = O.latent_cache_append(block_table, page, q_seq, q_pos, bits, cache0, fp8_rows=True)
    assert np.array_equal(cache[other], cache0[other])
    for t, r in enumerate(rows):
        codes, scale = O.quantize_e4m3_row(O.decode_bf16(bits[t, :512]).astype(np.float32))
        assert np.array_equal(cache[r, :512], codes)
        assert cache[r, 512:516].view("<f4")[0] == scale
        assert not cache[r, 516:528].any()
        assert np.array_equal(cache[r, 528:656].view("<u2"), bits[t, 512:])
    cacheb0 = rng.integers(0, 256, (pages * page, 1152)).astype(np.uint8)
    cacheb = O.latent_cache_append(block_table, page, q_seq, q_pos, bits, cacheb0, fp8_rows=False)
    assert np.array_equal(cacheb[other], cacheb0[other])
    assert all(np.array_equal(cacheb[r].view("<u2"), bits[t]) for t, r in enumerate(rows))


# --------------------------------------------------------------------------- MXFP8 (OCP microscaling)

def test_e8m0_all_codes():
    """E8M0 byte e is 2**(e - 127); 255 is NaN (OCP Microscaling formats)."""
    e = np.arange(256)
    v = O.decode_e8m0(e)
    assert np.isnan(v[255])
    assert v[127] == 1.0 and v[0] == 2.0 ** -127 and v[254] == 2.0 ** 127
    assert np.all(v[1:255] / v[0:254] == 2.0)


def test_mx_quantizer_rule_and_torch_cast():
    """Shared exponent = floor(log2 amax) - 8, so the block maximum lands in
    [256, 512) before saturation at 448; elements agree with torch's E4M3 cast of
    the power-of-two quotient (a library routine); an all-zero block gets byte 0."""
    rng = np.random.default_rng(5)
    x = (rng.normal(0, 1, (40, 128)) * np.repeat(np.exp2(rng.integers(-9, 9, (40, 4))), 32, axis=1)).astype(np.float32)
    x[3, 32:64] = 0.0
    codes, scales = O.quantize_mx_e4m3(x)
    assert codes.shape == x.shape and scales.shape == (40, 4) and scales.dtype == np.uint8
    assert scales[3, 1] == 0 and np.all(codes[3, 32:64] == 0)
    xb = x.reshape(40, 4, 32).astype(np.float64)
    amax = np.abs(xb).max(-1)
    e = scales.astype(np.int64) - 127
    nz = amax > 0
    assert np.all(np.floor(np.log2(amax[nz])) - 8 == e[nz])
    q = np.ldexp(xb, -e[..., None]).astype(np.float32)
    ref = torch.from_numpy(np.clip(q, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes.reshape(40, 4, 32), ref)
    back = O.dequantize_mx_e4m3(codes, scales)
    # E4M3 has 3 mantissa bits: relative error <= 2**-4 below saturation
    unsat = np.abs(q) <= 448
    err = np.abs(back.reshape(40, 4, 32) - xb)
    assert np.all(err[unsat] <= np.abs(xb[unsat]) * 2.0 ** -4 + np.ldexp(1.0, e[..., None] - 9).repeat(32, -1)[unsat])


def test_mx_generator_matches_oracle_quantizer():
    """The input generator's MXFP8 encoder (torch) and the oracle's (numpy,
    nearest-value search) agree code for code."""
    rng = np.random.default_rng(6)
    x = (rng.normal(0, 1, (64, 128)) * np.repeat(np.exp2(rng.integers(-6, 6, (64, 4))), 32, axis=1)).astype(np.float32)
    c0, e0 = O.quantize_mx_e4m3(x)
    c1, e1 = W._quant_blocks_mx(torch.from_numpy(x))
    assert np.array_equal(c0, c1) and np.array_equal(e0, e1)


def test_mx_indexer_one_block_closed_form():
    """H_I = 1, w = 1, the query nonzero only in element i of block b (code 1.0,
    exponent byte 127 + a): I[s] = max(k_code[s, i] * 2**(ek[s, b] - 127) * 2**a, 0)."""
    wl = small("decode_b64", ctx=None, ctx_range=(130, 131), B=1, H_I=1, D_I=64, idx_dtype="mx_e4m3")
    i, b, a = 37, 1, 3
    wl.q_i[:] = 0
    wl.q_i[0, 0, i] = 0x38
    wl.q_i_scale[0, 0, :] = 120            # other blocks hold zeros anyway
    wl.q_i_scale[0, 0, b] = 127 + a
    wl.w[0, 0] = 1.0
    got = O.indexer_scores_row(wl, 0)
    n = got.shape[0]
    rows = O.physical_rows(wl.block_table[0], wl.page_size, np.arange(n))
    kcode = torch.from_numpy(wl.k_i[rows, i].copy()).view(torch.float8_e4m3fn).double().numpy()
    expect = np.maximum(kcode * np.exp2(wl.k_i_scale[rows, b].astype(np.float64) - 127) * 2.0 ** a, 0.0)
    np.testing.assert_array_equal(got, expect.astype(np.float32))


def test_fp8_tile128_latent_row_decode():
    """656-byte rows with one scale per 128 latent dims: latent = code * scale of
    its tile (decoded with torch's E4M3 view), rope = bf16; the generator's tile
    scales are powers of two (so bf16 holds code * scale exactly)."""
    wl = small("decode_b4_long", ctx=[300], K=64, mla_dtype="e4m3_t128")
    row = wl.kv[7]
    scales = row[512:528].copy().view("<f4").astype(np.float64)
    assert np.all(np.log2(scales) == np.round(np.log2(scales)))
    lat = torch.from_numpy(row[:512].copy()).view(torch.float8_e4m3fn).double().numpy() * np.repeat(scales, 128)
    rope = torch.from_numpy(row[528:656].copy()).view(torch.bfloat16).double().numpy()
    got = O.latent_rows(wl, np.array([7]))[0]
    assert np.array_equal(got[:512], lat) and np.array_equal(got[512:], rope)
    # exact in bf16: widening code * scale to bf16 loses nothing
    b = torch.from_numpy(lat).to(torch.bfloat16).double().numpy()
    assert np.array_equal(b, lat)


def test_cache_append_oracle_mx_keys_and_tile128_rows():
    """The writers' variants store exactly the oracle quantiser's output at the
    token's row and leave every other row untouched."""
    rng = np.random.default_rng(9)
    bt = np.array([[3, 1, 0, 2]], dtype=np.int32)
    k_new = (rng.normal(0, 1, (2, 128)) * np.repeat(np.exp2(rng.integers(-5, 5, (2, 4))), 32, axis=1)).astype(np.float32)
    kc0 = rng.integers(0, 256, (256, 128)).astype(np.uint8)
    ks0 = rng.integers(0, 256, (256, 4)).astype(np.uint8)
    kc, ks = O.index_cache_append(bt, 64, np.array([0, 0]), np.array([5, 130]), k_new, kc0, ks0, mx=True)
    for t, pos in enumerate([5, 130]):
        row = int(bt[0, pos // 64]) * 64 + pos % 64
        c, e = O.quantize_mx_e4m3(k_new[t])
        assert np.array_equal(kc[row], c) and np.array_equal(ks[row], e)
        kc0[row], ks0[row] = kc[row], ks[row]
    assert np.array_equal(kc, kc0) and np.array_equal(ks, ks0)
    x = torch.from_numpy(rng.normal(0, 1, (1, 576)).astype(np.float32)).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    cache0 = rng.integers(0, 256, (128, 656)).astype(np.uint8)
    out = O.latent_cache_append(bt, 64, np.array([0]), np.array([70]), bits, cache0, fp8_rows=True, tile128=True)
    row = int(bt[0, 1]) * 64 + 6
    lat = x.float().numpy()[0, :512]
    c, e = O.quantize_mx_e4m3(lat, block=128)
    assert np.array_equal(out[row, :512], c)
    assert np.array_equal(out[row, 512:528].view("<f4"), np.ldexp(np.float32(1), e.astype(np.int32) - 127))
    assert np.array_equal(out[row, 528:].view("<u2"), bits[0, 512:])
    others = np.ones(128, bool)
    others[row] = False
    assert np.array_equal(out[others], cache0[others])


# --------------------------------------------------------------------------- the indexer prolog

def _bits(a):
    return W._bf16_bits(torch.as_tensor(np.asarray(a, dtype=np.float32)))


def test_project_one_hot_weight_and_brute_force():
    """W = e_i e_j^T picks input j into output i; on random tiny inputs the
    projection equals a pure-Python triple loop over the bf16 values."""
    rng = np.random.default_rng(0)
    x = _bits(rng.standard_normal((3, 5)))
    w = np.zeros((4, 5), np.float32)
    w[2, 3] = 1.0
    y = O.project(x, _bits(w))
    xv = O.decode_bf16(x)
    assert np.array_equal(y[:, 2], xv[:, 3]) and np.count_nonzero(y[:, [0, 1, 3]]) == 0
    wr = _bits(rng.standard_normal((4, 5)))
    wv = O.decode_bf16(wr)
    y = O.project(x, wr)
    for t in range(3):
        for i in range(4):
            acc = 0.0
            for j in range(5):
                acc += float(xv[t, j]) * float(wv[i, j])
            assert abs(y[t, i] - acc) <= 1e-12 * (1 + abs(acc))


def test_layer_norm_hand_example_and_invariants():
    v = np.array([1.0, 2.0, 3.0, 4.0])
    # mean 2.5, population variance 1.25
    ref = (v - 2.5) / math.sqrt(1.25)
    assert np.allclose(O.layer_norm(v, np.ones(4), np.zeros(4), eps=0.0), ref, rtol=0, atol=1e-15)
    assert np.allclose(O.layer_norm(v, 2 * np.ones(4), np.ones(4), eps=0.0), 2 * ref + 1, rtol=0, atol=1e-15)
    rng = np.random.default_rng(1)
    u = rng.standard_normal((5, 128)) * 3 + 7
    n = O.layer_norm(u, np.ones(128), np.zeros(128))
    assert np.allclose(n.mean(axis=1), 0, atol=1e-12)
    assert np.allclose((n ** 2).mean(axis=1), 1 / (1 + O.LAYERNORM_EPS / u.var(axis=1)), rtol=1e-12)
    # a constant vector normalises to beta (its deviation is zero)
    assert np.allclose(O.layer_norm(np.full(8, 3.0), np.ones(8), np.arange(8.0)), np.arange(8.0))


def test_indexer_prolog_brute_force_tiny():
    """Every output of the prolog from pure-Python loops over the bf16 inputs:
    the projections, the layer normalisation of the key, the per-(token, head)
    quantisation of the query (the quantisation rule is pinned on its own above),
    and the cache row of each new key."""
    pl = W.make_prolog("prolog_tiny", seed=3)
    r = O.indexer_prolog(pl)
    xv, xq = O.decode_bf16(pl.x), O.decode_bf16(pl.x_q)
    wq, wk, ww = O.decode_bf16(pl.w_q), O.decode_bf16(pl.w_k), O.decode_bf16(pl.w_w)
    for t in range(pl.T):
        for h in range(pl.H_I):
            qv = [sum(float(wq[h * pl.D_I + d, j]) * float(xq[t, j]) for j in range(pl.d_q)) for d in range(pl.D_I)]
            assert np.allclose(r["q"][t, h], qv, rtol=1e-12, atol=1e-12)
            amax = max(abs(np.float32(v)) for v in qv)
            assert r["q_scale"][t, h] == np.float32(np.float32(amax) / np.float32(448.0))
            codes, _ = O.quantize_e4m3_row(np.asarray(qv, np.float32))
            assert np.array_equal(r["q_codes"][t, h], codes)
        for h in range(pl.H_I):
            wv = sum(float(ww[h, j]) * float(xv[t, j]) for j in range(pl.d_model))
            assert abs(r["w"][t, h] - wv) <= 1e-12 * (1 + abs(wv))
        kv = [sum(float(wk[d, j]) * float(xv[t, j]) for j in range(pl.d_model)) for d in range(pl.D_I)]
        mean = sum(kv) / pl.D_I
        var = sum((v - mean) ** 2 for v in kv) / pl.D_I
        kn = [(v - mean) / math.sqrt(var + 1e-6) * float(pl.gamma[d]) + float(pl.beta[d]) for d, v in enumerate(kv)]
        assert np.allclose(r["k"][t], kn, rtol=1e-12, atol=1e-12)
        b, p = int(pl.q_seq[t]), int(pl.q_pos[t])
        row = int(pl.block_table[b, p // pl.page_size]) * pl.page_size + p % pl.page_size
        codes, scale = O.quantize_e4m3_row(np.asarray(kn, np.float32))
        assert np.array_equal(r["k_cache"][row], codes) and r["k_scale"][row] == scale
    # rows of no new token are untouched
    touched = {int(pl.block_table[int(b), int(p) // pl.page_size]) * pl.page_size + int(p) % pl.page_size
               for b, p in zip(pl.q_seq, pl.q_pos)}
    others = np.array(sorted(set(range(pl.cache_rows)) - touched))
    assert np.array_equal(r["k_cache"][others], pl.k_cache[others])
    assert np.array_equal(r["k_scale"][others], pl.k_scale[others])


def test_indexer_prolog_quantisation_error_bound():
    """Dequantised query and key stay within half an E4M3 step (relative 2**-4
    of the value, or half the smallest subnormal step) of the exact values --
    the error bound of round-to-nearest into E4M3."""
    pl = W.make_prolog("prolog_tiny", seed=4, H_I=4, D_I=16, d_model=96)
    r = O.indexer_prolog(pl)
    deq = O.decode_e4m3(r["q_codes"]) * r["q_scale"].astype(np.float64)[..., None]
    ulp_half = np.maximum(np.abs(r["q"]) * 2.0 ** -4, r["q_scale"].astype(np.float64)[..., None] * 2.0 ** -10)
    assert np.all(np.abs(deq - r["q"]) <= ulp_half * (1 + 1e-6))
    rows = [int(pl.block_table[int(b), int(p) // 64]) * 64 + int(p) % 64 for b, p in zip(pl.q_seq, pl.q_pos)]
    kd = O.decode_e4m3(r["k_cache"][rows]) * r["k_scale"][rows].astype(np.float64)[:, None]
    kh = np.maximum(np.abs(r["k"]) * 2.0 ** -4, r["k_scale"][rows].astype(np.float64)[:, None] * 2.0 ** -10)
    assert np.all(np.abs(kd - r["k"]) <= kh * (1 + 1e-6))
