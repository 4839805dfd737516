"""Plain CPU oracle for the DSA sparse-attention path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and its
Python binding) never imports, calls or links anything here, and this module
imports nothing from the product package: the two share only the seeded input
generator (``dsa_workloads``), which holds none of the method's arithmetic.

Everything is computed in float64 with numpy, one query at a time, in the order
the method states it:

1. lightning-indexer relevance scores with head-weight weighting
   (page "Day0 Inference Adaptation ... Kimi K3.1 Pro", section 3: relevance
   scores between queries and historical positions, head-weight weighting, then
   Top-K; page "Large Language Model Inference Acceleration in Practice",
   section 1.2 "DSA", LI sub-module).  Written out, the head-weighted score is
       I[t, s] = sum_h w[t, h] * ReLU(q_I[t, h] . k_I[s])
   with q_I, k_I the dequantised FP8 values (code * scale): one fp32 scale per
   key and per (query, head), or -- the pages' MXFP8 variant ("Day0 ... Kimi
   K3.1 Pro", section 4; "Large Language Model Inference Acceleration in
   Practice", section 4) -- one power-of-two E8M0 scale per 32 consecutive
   elements (OCP Microscaling formats: shared exponent floor(log2 amax) - 8).
2. per-query Top-K over the causal history s in [0, q_pos[t]], ties to the
   lower index (same page, section 1.2, "selects the Top-K most relevant
   positions").
3. sparse MLA attention (MQA form over the latent cache): softmax over the
   selected rows of scale * q . row[0:576], output sum p * row[0:512]
   (same page, section 1.2, SFA sub-module; section 3.1 on reading the selected
   rows from the paged KV cache).

The FP8 latent cache comes in two granularities: one fp32 scale per token
(656-byte rows, scale at byte 512), or -- the pages' per-token-tile-128 variant
("Large Language Model Inference Acceleration in Practice", section 4;
"Day0 ... Kimi K3.1 Pro", section 4) -- four fp32 scales per token at bytes
[512, 528), one per 128 latent dims.

Readings taken where the pages are silent:
* a query at position p sees s in [0, p] inclusive (its own key is cached);
* scores are formed in float64 and then rounded to float32 once -- the Top-K
  and every comparison downstream use those float32 values;
* -0.0 and +0.0 compare equal (value comparison), ties go to the lower index;
* the index list is a set: valid entries first (here in ascending index order),
  then -1 padding up to K;
* attention skips -1 entries; an empty selection gives out = 0, lse = -inf.

0. (the prolog side) writing a new token into the paged caches: its indexer
   key quantised to FP8 e4m3 with one fp32 scale, its latent row copied (bf16
   cache) or quantised the same way with the rope part kept bf16 (FP8 cache)
   (page "Large Language Model Inference Acceleration in Practice", section 3.2
   "Indexer Prolog" -- K normalisation and the KV-cache update -- and section 4
   "Layered Quantization"; page "Day0 ... Kimi K3.1 Pro", section 4).  The
   quantisation rule is the reading taken for the cache formats: scale =
   amax / 448 in float32 (1 for an all-zero row), code = the E4M3 value nearest
   to x / scale (float32 quotient), ties to the even code, magnitudes beyond
   448 saturated.

Parity pins for every function live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------


def e4m3_table() -> np.ndarray:
    """float64 value of every FP8 E4M3 code, from the OCP 8-bit floating point
    definition: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent
    field 0 encodes subnormals m/8 * 2**-6; S.1111.111 is NaN; there is no
    infinity, so the largest finite magnitude is 1.75 * 2**8 = 448."""
    out = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp_field = (code >> 3) & 0xF
        man = code & 0x7
        if exp_field == 0xF and man == 0x7:
            out[code] = math.nan
        elif exp_field == 0:
            out[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            out[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return out


_E4M3 = e4m3_table()


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the upper 16 bits of an IEEE binary32."""
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return wide.view(np.float32).astype(np.float64)


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code of each float32 value: the finite E4M3 value nearest to x, ties
    to the code with an even mantissa, magnitudes beyond 448 saturated to 448;
    the sign bit is kept (so -0.0 -> 0x80).  Codes 0..126 hold the positive
    finite magnitudes in increasing order (``e4m3_table``)."""
    x = np.asarray(x, dtype=np.float32)
    mags = _E4M3[:127]                                  # 0, 2**-9, ..., 448 (ascending)
    a = np.abs(x).astype(np.float64)
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, 126)   # first magnitude >= a
    lo = np.clip(hi - 1, 0, 126)
    d_hi = np.abs(mags[hi] - a)
    d_lo = np.abs(a - mags[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    mag_code = np.where(pick_lo, lo, hi)
    mag_code = np.where(a >= 448.0, 126, mag_code)      # saturate
    sign = np.signbit(x).astype(np.int64) << 7
    return (sign | mag_code).astype(np.uint8)


def decode_e8m0(e) -> np.ndarray:
    """OCP E8M0 scale byte -> float64: 2**(e - 127) for e in 0..254; 255 is NaN."""
    e = np.asarray(e, dtype=np.int64)
    return np.where(e == 255, math.nan, np.ldexp(1.0, e - 127))


def quantize_mx_e4m3(x, block: int = 32) -> tuple:
    """OCP MXFP8 (E4M3 elements, E8M0 shared scales) along the last axis: for each
    block of `block` consecutive values, shared exponent = floor(log2(amax)) - 8
    (8 = exponent of E4M3's largest normal, 448 = 1.75 * 2**8; -127 for an
    all-zero block), scale byte = exponent + 127, element codes = e4m3_encode of
    x / 2**exponent (an exact power-of-two quotient; saturates at 448).
    Returns (uint8 codes, uint8 scale bytes with the block axis last)."""
    x = np.asarray(x, dtype=np.float32)
    xb = x.reshape(*x.shape[:-1], x.shape[-1] // block, block)
    amax = np.max(np.abs(xb), axis=-1, keepdims=True).astype(np.float64)
    with np.errstate(divide="ignore"):
        exp = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, -127)
    exp = np.clip(exp, -127, 127).astype(np.int64)
    codes = e4m3_encode(np.ldexp(xb.astype(np.float64), -exp).astype(np.float32))
    return codes.reshape(x.shape), (exp + 127).astype(np.uint8)[..., 0]


def dequantize_mx_e4m3(codes, scales, block: int = 32) -> np.ndarray:
    """float64 values of MXFP8 data: code value * 2**(e - 127) of its block."""
    v = decode_e4m3(codes)
    v = v.reshape(*v.shape[:-1], v.shape[-1] // block, block)
    return (v * decode_e8m0(scales)[..., None]).reshape(np.asarray(codes).shape)


def quantize_e4m3_row(x) -> tuple:
    """One token's vector -> (uint8 codes, float32 scale): scale = amax / 448 in
    float32 (1 when the row is all zero), codes = e4m3_encode(x / scale) with the
    quotient formed in float32."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    scale = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    return e4m3_encode((x / scale).astype(np.float32)), scale


def physical_rows(block_table_row: np.ndarray, page_size: int, pos: np.ndarray) -> np.ndarray:
    """Logical position -> cache row through the page table:
    row = block_table[s // page_size] * page_size + s % page_size."""
    pos = np.asarray(pos, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[pos // page_size]
    if np.any(pages < 0):
        raise ValueError("position maps to an unused page-table slot")
    return pages * page_size + pos % page_size


def indexer_keys(wl, rows: np.ndarray) -> np.ndarray:
    """Dequantised indexer keys (float64): code * k_scale[row] for per-token
    scales, code * 2**(e - 127) of the element's 32-value block for MXFP8."""
    if wl.idx_dtype == "e4m3":
        return decode_e4m3(wl.k_i[rows]) * wl.k_i_scale[rows].astype(np.float64)[:, None]
    if wl.idx_dtype == "mx_e4m3":
        return dequantize_mx_e4m3(wl.k_i[rows], wl.k_i_scale[rows])
    return wl.k_i[rows].astype(np.float64)


def indexer_query(wl, t: int) -> np.ndarray:
    """Dequantised indexer query q_I[t, h] (float64 [H_I, D_I]): code * q_scale[t, h],
    or code * 2**(e - 127) of its 32-value block for MXFP8."""
    if wl.idx_dtype == "e4m3":
        return decode_e4m3(wl.q_i[t]) * wl.q_i_scale[t].astype(np.float64)[:, None]
    if wl.idx_dtype == "mx_e4m3":
        return dequantize_mx_e4m3(wl.q_i[t], wl.q_i_scale[t])
    return wl.q_i[t].astype(np.float64)


def latent_rows(wl, rows: np.ndarray) -> np.ndarray:
    """Dequantised latent cache rows (float64 [n, d_latent + d_rope])."""
    rows = np.asarray(rows, dtype=np.int64)
    if wl.mla_dtype == "bf16":
        return decode_bf16(wl.kv[rows])
    if wl.mla_dtype == "f32":
        return wl.kv[rows].astype(np.float64)
    raw = wl.kv[rows]
    if wl.mla_dtype == "e4m3_t128":
        # 656-byte FP8 row with four fp32 scales at [512,528), one per 128 latent dims
        scales = raw[:, 512:528].copy().view("<f4").astype(np.float64)   # [n, 4]
        latent = decode_e4m3(raw[:, :512]) * np.repeat(scales, 128, axis=1)
        rope = decode_bf16(raw[:, 528:656].copy().view("<u2"))
        return np.concatenate([latent, rope], axis=1)
    # 656-byte FP8 row: [0,512) e4m3 latent, [512,516) fp32 scale, [528,656) bf16 rope
    scale = raw[:, 512:516].copy().view("<f4").astype(np.float64)  # [n, 1]
    latent = decode_e4m3(raw[:, :512]) * scale
    rope = decode_bf16(raw[:, 528:656].copy().view("<u2"))
    return np.concatenate([latent, rope], axis=1)


def mla_query(wl, t: int) -> np.ndarray:
    if wl.mla_dtype == "f32":
        return wl.q[t].astype(np.float64)
    return decode_bf16(wl.q[t])


# ---------------------------------------------------------------------------
# step 1: lightning indexer scores
# ---------------------------------------------------------------------------


def indexer_scores_row(wl, t: int) -> np.ndarray:
    """Scores of query t over its causal history s in [0, q_pos[t]]:
    I[t, s] = sum_h w[t, h] * max(q_I[t, h] . k_I[s], 0), in float64,
    returned rounded once to float32 (length q_pos[t] + 1)."""
    b = int(wl.q_seq[t])
    n = int(wl.q_pos[t]) + 1
    rows = physical_rows(wl.block_table[b], wl.page_size, np.arange(n))
    k = indexer_keys(wl, rows)                 # [n, D_I]
    q = indexer_query(wl, t)                   # [H_I, D_I]
    dots = q @ k.T                             # [H_I, n]: q_I[t,h] . k_I[s]
    relu = np.maximum(dots, 0.0)
    weights = wl.w[t].astype(np.float64)       # [H_I]
    scores = weights @ relu                    # sum over heads h
    return scores.astype(np.float32)


def indexer_scores(wl, ts=None) -> np.ndarray:
    """float32 [len(ts), max_ctx]; -inf beyond each query's causal history."""
    ts = range(wl.T) if ts is None else ts
    ts = list(ts)
    out = np.full((len(ts), wl.max_ctx), -np.inf, dtype=np.float32)
    for i, t in enumerate(ts):
        row = indexer_scores_row(wl, t)
        out[i, :row.shape[0]] = row
    return out


# ---------------------------------------------------------------------------
# step 2: per-query Top-K
# ---------------------------------------------------------------------------


def topk_row(scores: np.ndarray, n: int, K: int) -> np.ndarray:
    """The K largest of scores[0:n] (float32 values compared as numbers), ties
    to the lower index; all n kept when n <= K.  Returns int32 [K]: the chosen
    positions in ascending order, then -1 padding."""
    vals = np.asarray(scores[:n], dtype=np.float64)
    order = np.lexsort((np.arange(n), -vals))  # primary: value desc, secondary: index asc
    chosen = np.sort(order[:min(K, n)])
    out = np.full(K, -1, dtype=np.int32)
    out[:chosen.shape[0]] = chosen
    return out


def topk(scores: np.ndarray, q_pos: np.ndarray, K: int) -> np.ndarray:
    T = scores.shape[0]
    return np.stack([topk_row(scores[t], int(q_pos[t]) + 1, K) for t in range(T)]) if T else \
        np.zeros((0, K), np.int32)


# ---------------------------------------------------------------------------
# step 3: sparse MLA attention over the selected latent rows
# ---------------------------------------------------------------------------


def sparse_mla_attn_row(wl, t: int, idx_row: np.ndarray):
    """For every head h of query t, over the selected positions S (idx >= 0):
    logit_s = scale * q[t, h] . row_s[0:d_qk]; p = softmax over S;
    out[h] = sum_s p_s * row_s[0:d_v]; lse[h] = log sum_s exp(logit_s).
    Returns float64 (out [H, d_v], lse [H])."""
    sel = np.asarray(idx_row, dtype=np.int64)
    sel = sel[sel >= 0]
    H, dv = wl.H, wl.d_v
    if sel.shape[0] == 0:
        return np.zeros((H, dv)), np.full(H, -np.inf)
    b = int(wl.q_seq[t])
    rows = physical_rows(wl.block_table[b], wl.page_size, sel)
    kv = latent_rows(wl, rows)                 # [m, d_qk]
    q = mla_query(wl, t)                       # [H, d_qk]
    logits = wl.softmax_scale * (q @ kv.T)     # [H, m]
    mx = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - mx)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    out = p @ kv[:, :dv]
    lse = (mx + np.log(denom))[:, 0]
    return out, lse


def sparse_mla_attn(wl, idx: np.ndarray, ts=None):
    ts = list(range(wl.T)) if ts is None else list(ts)
    out = np.zeros((len(ts), wl.H, wl.d_v))
    lse = np.zeros((len(ts), wl.H))
    for i, t in enumerate(ts):
        out[i], lse[i] = sparse_mla_attn_row(wl, t, idx[i])
    return out, lse


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------


def decode_step(wl, ts=None):
    """scores -> Top-K -> sparse attention for the queries ts (default: all)."""
    ts = list(range(wl.T)) if ts is None else list(ts)
    scores = indexer_scores(wl, ts)
    q_pos = np.asarray([wl.q_pos[t] for t in ts])
    idx = topk(scores, q_pos, wl.K)
    out, lse = sparse_mla_attn(wl, idx, ts)
    return scores, idx, out, lse


# ---------------------------------------------------------------------------
# step 0: writing new tokens into the paged caches (the prolog side)
# ---------------------------------------------------------------------------


def index_cache_append(block_table, page_size, q_seq, q_pos, k_new, k_cache, k_scale, mx: bool = False):
    """Quantise k_new[t] (float32 [T, D]) and store it at the cache row of
    position q_pos[t] of sequence q_seq[t].  Returns updated copies of k_cache
    (uint8 [rows, D]) and k_scale: float32 [rows] (one scale per key), or with
    mx, uint8 [rows, D / 32] E8M0 bytes (quantize_mx_e4m3)."""
    k_cache = np.array(k_cache, dtype=np.uint8, copy=True)
    k_scale = np.array(k_scale, dtype=np.uint8 if mx else np.float32, copy=True)
    for t in range(len(q_pos)):
        row = int(physical_rows(block_table[int(q_seq[t])], page_size, np.array([q_pos[t]]))[0])
        if mx:
            codes, scale = quantize_mx_e4m3(k_new[t])
        else:
            codes, scale = quantize_e4m3_row(k_new[t])
        k_cache[row] = codes
        k_scale[row] = scale
    return k_cache, k_scale


def latent_cache_append(block_table, page_size, q_seq, q_pos, kv_new_bits, cache, fp8_rows: bool,
                        d_latent: int = 512, d_rope: int = 64, tile128: bool = False):
    """Store the new latent rows (bfloat16 bit patterns, uint16 [T, d_latent +
    d_rope]) at the cache rows of their positions.  `cache` is uint8 [rows,
    row_bytes].  bf16 cache: the row's bytes are the input's.  FP8 cache (656-byte
    rows): [0, 512) e4m3 codes of the latent part quantised as one vector,
    [512, 516) its float32 scale, [516, 528) zero, [528, 656) the rope part's bf16
    bytes.  With tile128 the four 128-value tiles of the latent part are
    quantised separately by the MX shared-exponent rule (quantize_mx_e4m3 with
    128-element blocks: power-of-two scales) and their four float32 scales fill
    [512, 528).  Returns an updated copy of the cache."""
    cache = np.array(cache, dtype=np.uint8, copy=True)
    bits = np.asarray(kv_new_bits, dtype=np.uint16)
    for t in range(len(q_pos)):
        row = int(physical_rows(block_table[int(q_seq[t])], page_size, np.array([q_pos[t]]))[0])
        if not fp8_rows:
            b = bits[t].astype("<u2").tobytes()
            cache[row, :len(b)] = np.frombuffer(b, dtype=np.uint8)
            continue
        latent = decode_bf16(bits[t, :d_latent]).astype(np.float32)
        if tile128:
            codes, exps = quantize_mx_e4m3(latent, block=128)
            scales = np.ldexp(np.float32(1.0), exps.astype(np.int32) - 127).astype("<f4")
            cache[row, :d_latent] = codes
            cache[row, d_latent:d_latent + 16] = np.frombuffer(scales.tobytes(), dtype=np.uint8)
        else:
            codes, scale = quantize_e4m3_row(latent)
            cache[row, :d_latent] = codes
            cache[row, d_latent:d_latent + 4] = np.frombuffer(np.float32(scale).astype("<f4").tobytes(),
                                                              dtype=np.uint8)
            cache[row, d_latent + 4:d_latent + 16] = 0
        rope = bits[t, d_latent:d_latent + d_rope].astype("<u2").tobytes()
        cache[row, d_latent + 16:d_latent + 16 + len(rope)] = np.frombuffer(rope, dtype=np.uint8)
    return cache


# ---------------------------------------------------------------------------
# the indexer prolog: step 1's query, head weights and new key made from the new
# tokens' hidden states (page "Large Language Model Inference Acceleration in
# Practice", section 3.2 "Indexer Prolog": query projection, key normalisation
# with the key-cache update, query quantisation, head-weight projection; the
# pages give the four steps, not their formulas -- the readings below are the
# plainest that fit: linear projections, a layer normalisation of the key, and
# the cache formats' own quantisation rule)
# ---------------------------------------------------------------------------

LAYERNORM_EPS = 1e-6


def project(x_bits, w_bits) -> np.ndarray:
    """y[t] = W x[t] for every token: x bfloat16 bit patterns [T, d], W bfloat16
    bit patterns [n, d] (output x input), sums in float64.  Returns float64 [T, n]."""
    return decode_bf16(x_bits) @ decode_bf16(w_bits).T


def layer_norm(v, gamma, beta, eps: float = LAYERNORM_EPS) -> np.ndarray:
    """Over the last axis: (v - mean) / sqrt(var + eps) * gamma + beta, with the
    mean and the population variance (mean square deviation) of v; float64."""
    v = np.asarray(v, dtype=np.float64)
    mean = v.mean(axis=-1, keepdims=True)
    var = ((v - mean) ** 2).mean(axis=-1, keepdims=True)
    return (v - mean) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def indexer_prolog(pl) -> dict:
    """The prolog of one batch of new tokens `pl` (dsa_workloads.PrologWorkload):

    * q[t] = W_q x_q[t] as H_I heads of D_I values; each (t, h) vector quantised
      by the cache formats' rule (quantize_e4m3_row: fp32 scale amax / 448, E4M3
      codes of the fp32 quotient) -- the indexer query of step 1;
    * w[t] = W_w x[t] -- the head weights of step 1;
    * k[t] = layer_norm(W_k x[t], gamma, beta) -- the new index key, quantised
      and written to the cache row of position q_pos[t] (index_cache_append).

    Values are formed in float64 and rounded to float32 where the rule quantises
    them.  Returns q (float64 [T, H_I, D_I]), q_codes, q_scale, w (float64
    [T, H_I]), k (float64 [T, D_I]) and the updated k_cache / k_scale."""
    T = pl.T
    q = project(pl.x_q, pl.w_q).reshape(T, pl.H_I, pl.D_I)
    q_codes = np.empty((T, pl.H_I, pl.D_I), dtype=np.uint8)
    q_scale = np.empty((T, pl.H_I), dtype=np.float32)
    for t in range(T):
        for h in range(pl.H_I):
            q_codes[t, h], q_scale[t, h] = quantize_e4m3_row(q[t, h].astype(np.float32))
    w = project(pl.x, pl.w_w)
    k = layer_norm(project(pl.x, pl.w_k), pl.gamma, pl.beta)
    k_cache, k_scale = index_cache_append(pl.block_table, pl.page_size, pl.q_seq, pl.q_pos,
                                          k.astype(np.float32), pl.k_cache, pl.k_scale)
    return dict(q=q, q_codes=q_codes, q_scale=q_scale, w=w, k=k, k_cache=k_cache, k_scale=k_scale)
