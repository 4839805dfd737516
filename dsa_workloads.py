"""Seeded synthetic inputs for the DSA sparse-attention path.

This module only *generates* inputs: random draws, the paged-cache layout and the
cache storage formats (FP8 e4m3 codes with per-row fp32 scales, bf16 bits).  It
holds none of the method's arithmetic (no scoring, no selection, no attention):
both the CPU oracle and the CUDA path consume the same bytes produced here.

Storage formats (the "cache format" inputs the pages' quantised paths assume,
"Day0 Inference Adaptation ... Kimi K3.1 Pro", section 4; the per-token fp32
scale replaces the pages' MXFP8 group scales, see the workload list below):

* indexer keys  ``k_i``  : ``uint8 [cache_rows, D_I]`` e4m3 codes, ``k_i_scale`` fp32 per row
* indexer query ``q_i``  : ``uint8 [T, H_I, D_I]`` e4m3 codes, ``q_i_scale`` fp32 per (t, h)
* head weights  ``w``    : fp32 ``[T, H_I]``
* MLA query     ``q``    : bf16 bits ``uint16 [T, H, d_latent + d_rope]``
* latent cache  ``kv``   : bf16 bits ``uint16 [cache_rows, d_latent + d_rope]``, or
  the 656-byte FP8 row (``uint8 [cache_rows, 656]``): bytes [0, 512) e4m3 latent,
  [512, 516) fp32 scale, [516, 528) zero, [528, 656) 64 bf16 rope values
* the tiny check uses fp32 everywhere (``float32`` arrays, no scales)

Quantisation rule used to *produce* e4m3 data: scale = amax / 448 over the row
(1 for an all-zero row); code = round-to-nearest-even of x / scale, saturated to
+-448, done by ``torch``'s float8_e4m3fn cast.

Draw order for seed ``s`` (one ``torch.Generator`` on the CPU):
context lengths -> page permutation -> low-rank bases -> indexer keys ->
indexer queries -> head weights -> latent rows -> MLA queries.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

PAGE_SIZE = 64
FP8_ROW_BYTES = 656          # 512 e4m3 + 4 scale + 12 reserved + 128 rope
FP8_SCALE_OFFSET = 512
FP8_ROPE_OFFSET = 528
E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    # sequences, queries and paging
    B: int
    T: int
    K: int
    page_size: int
    max_ctx: int                 # upper bound of q_pos[t] + 1 over t
    q_per_seq: int               # queries per sequence when uniform & consecutive, else 0
    q_seq: np.ndarray            # int32 [T]
    q_pos: np.ndarray            # int32 [T]
    seq_lens: np.ndarray         # int32 [B]
    block_table: np.ndarray      # int32 [B, max_pages]  (-1 = unused slot)
    cache_rows: int
    # lightning indexer
    idx_dtype: str               # "e4m3" (per-token / per-head fp32 scales) | "mx_e4m3" (E8M0 per 32) | "f32"
    H_I: int
    D_I: int
    q_i: np.ndarray
    q_i_scale: np.ndarray        # float32 [T, H_I]
    w: np.ndarray                # float32 [T, H_I]
    k_i: np.ndarray
    k_i_scale: np.ndarray        # float32 [cache_rows]
    # MLA latent attention
    mla_dtype: str               # "bf16" | "e4m3" (per-token scale) | "e4m3_t128" (scale per 128 latent dims) | "f32"
    H: int
    d_latent: int
    d_rope: int
    q: np.ndarray
    kv: np.ndarray
    row_bytes: int
    softmax_scale: float

    @property
    def d_qk(self) -> int:
        return self.d_latent + self.d_rope

    @property
    def d_v(self) -> int:
        return self.d_latent


@dataclasses.dataclass
class Spec:
    """Shape/distribution recipe of one workload."""
    name: str
    ctx: list                    # context length per sequence (or None -> drawn)
    q_len: int                   # query tokens per sequence (the last q_len positions)
    K: int
    H_I: int = 64
    D_I: int = 128
    idx_dtype: str = "e4m3"
    mx_block_spread: int = 4     # "mx_e4m3": block magnitudes 2**U{-4..4} before quantising
    w_var: float = 1.0 / 64.0
    H: int = 128
    d_latent: int = 512
    d_rope: int = 64
    mla_dtype: str = "bf16"
    softmax_scale: float = 1.0 / math.sqrt(192.0)
    shuffle_pages: bool = False
    ctx_range: Optional[tuple] = None   # (lo, hi) inclusive integer-uniform draw
    B: int = 1
    low_rank: int = 0            # rank of the structured component (0 = none)
    # per-element std of the structured component (the N(0,1) part has std 1):
    # large enough that it shapes the indexer scores (structured : noise ~ 1 : 1
    # in a 128-d dot product) and the attention logits (~2 : 1 over 576 dims),
    # small enough that the inputs stay close to N(0, 1) and the bf16 outputs stay
    # in the range where a bf16 result can meet the stated 2e-2 max-abs tolerance
    low_rank_amp: float = 0.5
    # "e4m3_t128" rows: tile scales as powers of two (the cache writer's rule) or,
    # when False, any fp32 value (amax / 448 of the tile)
    t128_pow2: bool = True


def spec(name: str, **over) -> Spec:
    """Named workload recipes (seeded, synthetic)."""
    base = {
        # 1 sequence of 256 tokens, 8 queries at 248..255, fp32 throughout
        "tiny_fp32": dict(ctx=[256], q_len=8, K=32, H_I=4, D_I=32, idx_dtype="f32",
                          w_var=0.25, H=4, d_latent=64, d_rope=16, mla_dtype="f32",
                          softmax_scale=1.0 / math.sqrt(80.0)),
        # one decode token against a 32768-token context, contiguous pages
        "decode_b1": dict(ctx=[32768], q_len=1, K=2048),
        # 64 sequences, ctx ~ U{2048..8192}, shuffled 64-token pages
        "decode_b64": dict(ctx=None, ctx_range=(2048, 8192), B=64, q_len=1, K=2048,
                           shuffle_pages=True),
        # causal prefill of 16384 tokens with a rank-8 structured component
        "prefill_16k": dict(ctx=[16384], q_len=16384, K=2048, low_rank=8),
        # 4 x 131072 context, FP8 latent cache with per-token fp32 scale
        "decode_b4_long": dict(ctx=[131072] * 4, B=4, q_len=1, K=2048, mla_dtype="e4m3"),
        # the same two decode shapes with MXFP8 index keys and queries (E8M0 per 32)
        "decode_b64_mx": dict(ctx=None, ctx_range=(2048, 8192), B=64, q_len=1, K=2048,
                              shuffle_pages=True, idx_dtype="mx_e4m3"),
        "decode_b4_long_mx": dict(ctx=[131072] * 4, B=4, q_len=1, K=2048, mla_dtype="e4m3",
                                  idx_dtype="mx_e4m3"),
        # long decode with the FP8 latent cache scaled per 128-dim tile
        "decode_b4_long_t128": dict(ctx=[131072] * 4, B=4, q_len=1, K=2048, mla_dtype="e4m3_t128"),
    }[name]
    base.update(over)
    if base.get("ctx") is not None:
        base["B"] = len(base["ctx"])
    return Spec(name=name, **base)


def _quant_rows_e4m3(x: torch.Tensor):
    """Per-row e4m3 quantisation of the last axis: returns (uint8 codes, fp32 scales)."""
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (x / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).numpy(), scale.squeeze(-1).to(torch.float32).numpy()


MX_BLOCK = 32        # elements sharing one E8M0 scale (OCP MXFP8)
E4M3_EMAX = 8        # exponent of the largest normal E4M3 value (448 = 1.75 * 2**8)


def _quant_blocks_mx(x: torch.Tensor, block: int = MX_BLOCK):
    """OCP MXFP8 along the last axis: blocks of `block` (32) elements share an
    E8M0 scale 2**(e - 127) with e - 127 = floor(log2(amax of the block)) - 8
    (-127 for an all-zero block); elements are the E4M3 values nearest to
    x / scale (ties to even), clamped to +-448.  Returns (uint8 codes, uint8 E8M0
    exponents with the block axis last)."""
    shp = x.shape
    xb = x.reshape(*shp[:-1], shp[-1] // block, block)
    amax = xb.abs().amax(dim=-1, keepdim=True)
    _, e = torch.frexp(amax)                          # amax = m * 2**e, m in [0.5, 1)
    sexp = torch.where(amax > 0, e - 1 - E4M3_EMAX, torch.full_like(e, -127)).clamp(-127, 127)
    codes = torch.ldexp(xb, -sexp).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return (codes.view(torch.uint8).reshape(shp).numpy(),
            (sexp + 127).to(torch.uint8).squeeze(-1).numpy())


def _spread_blocks(g: torch.Generator, x: torch.Tensor, spread: int, block: int = MX_BLOCK, top: int = None):
    """Multiplies every `block`-element block of the last axis by 2**r, r uniform
    in [-spread, top] (top = spread unless given; seeded), so that blocks of one
    vector differ in range."""
    shp = x.shape
    top = spread if top is None else top
    r = torch.randint(-spread, top + 1, (*shp[:-1], shp[-1] // block, 1), generator=g)
    x.view(*shp[:-1], shp[-1] // block, block).mul_(torch.pow(2.0, r.to(torch.float32)))


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _randn(g: torch.Generator, shape, chunk_rows: int = 1 << 16) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.float32)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g)
    return out


def _add_low_rank(g, x: torch.Tensor, basis: torch.Tensor, amp: float, chunk_rows: int = 1 << 15):
    """x[..., :] += amp * z @ basis with z ~ N(0, 1)^rank drawn per row (in place)."""
    flat = x.view(-1, x.shape[-1])
    rank = basis.shape[0]
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        z = torch.randn((r1 - r0, rank), generator=g)
        flat[r0:r1] += amp * (z @ basis)


def make(name_or_spec, seed: int = 0, **over) -> Workload:
    sp = name_or_spec if isinstance(name_or_spec, Spec) else spec(name_or_spec, **over)
    g = torch.Generator(device="cpu").manual_seed(seed)
    P = PAGE_SIZE

    # --- context lengths and paging --------------------------------------
    if sp.ctx is None:
        lo, hi = sp.ctx_range
        ctx = torch.randint(lo, hi + 1, (sp.B,), generator=g).tolist()
    else:
        ctx = list(sp.ctx)
    B = len(ctx)
    pages_per_seq = [(c + P - 1) // P for c in ctx]
    n_pages = sum(pages_per_seq)
    if sp.shuffle_pages:
        perm = torch.randperm(n_pages, generator=g).numpy().astype(np.int32)
    else:
        perm = np.arange(n_pages, dtype=np.int32)
    max_pages = max(pages_per_seq)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b, npg in enumerate(pages_per_seq):
        block_table[b, :npg] = perm[off:off + npg]
        off += npg
    cache_rows = n_pages * P

    q_len = sp.q_len
    q_seq = np.repeat(np.arange(B, dtype=np.int32), q_len)
    q_pos = np.concatenate([np.arange(c - q_len, c, dtype=np.int32) for c in ctx])
    T = len(q_seq)

    # --- low-rank bases ----------------------------------------------------
    dk = sp.d_latent + sp.d_rope
    if sp.low_rank:
        u_idx = torch.randn((sp.low_rank, sp.D_I), generator=g) / math.sqrt(sp.low_rank)
        u_mla = torch.randn((sp.low_rank, dk), generator=g) / math.sqrt(sp.low_rank)

    # --- lightning indexer inputs -----------------------------------------
    k_f = _randn(g, (cache_rows, sp.D_I))
    if sp.low_rank:
        _add_low_rank(g, k_f, u_idx, sp.low_rank_amp)
    q_f = _randn(g, (T, sp.H_I, sp.D_I))
    if sp.low_rank:
        _add_low_rank(g, q_f, u_idx, sp.low_rank_amp)
    w = (torch.randn((T, sp.H_I), generator=g) * math.sqrt(sp.w_var)).numpy()
    if sp.idx_dtype == "e4m3":
        k_i, k_i_scale = _quant_rows_e4m3(k_f)
        q_i, q_i_scale = _quant_rows_e4m3(q_f)
    elif sp.idx_dtype == "mx_e4m3":
        _spread_blocks(g, k_f, sp.mx_block_spread)
        _spread_blocks(g, q_f, sp.mx_block_spread)
        k_i, k_i_scale = _quant_blocks_mx(k_f)
        q_i, q_i_scale = _quant_blocks_mx(q_f)
    elif sp.idx_dtype == "f32":
        k_i, k_i_scale = k_f.numpy(), np.ones(cache_rows, np.float32)
        q_i, q_i_scale = q_f.numpy(), np.ones((T, sp.H_I), np.float32)
    else:
        raise ValueError(sp.idx_dtype)
    del k_f, q_f

    # --- MLA latent cache and queries --------------------------------------
    kv_f = _randn(g, (cache_rows, dk))
    if sp.low_rank:
        _add_low_rank(g, kv_f, u_mla, sp.low_rank_amp)
    if sp.mla_dtype == "bf16":
        kv = _bf16_bits(kv_f)
        row_bytes = dk * 2
    elif sp.mla_dtype == "e4m3":
        assert sp.d_latent == 512 and sp.d_rope == 64
        codes, scale = _quant_rows_e4m3(kv_f[:, :sp.d_latent])
        kv = np.zeros((cache_rows, FP8_ROW_BYTES), dtype=np.uint8)
        kv[:, :512] = codes
        kv[:, FP8_SCALE_OFFSET:FP8_SCALE_OFFSET + 4] = scale.astype("<f4").view(np.uint8).reshape(-1, 4)
        kv[:, FP8_ROPE_OFFSET:] = _bf16_bits(kv_f[:, sp.d_latent:]).view(np.uint8).reshape(cache_rows, -1)
        row_bytes = FP8_ROW_BYTES
    elif sp.mla_dtype == "e4m3_t128":
        # the same 656-byte row with four scales, one per 128 latent dims, each a
        # power of two (the shared-exponent rule of the MX formats on 128-blocks)
        assert sp.d_latent == 512 and sp.d_rope == 64
        lat = kv_f[:, :sp.d_latent].contiguous()
        _spread_blocks(g, lat, 2, block=128, top=0)   # tiles shrunk by 2**{0,-1,-2}
        if sp.t128_pow2:
            codes, exps = _quant_blocks_mx(lat, block=128)
            scales = np.ldexp(np.float32(1.0), exps.astype(np.int32) - 127).astype("<f4")   # [rows, 4]
        else:   # per-tile amax / 448: arbitrary fp32 scales
            c4, s4 = _quant_rows_e4m3(lat.view(cache_rows, 4, 128))
            codes, scales = c4.reshape(cache_rows, 512), s4.astype("<f4")
        kv = np.zeros((cache_rows, FP8_ROW_BYTES), dtype=np.uint8)
        kv[:, :512] = codes
        kv[:, FP8_SCALE_OFFSET:FP8_SCALE_OFFSET + 16] = scales.view(np.uint8).reshape(-1, 16)
        kv[:, FP8_ROPE_OFFSET:] = _bf16_bits(kv_f[:, sp.d_latent:]).view(np.uint8).reshape(cache_rows, -1)
        row_bytes = FP8_ROW_BYTES
    elif sp.mla_dtype == "f32":
        kv = kv_f.numpy()
        row_bytes = dk * 4
    else:
        raise ValueError(sp.mla_dtype)
    del kv_f
    q_m = _randn(g, (T, sp.H, dk))
    if sp.low_rank:
        _add_low_rank(g, q_m, u_mla, sp.low_rank_amp)
    q = q_m.numpy() if sp.mla_dtype == "f32" else _bf16_bits(q_m)
    del q_m

    return Workload(
        name=sp.name, B=B, T=T, K=sp.K, page_size=P, max_ctx=int(max(ctx)),
        q_per_seq=q_len, q_seq=q_seq, q_pos=q_pos,
        seq_lens=np.asarray(ctx, dtype=np.int32), block_table=block_table,
        cache_rows=cache_rows,
        idx_dtype=sp.idx_dtype, H_I=sp.H_I, D_I=sp.D_I, q_i=q_i,
        q_i_scale=np.ascontiguousarray(q_i_scale, dtype=np.uint8 if sp.idx_dtype == "mx_e4m3" else np.float32),
        w=np.ascontiguousarray(w, dtype=np.float32), k_i=k_i,
        k_i_scale=np.ascontiguousarray(k_i_scale, dtype=np.uint8 if sp.idx_dtype == "mx_e4m3" else np.float32),
        mla_dtype=sp.mla_dtype, H=sp.H, d_latent=sp.d_latent, d_rope=sp.d_rope,
        q=q, kv=kv, row_bytes=row_bytes, softmax_scale=float(sp.softmax_scale),
    )


NAMES = ("tiny_fp32", "decode_b1", "decode_b64", "prefill_16k", "decode_b4_long")


def device_tensors(wl: Workload, device, copies: int = 1) -> dict:
    """Copies a workload's arrays to ``device`` as torch tensors, grouped under the
    field names of the binding's Seq / Indexer / Mla records (plus ``K``).
    ``copies > 1`` returns a list of independent copies of the cache-side and
    query-side tensors (used to rotate inputs past the L2 cache)."""
    def t(a, dtype=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            x = x.view(dtype)
        return x.to(device)

    def one():
        seq = dict(q_seq=t(wl.q_seq), q_pos=t(wl.q_pos), block_table=t(wl.block_table),
                   max_ctx=wl.max_ctx, cache_rows=wl.cache_rows, page_size=wl.page_size,
                   q_per_seq=wl.q_per_seq)
        idx = dict(q=t(wl.q_i), w=t(wl.w), k_cache=t(wl.k_i), q_scale=t(wl.q_i_scale),
                   k_scale=t(wl.k_i_scale))
        if wl.idx_dtype == "mx_e4m3":
            idx["dtype"] = 3  # MXFP8: E4M3 codes + one E8M0 scale byte per 32 elements
        if wl.mla_dtype == "bf16":
            q, kv = t(wl.q.view(np.int16), torch.bfloat16), t(wl.kv.view(np.int16), torch.bfloat16)
            dt = None
        elif wl.mla_dtype == "e4m3":
            q, kv = t(wl.q.view(np.int16), torch.bfloat16), t(wl.kv)
            dt = 2  # FP8 row format
        elif wl.mla_dtype == "e4m3_t128":
            q, kv = t(wl.q.view(np.int16), torch.bfloat16), t(wl.kv)
            dt = 4  # FP8 rows with a power-of-two scale per 128 latent dims
        else:
            q, kv = t(wl.q), t(wl.kv)
            dt = None
        mla = dict(q=q, kv_cache=kv, d_latent=wl.d_latent, d_rope=wl.d_rope,
                   softmax_scale=wl.softmax_scale, dtype=dt)
        return dict(seq=seq, indexer=idx, mla=mla, K=wl.K)

    if copies == 1:
        return one()
    return [one() for _ in range(copies)]


# ----------------------------------------------------------------------------- the indexer prolog

@dataclasses.dataclass
class PrologWorkload:
    """New tokens for the indexer prolog: hidden states x [T, d_model] and query
    latents x_q [T, d_q] (bf16 bit patterns), the projection weights (bf16 bit
    patterns, output x input), the key normalisation's gamma / beta (fp32), and a
    paged index-key cache the new keys are written into."""
    name: str
    B: int
    T: int
    q_seq: np.ndarray          # int32 [T]
    q_pos: np.ndarray          # int32 [T] position of each new token
    block_table: np.ndarray    # int32 [B, pages]
    page_size: int
    cache_rows: int
    max_ctx: int
    d_model: int
    d_q: int
    H_I: int
    D_I: int
    x: np.ndarray              # uint16 [T, d_model]
    x_q: np.ndarray            # uint16 [T, d_q]
    w_q: np.ndarray            # uint16 [H_I * D_I, d_q]
    w_k: np.ndarray            # uint16 [D_I, d_model]
    w_w: np.ndarray            # uint16 [H_I, d_model]
    gamma: np.ndarray          # float32 [D_I]
    beta: np.ndarray           # float32 [D_I]
    k_cache: np.ndarray        # uint8 [cache_rows, D_I] (earlier keys)
    k_scale: np.ndarray        # float32 [cache_rows]


PROLOG_SPECS = {
    # sizes of the projections are not on the pages: a 7168-wide hidden state and
    # a 1536-wide query latent, 64 indexer heads of 128 (the decode configurations)
    "prolog_decode_b64": dict(B=64, q_len=1, ctx=4096, d_model=7168, d_q=1536, H_I=64, D_I=128),
    "prolog_prefill_4k": dict(B=1, q_len=4096, ctx=4096, d_model=7168, d_q=1536, H_I=64, D_I=128),
    "prolog_tiny": dict(B=2, q_len=3, ctx=70, d_model=64, d_q=32, H_I=2, D_I=8),
}


def make_prolog(name: str, seed: int = 0, **over) -> PrologWorkload:
    """Seeded draws: x, x_q ~ N(0, 1); W_q ~ N(0, 1/d_q) (so q ~ N(0, 1));
    W_k ~ N(0, 1/d_model); W_w ~ N(0, 1/(H_I d_model)) (so w ~ N(0, 1/H_I), the
    head weights of the decode configurations); gamma ~ 1 + N(0, 0.1^2),
    beta ~ N(0, 0.1^2); earlier cache keys random E4M3 codes with scale 0.01.
    Sequence b's new tokens sit at positions ctx - q_len .. ctx - 1; pages are a
    seeded permutation of the pool."""
    sp = dict(PROLOG_SPECS[name])
    sp.update(over)
    g = torch.Generator(device="cpu").manual_seed(seed)
    B, q_len, ctx, P = sp["B"], sp["q_len"], sp["ctx"], PAGE_SIZE
    dm, dq, H, D = sp["d_model"], sp["d_q"], sp["H_I"], sp["D_I"]
    npg = (ctx + P - 1) // P
    perm = torch.randperm(B * npg, generator=g).numpy().astype(np.int32)
    block_table = perm.reshape(B, npg)
    T = B * q_len
    q_seq = np.repeat(np.arange(B, dtype=np.int32), q_len)
    q_pos = np.tile(np.arange(ctx - q_len, ctx, dtype=np.int32), B)
    x = _bf16_bits(torch.randn((T, dm), generator=g))
    x_q = _bf16_bits(torch.randn((T, dq), generator=g))
    w_q = _bf16_bits(torch.randn((H * D, dq), generator=g) / math.sqrt(dq))
    w_k = _bf16_bits(torch.randn((D, dm), generator=g) / math.sqrt(dm))
    w_w = _bf16_bits(torch.randn((H, dm), generator=g) / math.sqrt(H * dm))
    gamma = (1.0 + 0.1 * torch.randn((D,), generator=g)).numpy().astype(np.float32)
    beta = (0.1 * torch.randn((D,), generator=g)).numpy().astype(np.float32)
    rows = B * npg * P
    k_cache = torch.randint(0, 126, (rows, D), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    k_scale = np.full(rows, 0.01, dtype=np.float32)
    return PrologWorkload(name=name, B=B, T=T, q_seq=q_seq, q_pos=q_pos, block_table=block_table, page_size=P,
                          cache_rows=rows, max_ctx=ctx, d_model=dm, d_q=dq, H_I=H, D_I=D, x=x, x_q=x_q,
                          w_q=w_q, w_k=w_k, w_w=w_w, gamma=gamma, beta=beta, k_cache=k_cache, k_scale=k_scale)


def prolog_device_tensors(pl: PrologWorkload, device) -> dict:
    """A prolog workload's arrays on ``device``, grouped as the binding's Seq and
    Prolog records plus the key cache they update."""
    def t(a, dtype=None):
        x = torch.from_numpy(np.ascontiguousarray(a))
        return (x.view(dtype) if dtype is not None else x).to(device)
    bf = lambda a: t(a.view(np.int16), torch.bfloat16)
    seq = dict(q_seq=t(pl.q_seq), q_pos=t(pl.q_pos), block_table=t(pl.block_table), max_ctx=pl.max_ctx,
               cache_rows=pl.cache_rows, page_size=pl.page_size, q_per_seq=0)
    pro = dict(x=bf(pl.x), x_q=bf(pl.x_q), w_q=bf(pl.w_q), w_k=bf(pl.w_k), w_w=bf(pl.w_w), gamma=t(pl.gamma),
               beta=t(pl.beta))
    return dict(seq=seq, prolog=pro, k_cache=t(pl.k_cache), k_scale=t(pl.k_scale))
