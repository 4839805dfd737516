"""GPU parity of the indexer prolog (query projection and quantisation, head-weight
projection, key projection + layer normalisation + quantisation into the paged
key cache) against the CPU oracle, through the C ABI.

Quantised outputs: the GPU sums in fp32 where the oracle sums in fp64, so a value
sitting on a rounding boundary may take the neighbouring E4M3 code.  Each
dequantised value must lie within half an E4M3 step of the exact value (the
error bound of round-to-nearest) plus a slack for the fp32 sums (2e-6 of the
vector's largest magnitude), the scales within 1e-5 relative, and at most 0.1 %
of the codes may differ from the oracle's.  Head weights: within 2e-5 of
(|w| + rms w)."""
import numpy as np
import pytest
import torch

import dsa_indexed_sparse_gb300 as dsa
import dsa_workloads as W
from oracle import dsa_oracle as O

pytestmark = pytest.mark.gpu


def _run(pl, dev):
    d = W.prolog_device_tensors(pl, dev)
    seq, pro = dsa.Seq(**d["seq"]), dsa.Prolog(**d["prolog"])
    T, H = pl.T, pl.H_I
    q_codes = torch.full((T, H, pl.D_I), 0xAA, dtype=torch.uint8, device=dev)
    q_scale = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
    w = torch.full((T, H), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(dsa.indexer_prolog_workspace_size(seq, pro), dtype=torch.uint8, device=dev)
    dsa.indexer_prolog(seq, pro, q_codes, q_scale, w, d["k_cache"], d["k_scale"], ws)
    plan = dsa.last_plan()
    dsa.check_status()
    return (q_codes.cpu().numpy(), q_scale.cpu().numpy(), w.cpu().numpy(), d["k_cache"].cpu().numpy(),
            d["k_scale"].cpu().numpy(), plan)


def _check_quantised(codes, scale, exact, o_codes, o_scale):
    """codes [..., D], scale [...]: GPU; exact float64 [..., D]; o_*: oracle's."""
    assert np.all(np.isfinite(scale))
    assert np.all(np.abs(scale - o_scale) <= 1e-5 * o_scale), "scale mismatch"
    deq = O.decode_e4m3(codes) * scale.astype(np.float64)[..., None]
    amax = np.abs(exact).max(axis=-1, keepdims=True)
    half = np.maximum(np.abs(exact) * 2.0 ** -4, scale.astype(np.float64)[..., None] * 2.0 ** -10)
    err = np.abs(deq - exact)
    bad = err > half * (1 + 1e-6) + 2e-6 * amax
    assert not bad.any(), f"{bad.sum()} values beyond the rounding bound, e.g. {err[bad][:3]}"
    frac = np.mean(codes != o_codes)
    assert frac <= 1e-3, f"{frac:.2e} of the codes differ from the oracle's"


@pytest.mark.parametrize("name,over", [
    ("prolog_decode_b64", {}),                                           # 64 tokens: split-K projections
    ("prolog_decode_b64", dict(B=5, d_model=1024, d_q=512, H_I=16)),     # head weights fewer than a tile
    ("prolog_prefill_4k", dict(q_len=300, ctx=300, d_model=512, d_q=256)),   # 300 tokens, three token tiles
])
def test_indexer_prolog_matches_oracle(dev, name, over):
    pl = W.make_prolog(name, seed=5, **over)
    q_codes, q_scale, w, k_cache, k_scale, plan = _run(pl, dev)
    assert plan.startswith("prolog_proj"), plan
    r = O.indexer_prolog(pl)
    _check_quantised(q_codes, q_scale, r["q"], r["q_codes"], r["q_scale"])
    rms = np.sqrt(np.mean(r["w"] ** 2))
    assert np.all(np.abs(w - r["w"]) <= 2e-5 * (np.abs(r["w"]) + rms)), "head weights"
    rows = np.array([int(pl.block_table[int(b), int(p) // pl.page_size]) * pl.page_size + int(p) % pl.page_size
                     for b, p in zip(pl.q_seq, pl.q_pos)])
    _check_quantised(k_cache[rows], k_scale[rows], r["k"], r["k_cache"][rows], r["k_scale"][rows])
    others = np.setdiff1d(np.arange(pl.cache_rows), rows)
    assert np.array_equal(k_cache[others], pl.k_cache[others]) and np.array_equal(k_scale[others], pl.k_scale[others])


def test_indexer_prolog_feeds_the_indexer(dev):
    """The prolog's query codes, scales and head weights used as the indexer's
    inputs give the oracle's scores of the same codes (the formats line up)."""
    pl = W.make_prolog("prolog_decode_b64", seed=6, B=3, ctx=700, d_model=512, d_q=256)
    q_codes, q_scale, w, k_cache, k_scale, _ = _run(pl, dev)
    wl = W.make("decode_b64", seed=6, ctx=[700] * 3, B=3, K=64)
    assert wl.cache_rows == pl.cache_rows and wl.T == pl.T
    wl.block_table, wl.q_pos, wl.q_seq = pl.block_table.astype(np.int32), pl.q_pos, pl.q_seq
    wl.q_i, wl.q_i_scale, wl.w = q_codes, q_scale, w
    wl.k_i, wl.k_i_scale = k_cache, k_scale
    from tests import parity as P
    run = P.Run(wl, dev)
    g, plan = run.scores()
    P.check_scores(g, O.indexer_scores(wl), wl.q_pos)
