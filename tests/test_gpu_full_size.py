"""GPU parity at the full benchmark sizes (decode batch 1 at 32768 positions,
decode batch 64 over ragged shuffled pages, long-context batch 4 with the FP8
latent cache -- also with MXFP8 index keys -- and the 16384-token causal
prefill), in the launch configuration
the benchmark times: one ``dsa_decode_step`` over the whole batch.

The oracle is too slow for every output at these sizes, so each test samples
query rows (first, last, around the K boundary of the prefill, and seeded
random ones) and checks them one by one: indexer scores, the Top-K index set
against the oracle's own ranking of the oracle scores (bit-exact), the fused
step's selection against the end-to-end rule, and the attention output of the
fused step against the oracle on the same selection."""
import numpy as np
import pytest
import torch

import dsa_indexed_sparse_gb300 as dsa
import dsa_workloads as W
from oracle import dsa_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu


def _samples(wl, n_random, seed):
    T = wl.T
    fixed = [0, T - 1]
    if wl.name.startswith("prefill"):
        fixed += [t for t in (1, wl.K - 2, wl.K - 1, wl.K, wl.K + 1) if t < T]
    rng = np.random.default_rng(seed)
    extra = rng.choice(T, size=min(T, n_random), replace=False).tolist()
    return sorted(set(int(t) for t in fixed + extra if 0 <= t < T))


SIZES = {
    "decode_b1": 0,
    "decode_b64": 4,
    "decode_b4_long": 0,
    "prefill_16k": 3,
    "decode_b4_long_mx": 0,   # MXFP8 index keys at the long-context size
    "decode_b4_long_t128": 0,  # FP8 latent rows scaled per 128 dims, long context
}


@pytest.fixture(scope="module", params=sorted(SIZES))
def full(request, dev):
    name = request.param
    wl = W.make(name, seed=0)
    run = P.Run(wl, dev)
    ts = _samples(wl, SIZES[name], seed=7)
    o_scores = O.indexer_scores(wl, ts)
    yield wl, run, ts, o_scores
    del run
    torch.cuda.empty_cache()


def _decode_step_rows(run, ts):
    """One fused step over the whole batch; returns the sampled rows only."""
    wl, dev = run.wl, run.dev
    out = torch.full((wl.T, wl.H, wl.d_v), float("nan"), dtype=run.out_dtype, device=dev)
    lse = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=dev)
    sel = torch.full((wl.T, wl.K), -7, dtype=torch.int32, device=dev)
    n = dsa.decode_workspace_size(run.seq, run.idxr, run.mla, wl.K)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    dsa.decode_step(run.seq, run.idxr, run.mla, wl.K, out, ws, lse=lse, idx_out=sel)
    plan = dsa.last_plan()
    dsa.check_status()
    it = torch.tensor(ts, dtype=torch.long, device=dev)
    rows = (out.index_select(0, it).float().cpu().numpy(), lse.index_select(0, it).cpu().numpy(),
            sel.index_select(0, it).cpu().numpy())
    del out, lse, sel, ws
    return rows + (plan,)


def test_full_size_indexer_scores(full):
    wl, run, ts, o_scores = full
    s = torch.full((wl.T, run.ld), float("nan"), dtype=torch.float32, device=run.dev)
    dsa.indexer_scores(run.seq, run.idxr, s)
    plan = dsa.last_plan()
    dsa.check_status()
    g = s.index_select(0, torch.tensor(ts, dtype=torch.long, device=run.dev)).cpu().numpy()
    del s
    assert "indexer_tc" in plan, plan
    P.check_scores(g, o_scores, wl.q_pos, ts)


def test_full_size_topk_bit_exact_on_oracle_scores(full):
    """The sampled rows as their own batch (same contexts, same page tables)."""
    wl, run, ts, o_scores = full
    dev = run.dev
    sub = dsa.Seq(q_seq=torch.tensor([int(wl.q_seq[t]) for t in ts], dtype=torch.int32, device=dev),
                  q_pos=torch.tensor([int(wl.q_pos[t]) for t in ts], dtype=torch.int32, device=dev),
                  block_table=run.seq.block_table, max_ctx=wl.max_ctx, cache_rows=wl.cache_rows,
                  page_size=wl.page_size, q_per_seq=0)
    pad = np.full((len(ts), run.ld), -np.inf, dtype=np.float32)
    pad[:, :o_scores.shape[1]] = o_scores[:, :run.ld]
    s = torch.from_numpy(pad).to(dev)
    idx = torch.full((len(ts), wl.K), -7, dtype=torch.int32, device=dev)
    dsa.topk(sub, s, wl.K, idx)
    plan = dsa.last_plan()
    dsa.check_status()
    assert "topk_radix" in plan, plan
    q_pos = np.asarray([wl.q_pos[t] for t in ts])
    o_idx = O.topk(o_scores, q_pos, wl.K)
    P.check_topk_exact(idx.cpu().numpy(), o_idx, q_pos, wl.K)


def test_full_size_decode_step(full):
    wl, run, ts, o_scores = full
    g_out, g_lse, g_idx, plan = _decode_step_rows(run, ts)
    assert P.step_plan_ok(plan), plan
    P.check_selection(g_idx, o_scores, wl.q_pos, wl.K, ts)
    o_out, o_lse = O.sparse_mla_attn(wl, g_idx, ts)
    P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


def test_full_size_topk_every_row_in_the_step_launch(dev):
    """Decode batch 64, all 64 queries: dsa_topk in one launch over the whole
    batch (the cluster size the benchmark's Top-K stage uses) is bit-exact on the
    oracle's scores of every row, and the decode step's own selection (the fused
    plan) equals dsa_topk run on the GPU's scores, bit for bit."""
    wl = W.make("decode_b64", seed=0)
    run = P.Run(wl, dev)
    o_scores = O.indexer_scores(wl)
    g_idx, plan = run.topk(o_scores)
    assert "topk_radix[cluster=2," in plan, plan
    P.check_topk_exact(g_idx, O.topk(o_scores, wl.q_pos, wl.K), wl.q_pos, wl.K)
    _, _, s_idx, step_plan = run.decode_step()
    np.testing.assert_array_equal(s_idx, run.chained_indices())
    P.check_selection(s_idx, o_scores, wl.q_pos, wl.K)
