"""GPU parity of every stage against the CPU oracle, through the C ABI, on
seeded inputs spanning several tiles, ragged tails and the edge cases of the
method (history shorter than / equal to / one more than K, one-token history,
shuffled pages, query groups of 1, 2 and 4, and 2-8 consecutive query tokens
per sequence as in speculative verification)."""
import re

import numpy as np
import pytest
import torch

import dsa_workloads as W
from oracle import dsa_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu

CASES = {
    "b1_ctx1": ("decode_b1", dict(ctx=[1], K=32)),
    "b1_ctx63": ("decode_b1", dict(ctx=[63], K=32)),
    "b1_ctx64_K64": ("decode_b1", dict(ctx=[64], K=64)),
    "b1_ctx65_K64": ("decode_b1", dict(ctx=[65], K=64)),
    "b1_ctx300_K2048": ("decode_b1", dict(ctx=[300], K=2048)),
    "b1_ctx5000": ("decode_b1", dict(ctx=[5000], K=2048)),
    # 43 row slices of 96 rows: the slice merge takes more than one batch per warp
    "b1_ctx7000_K4096": ("decode_b1", dict(ctx=[7000], K=4096)),
    "b7_shuffled": ("decode_b64", dict(ctx_range=(100, 3000), B=7, K=256)),
    "b5_shuffled_K2048": ("decode_b64", dict(ctx_range=(2048, 8192), B=5, K=2048)),
    "fp8_b2": ("decode_b4_long", dict(ctx=[3000, 4100], B=2, K=2048)),
    "prefill_700": ("prefill_16k", dict(ctx=[700], q_len=700, K=64)),
    "qlen2": ("decode_b1", dict(ctx=[900], q_len=2, K=128)),
    "qlen3": ("decode_b1", dict(ctx=[900], q_len=3, K=128)),
    # speculative-verify shapes: several consecutive query tokens per sequence
    "qlen5": ("decode_b1", dict(ctx=[700], q_len=5, K=64)),
    "qlen8": ("decode_b1", dict(ctx=[900], q_len=8, K=128)),
    "qlen8_b3_shuffled": ("decode_b64", dict(ctx_range=(300, 2500), B=3, q_len=8, K=256)),
    # FP8 cache at a batch where every query gets one row slice: 64 tiles per CTA
    "fp8_b80_single_slice": ("decode_b4_long", dict(ctx=[2100] * 80, B=80, K=2048)),
    # MXFP8 index keys and queries (E8M0 scale per 32 elements; block magnitudes
    # spread over 2**-4..2**4): ragged shuffled batch, several query tokens per
    # sequence, a causal prefill, and with the FP8 latent cache
    "mx_b5_shuffled": ("decode_b64", dict(ctx_range=(100, 3000), B=5, K=256, idx_dtype="mx_e4m3")),
    "mx_qlen4": ("decode_b1", dict(ctx=[900], q_len=4, K=128, idx_dtype="mx_e4m3")),
    "mx_prefill_300": ("prefill_16k", dict(ctx=[300], q_len=300, K=64, idx_dtype="mx_e4m3")),
    "mx_fp8_b2": ("decode_b4_long", dict(ctx=[3000, 4100], B=2, K=2048, idx_dtype="mx_e4m3")),
    # FP8 latent rows with one power-of-two scale per 128 latent dims (the tiles
    # of one row scaled by 2**{0,-1,-2})
    "t128_b2": ("decode_b4_long", dict(ctx=[3000, 4100], B=2, K=2048, mla_dtype="e4m3_t128")),
    "t128_prefill_400": ("prefill_16k", dict(ctx=[400], q_len=400, K=64, mla_dtype="e4m3_t128")),
    # tile scales that are not powers of two (amax / 448 per tile): the kernel
    # rounds code x scale to bf16, held to the FP8-cache tolerance
    "t128_any_scale_b2": ("decode_b4_long", dict(ctx=[3000, 4100], B=2, K=2048, mla_dtype="e4m3_t128",
                                                 t128_pow2=False)),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request, dev):
    name, over = CASES[request.param]
    wl = W.make(name, seed=1, **over)
    oracle_scores = O.indexer_scores(wl)
    return wl, P.Run(wl, dev), oracle_scores


def test_indexer_scores(case):
    wl, run, o_scores = case
    g, plan = run.scores()
    assert "indexer_tc" in plan, plan
    P.check_scores(g, o_scores, wl.q_pos)


def test_topk_bit_exact_on_oracle_scores(case):
    wl, run, o_scores = case
    o_idx = O.topk(o_scores, wl.q_pos, wl.K)
    g_idx, plan = run.topk(o_scores)
    assert "topk_radix" in plan
    P.check_topk_exact(g_idx, o_idx, wl.q_pos, wl.K)


def test_attention_on_oracle_selection(case):
    wl, run, o_scores = case
    o_idx = O.topk(o_scores, wl.q_pos, wl.K)
    g_out, g_lse, plan = run.attn(o_idx)
    assert "attn_tc" in plan, plan
    if wl.K == 4096 and wl.T == 1:
        assert "split=43" in plan and "attn_combine" in plan, plan
    o_out, o_lse = O.sparse_mla_attn(wl, o_idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


def test_decode_step_end_to_end(case):
    wl, run, o_scores = case
    g_out, g_lse, g_idx, plan = run.decode_step()
    assert P.step_plan_ok(plan), plan
    P.check_selection(g_idx, o_scores, wl.q_pos, wl.K)
    if "indexer_topk_fused" in plan:
        # the fused plan selects exactly what the chained plan selects
        np.testing.assert_array_equal(g_idx, run.chained_indices())
    o_out, o_lse = O.sparse_mla_attn(wl, g_idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


def test_tiny_fp32_config(dev):
    """The tiny fp32 configuration runs the generic CUDA-core kernels."""
    wl = W.make("tiny_fp32")
    run = P.Run(wl, dev)
    o_scores = O.indexer_scores(wl)
    g, plan = run.scores()
    assert "indexer_generic<f32>" in plan
    P.check_scores(g, o_scores, wl.q_pos)
    o_idx = O.topk(o_scores, wl.q_pos, wl.K)
    g_idx, _ = run.topk(o_scores)
    P.check_topk_exact(g_idx, o_idx, wl.q_pos, wl.K)
    g_out, g_lse, plan = run.attn(o_idx)
    assert plan == "attn_generic"
    o_out, o_lse = O.sparse_mla_attn(wl, o_idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, "f32")
    g_out, g_lse, g_idx, plan = run.decode_step()
    P.check_selection(g_idx, o_scores, wl.q_pos, wl.K)
    o_out, o_lse = O.sparse_mla_attn(wl, g_idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, "f32")


def test_hand_worked_example_on_gpu(dev):
    from tests.fixtures import hand_example
    wl, exp = hand_example()
    run = P.Run(wl, dev)
    g, _ = run.scores()
    np.testing.assert_array_equal(g[0, :4], np.array(exp["scores"], np.float32))
    g_out, g_lse, g_idx, _ = run.decode_step()
    assert P.as_sets(g_idx)[0] == exp["topk_set"]
    np.testing.assert_allclose(g_out[0, 0], exp["out"], rtol=2e-6)
    np.testing.assert_allclose(g_lse[0, 0], exp["lse"], rtol=2e-6)


def test_generic_indexer_e4m3_matches_oracle(dev):
    """e4m3 with dims the tensor-core path does not cover (H_I = 8, D_I = 64)."""
    wl = W.make("decode_b1", seed=3, ctx=[777], K=64, H_I=8, D_I=64)
    run = P.Run(wl, dev)
    g, plan = run.scores()
    assert plan == "indexer_generic<e4m3>"
    P.check_scores(g, O.indexer_scores(wl), wl.q_pos)


def test_generic_indexer_mxfp8_matches_oracle(dev):
    """MXFP8 with dims the tensor-core path does not cover (H_I = 6, D_I = 64)."""
    wl = W.make("decode_b64", seed=4, ctx_range=(300, 900), B=2, K=64, H_I=6, D_I=64, idx_dtype="mx_e4m3")
    run = P.Run(wl, dev)
    g, plan = run.scores()
    assert plan == "indexer_generic<mxfp8>"
    P.check_scores(g, O.indexer_scores(wl), wl.q_pos)


def test_mxfp8_tensor_core_plan(dev):
    wl = W.make("decode_b64", seed=5, ctx_range=(200, 400), B=3, K=64, q_len=2, idx_dtype="mx_e4m3")
    _, plan = P.Run(wl, dev).scores()
    assert plan.startswith("indexer_tc<G=1,mxfp8>"), plan


# --------------------------------------------------------------------------- top-k edges

def _topk_run(dev, scores, q_pos, K):
    T, L = scores.shape
    wl = W.make("decode_b1", ctx=[L], K=K, H_I=4, D_I=32, H=4, d_latent=64, d_rope=16)
    wl.T = T
    wl.q_seq = np.zeros(T, np.int32)
    wl.q_pos = np.asarray(q_pos, np.int32)
    wl.q_per_seq = 0
    wl.max_ctx = L
    run = P.Run(wl, dev)
    g_idx, plan = run.topk(scores, K)
    o_idx = O.topk(scores, wl.q_pos, K)
    P.check_topk_exact(g_idx, o_idx, wl.q_pos, K)
    return plan


@pytest.mark.parametrize("K", [1, 7, 2048])
def test_topk_ties_and_boundaries(dev, K):
    rng = np.random.default_rng(K)
    L = 5000
    rows = [
        np.zeros(L),                                    # all equal
        rng.integers(-3, 4, L).astype(np.float64),      # heavy ties across the K-th value
        np.arange(L, dtype=np.float64),                 # increasing
        -np.arange(L, dtype=np.float64),                # decreasing
        rng.standard_normal(L),
        np.where(rng.random(L) < 0.5, -0.0, 0.0),       # signed zeros only
    ]
    scores = np.stack(rows).astype(np.float32)
    q_pos = [L - 1, K - 2, K - 1, K, L - 1, 2 * K + 5]
    q_pos = [min(max(p, 0), L - 1) for p in q_pos]
    _topk_run(dev, scores, q_pos, K)


def test_topk_long_history_cluster_and_uncached(dev):
    """Long histories are split over a cluster of CTAs; beyond the clusters'
    shared-memory key cache the scores are re-read from L2.  The all-equal row
    puts every key of every CTA's slice on the threshold (ties across the whole
    cluster, taken in position order)."""
    rng = np.random.default_rng(5)
    L = 70000
    scores = np.stack([rng.standard_normal(L), rng.integers(0, 50, L).astype(np.float64),
                       np.zeros(L)]).astype(np.float32)
    plan = _topk_run(dev, scores, [L - 1, 60001, L - 1], 2048)
    m = re.search(r"cluster=(\d+),smem", plan)
    assert m and int(m.group(1)) > 1, plan
    L = 400000
    scores = np.stack([rng.standard_normal(L), rng.integers(0, 9, L).astype(np.float64)]).astype(np.float32)
    plan = _topk_run(dev, scores, [L - 1, 390001], 2048)
    assert "global" in plan, plan


# --------------------------------------------------------------------------- attention edges

def test_attention_minus_one_entries_and_empty(dev):
    wl = W.make("decode_b1", seed=4, ctx=[3000], q_len=2, K=512)
    run = P.Run(wl, dev)
    idx = O.topk(O.indexer_scores(wl), wl.q_pos, wl.K)
    rng = np.random.default_rng(0)
    idx[0][rng.random(wl.K) < 0.3] = -1              # holes anywhere
    idx[1][:] = -1                                   # empty selection
    g_out, g_lse, plan = run.attn(idx)
    assert "attn_tc" in plan
    o_out, o_lse = O.sparse_mla_attn(wl, idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, "bf16")
    assert np.all(g_out[1] == 0) and np.all(np.isneginf(g_lse[1]))


def test_attention_split_equals_single_slice(dev):
    wl = W.make("decode_b1", seed=6, ctx=[6000], K=2048)
    run = P.Run(wl, dev)
    idx = O.topk(O.indexer_scores(wl), wl.q_pos, wl.K)
    a_out, a_lse, plan_a = run.attn(idx, workspace=True)
    b_out, b_lse, plan_b = run.attn(idx, workspace=False)
    assert "split=1," in plan_b and "split=1," not in plan_a, (plan_a, plan_b)
    # both are checked against the oracle elsewhere; here they must agree within
    # the same tolerances (they round P against different running maxima)
    assert np.abs(a_out - b_out).max() <= 2e-2 and np.abs(a_out - b_out).mean() <= 2e-3
    assert np.abs(a_lse - b_lse).max() <= 2e-3


@pytest.mark.parametrize("name,over", [("decode_b4_long", dict(ctx=[5000], B=1, K=2048)),
                                       ("decode_b1", dict(ctx=[6000], K=2048))])
def test_attention_single_slice_many_tiles(dev, name, over):
    """No workspace: one row slice per query, so each CTA streams all of its
    2048 rows through the stage ring (every stage reused many times)."""
    wl = W.make(name, seed=8, **over)
    run = P.Run(wl, dev)
    idx = O.topk(O.indexer_scores(wl), wl.q_pos, wl.K)
    g_out, g_lse, plan = run.attn(idx, workspace=False)
    assert "split=1," in plan, plan
    o_out, o_lse = O.sparse_mla_attn(wl, idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


@pytest.mark.parametrize("workspace", [True, False])
def test_attention_running_max_jumps(dev, workspace):
    """Rows late in the selection whose logit for one head lies far (> 2**64 in
    exp2 units) above every earlier one: the kernel must rescale its TMEM
    accumulator mid-stream.  Four planted rows, one per TMEM lane quarter, each
    in the second tile of a row slice; their rope part is 16 x that head's rope
    query, so the latent (value) part stays N(0, 1)."""
    wl = W.make("decode_b1", seed=9, ctx=[6000], K=2048)
    idx = O.topk(O.indexer_scores(wl), wl.q_pos, wl.K)
    q = (wl.q[0].astype(np.uint32) << 16).view(np.float32)             # [H, 576]
    kv = wl.kv.copy()
    for rank, h in [(540, 5), (730, 37), (1500, 69), (1910, 101)]:
        pos = int(idx[0][rank])
        row = int(wl.block_table[0, pos // wl.page_size]) * wl.page_size + pos % wl.page_size
        k = (kv[row].astype(np.uint32) << 16).view(np.float32).copy()
        k[512:] = 16.0 * q[h, 512:]
        kv[row] = W._bf16_bits(torch.from_numpy(k))
    wl.kv = kv
    run = P.Run(wl, dev)
    g_out, g_lse, plan = run.attn(idx, workspace=workspace)
    assert ("split=1," in plan) != workspace, plan
    o_out, o_lse = O.sparse_mla_attn(wl, idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, "bf16")
    # the planted rows dominate their heads: the output is (nearly) their value rows
    s = o_lse[0, [5, 37, 69, 101]]
    assert np.all(s > 60.0), s


# --------------------------------------------------------------------------- device checks

def test_device_check_flags_bad_page_and_position(dev):
    import dsa_indexed_sparse_gb300 as dsa
    wl = W.make("decode_b1", seed=2, ctx=[500], K=64)
    wl.block_table = wl.block_table.copy()
    wl.block_table[0, 3] = 10 ** 6                   # page id beyond the pool
    run = P.Run(wl, dev)
    with pytest.raises(dsa.DSAError) as e:
        run.scores()
    assert e.value.status == 6 and "bad_index" in str(e.value)
    wl2 = W.make("decode_b1", seed=2, ctx=[500], K=64)
    wl2.max_ctx = 400                                # q_pos = 499 >= max_ctx
    run2 = P.Run(wl2, dev)
    with pytest.raises(dsa.DSAError) as e:
        run2.topk(O.indexer_scores(W.make("decode_b1", seed=2, ctx=[500], K=64))[:, :400])
    assert e.value.status == 6 and "bad_q_pos" in str(e.value)
    dsa.check_status()                               # cleared


# --------------------------------------------------------------------------- bounded waits

@pytest.mark.parametrize("name,over", [("decode_b1", dict(ctx=[3000], K=512)),            # bf16 rows, split
                                       ("decode_b4_long", dict(ctx=[2500], B=1, K=2048))])  # FP8 rows
def test_bounded_wait_runs_out_and_the_next_step_is_clean(dev, name, over):
    """A producer warp withholds its arrival on the first tile (testing aid):
    the issuing warp's bounded wait runs out after 2 ms, every warp unwinds,
    TMEM is released and dsa_check_status() reports DSA_ERR_TIMEOUT; the
    context stays usable and the next normal step matches the oracle."""
    import dsa_indexed_sparse_gb300 as dsa
    wl = W.make(name, seed=13, **over)
    run = P.Run(wl, dev)
    dsa.debug_withhold_arrival(True, 2_000_000)
    try:
        with pytest.raises(dsa.DSAError) as e:
            run.decode_step()
    finally:
        dsa.debug_withhold_arrival(False)
    assert e.value.status == 5 and "timeout" in str(e.value), str(e.value)
    dsa.check_status()                               # read and cleared
    with pytest.raises(dsa.DSAError) as e:
        dsa.debug_withhold_arrival(True, 10)         # bound outside [1 us, 1 s]
    assert e.value.status == 1
    o_scores = O.indexer_scores(wl)
    g_out, g_lse, g_idx, plan = run.decode_step()
    assert "attn_tc" in plan, plan
    P.check_selection(g_idx, o_scores, wl.q_pos, wl.K)
    o_out, o_lse = O.sparse_mla_attn(wl, g_idx)
    P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


@pytest.mark.parametrize("name,over,cluster", [
    ("decode_b64", dict(ctx_range=(1000, 3000), B=40, K=256), 2),        # two CTAs per query
    ("decode_b64", dict(ctx_range=(100, 5000), B=80, K=512), 1),         # one CTA per query, rows with n <= K
    ("decode_b1", dict(ctx=[20000] * 40, K=2048), 2),                    # 10000 keys per CTA
    ("decode_b4_long", dict(ctx=[9000] * 40, B=40, K=2048), 2),          # FP8 latent rows
    ("decode_b64", dict(ctx_range=(300, 3000), B=50, K=256, idx_dtype="mx_e4m3"), 2),   # MXFP8 keys
])
def test_fused_decode_plan(dev, name, over, cluster):
    """The fused plan (indexer scores kept in shared memory, Top-K selected in the
    same kernel by the CTAs of a cluster per query): its selection equals the
    chained plan's bit for bit, meets the end-to-end rule against the oracle, and
    the attention on it matches the oracle."""
    wl = W.make(name, seed=21, **over)
    run = P.Run(wl, dev)
    g_out, g_lse, g_idx, plan = run.decode_step()
    m = re.search(r"indexer_topk_fused<[a-z0-9]+>\[cluster=(\d+)", plan)
    assert m and int(m.group(1)) == cluster, plan
    np.testing.assert_array_equal(g_idx, run.chained_indices())
    ts = list(range(0, wl.T, max(1, wl.T // 8)))           # oracle rows: a spread sample
    o_scores = O.indexer_scores(wl, ts)
    P.check_selection(g_idx[ts], o_scores, wl.q_pos, wl.K, ts)
    o_out, o_lse = O.sparse_mla_attn(wl, g_idx[ts], ts)
    P.check_attn(g_out[ts], g_lse[ts], o_out, o_lse, wl.mla_dtype)


def test_fused_plan_ties_across_cluster_slices(dev):
    """Index keys made identical for every position: every score ties, so the
    selection must be positions 0..K-1 in every plan (ties to the lower
    position across the CTAs of the cluster)."""
    wl = W.make("decode_b1", seed=22, ctx=[9000] * 40, K=1000)
    wl.k_i = np.tile(wl.k_i[:1], (wl.k_i.shape[0], 1))
    wl.k_i_scale = np.full_like(wl.k_i_scale, wl.k_i_scale[0])
    run = P.Run(wl, dev)
    _, _, g_idx, plan = run.decode_step()
    assert "indexer_topk_fused<e4m3>[cluster=2" in plan, plan
    np.testing.assert_array_equal(g_idx, np.tile(np.arange(wl.K, dtype=np.int32), (wl.T, 1)))
