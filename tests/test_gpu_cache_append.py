"""GPU parity of the cache writers (the prolog side of a step) against the
oracle: the new tokens' index keys (e4m3 codes + per-token fp32 scale) and
latent rows (bf16 / fp32 copies, 656-byte FP8 rows) must be bit-exact, every
other cache row untouched; then the indexer scoring the appended cache agrees
with the oracle scoring the oracle's cache."""
import dataclasses

import numpy as np
import pytest
import torch

import dsa_indexed_sparse_gb300 as dsa
import dsa_workloads as W
from oracle import dsa_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu


def _layout(seed):
    # 3 sequences with shuffled pages; 4 new tokens each at their last positions
    return W.make("decode_b64", seed=seed, ctx_range=(200, 900), B=3, q_len=4, K=64)


def _seq(wl, dev):
    return dsa.Seq(**W.device_tensors(wl, dev)["seq"])


def _new_keys(rng, T, D):
    k = rng.normal(0, 1, (T, D)).astype(np.float32) * rng.uniform(0.01, 50, (T, 1)).astype(np.float32)
    k[1] = 0.0                                  # an all-zero row: scale 1, codes 0
    k[2, :7] = [448.0, -1e-6, 3e-3, -2.5, 0.0, -0.0, 1e4]
    return k


@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_index_cache_append_bit_exact(dev, src):
    wl = _layout(31)
    rng = np.random.default_rng(32)
    D = wl.D_I
    k_new = _new_keys(rng, wl.T, D)
    t_new = torch.from_numpy(k_new)
    if src == "bf16":
        t_new = t_new.to(torch.bfloat16)
        k_new = t_new.float().numpy()            # what the kernel sees
    kc0 = rng.integers(0, 256, (wl.cache_rows, D)).astype(np.uint8)
    ks0 = rng.normal(0, 1, wl.cache_rows).astype(np.float32)
    kc = torch.from_numpy(kc0.copy()).to(dev)
    ks = torch.from_numpy(ks0.copy()).to(dev)
    dsa.index_cache_append(_seq(wl, dev), t_new.to(dev), kc, ks)
    assert dsa.last_plan().startswith("index_append")
    dsa.check_status()
    o_kc, o_ks = O.index_cache_append(wl.block_table, wl.page_size, wl.q_seq, wl.q_pos, k_new, kc0, ks0)
    assert np.array_equal(kc.cpu().numpy(), o_kc)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), o_ks.view(np.uint32))


def test_latent_cache_append_bf16_and_fp8_rows(dev):
    wl = _layout(33)
    rng = np.random.default_rng(34)
    x = rng.normal(0, 1, (wl.T, 576)).astype(np.float32) * rng.uniform(0.01, 30, (wl.T, 1)).astype(np.float32)
    x[0, :512] = 0.0                             # latent part all zero, rope not
    t_new = torch.from_numpy(x).to(torch.bfloat16)
    bits = t_new.view(torch.int16).numpy().view(np.uint16)
    q = torch.zeros((1, 128, 576), dtype=torch.bfloat16, device=dev)
    for fp8 in (False, True):
        row_bytes = 656 if fp8 else 1152
        cache0 = rng.integers(0, 256, (wl.cache_rows, row_bytes)).astype(np.uint8)
        if fp8:
            cache = torch.from_numpy(cache0.copy()).to(dev)
            mla = dsa.Mla(q=q, kv_cache=cache, d_latent=512, d_rope=64, softmax_scale=1.0, dtype=dsa.DSA_E4M3)
        else:
            cache = torch.from_numpy(cache0.copy()).to(dev).view(torch.bfloat16)
            mla = dsa.Mla(q=q, kv_cache=cache, d_latent=512, d_rope=64, softmax_scale=1.0)
        dsa.latent_cache_append(_seq(wl, dev), mla, t_new.to(dev))
        assert dsa.last_plan() == ("latent_append<fp8_row>" if fp8 else "latent_append<bf16>")
        dsa.check_status()
        got = cache.view(torch.uint8).cpu().numpy() if not fp8 else cache.cpu().numpy()
        want = O.latent_cache_append(wl.block_table, wl.page_size, wl.q_seq, wl.q_pos, bits, cache0, fp8_rows=fp8)
        assert np.array_equal(got, want), f"fp8={fp8}"


def test_latent_cache_append_f32_rows(dev):
    wl = _layout(35)
    rng = np.random.default_rng(36)
    x = rng.normal(0, 1, (wl.T, 80)).astype(np.float32)
    cache0 = rng.normal(0, 1, (wl.cache_rows, 80)).astype(np.float32)
    cache = torch.from_numpy(cache0.copy()).to(dev)
    q = torch.zeros((1, 4, 80), dtype=torch.float32, device=dev)
    mla = dsa.Mla(q=q, kv_cache=cache, d_latent=64, d_rope=16, softmax_scale=1.0)
    dsa.latent_cache_append(_seq(wl, dev), mla, torch.from_numpy(x).to(dev))
    dsa.check_status()
    want = cache0.copy()
    for t in range(wl.T):
        row = O.physical_rows(wl.block_table[wl.q_seq[t]], wl.page_size, np.array([wl.q_pos[t]]))[0]
        want[row] = x[t]
    assert np.array_equal(cache.cpu().numpy(), want)


def test_append_then_score_matches_oracle(dev):
    """The keys the writer appends are the keys the indexer then scores."""
    wl = _layout(37)
    rng = np.random.default_rng(38)
    k_new = _new_keys(rng, wl.T, wl.D_I)
    d = W.device_tensors(wl, dev)
    seq, idxr = dsa.Seq(**d["seq"]), dsa.Indexer(**d["indexer"])
    dsa.index_cache_append(seq, torch.from_numpy(k_new).to(dev), idxr.k_cache, idxr.k_scale)
    ld = (wl.max_ctx + 3) // 4 * 4
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=dev)
    dsa.indexer_scores(seq, idxr, scores)
    dsa.check_status()
    o_kc, o_ks = O.index_cache_append(wl.block_table, wl.page_size, wl.q_seq, wl.q_pos, k_new, wl.k_i, wl.k_i_scale)
    o_scores = O.indexer_scores(dataclasses.replace(wl, k_i=o_kc, k_i_scale=o_ks))
    P.check_scores(scores.cpu().numpy(), o_scores, wl.q_pos)


def test_append_flags_bad_position(dev):
    wl = _layout(39)
    d = W.device_tensors(wl, dev)
    d["seq"]["q_pos"] = d["seq"]["q_pos"].clone()
    d["seq"]["q_pos"][2] = wl.max_ctx            # beyond max_ctx: skipped and flagged
    seq = dsa.Seq(**d["seq"])
    kc = torch.zeros((wl.cache_rows, wl.D_I), dtype=torch.uint8, device=dev)
    ks = torch.zeros(wl.cache_rows, dtype=torch.float32, device=dev)
    dsa.index_cache_append(seq, torch.ones((wl.T, wl.D_I), device=dev), kc, ks)
    with pytest.raises(dsa.DSAError) as e:
        dsa.check_status()
    assert e.value.status == 6 and "bad_q_pos" in str(e.value)
    # the other tokens were written
    assert int((ks != 0).sum()) == wl.T - 1


@pytest.mark.parametrize("src", ["f32", "bf16"])
def test_index_cache_append_mx_bit_exact(dev, src):
    wl = _layout(41)
    rng = np.random.default_rng(42)
    D = wl.D_I
    k_new = (rng.normal(0, 1, (wl.T, D)) * np.repeat(np.exp2(rng.integers(-6, 6, (wl.T, D // 32))), 32, axis=1)
             ).astype(np.float32)
    k_new[1] = 0.0                               # all-zero blocks: exponent byte 0, codes 0
    k_new[2, :32] = 0.0
    k_new[3, 32:39] = [448.0, -1e-6, 3e-3, -2.5, 0.0, -0.0, 1e4]
    t_new = torch.from_numpy(k_new)
    if src == "bf16":
        t_new = t_new.to(torch.bfloat16)
        k_new = t_new.float().numpy()
    kc0 = rng.integers(0, 256, (wl.cache_rows, D)).astype(np.uint8)
    ke0 = rng.integers(0, 256, (wl.cache_rows, D // 32)).astype(np.uint8)
    kc = torch.from_numpy(kc0.copy()).to(dev)
    ke = torch.from_numpy(ke0.copy()).to(dev)
    dsa.index_cache_append(_seq(wl, dev), t_new.to(dev), kc, ke, mx=True)
    assert dsa.last_plan().startswith("index_append_mx")
    dsa.check_status()
    o_kc, o_ke = O.index_cache_append(wl.block_table, wl.page_size, wl.q_seq, wl.q_pos, k_new, kc0, ke0, mx=True)
    assert np.array_equal(kc.cpu().numpy(), o_kc)
    assert np.array_equal(ke.cpu().numpy(), o_ke)


def test_latent_cache_append_tile128_rows(dev):
    wl = _layout(43)
    rng = np.random.default_rng(44)
    x = rng.normal(0, 1, (wl.T, 576)).astype(np.float32)
    x[:, :512] *= np.repeat(np.exp2(rng.integers(-3, 3, (wl.T, 4))), 128, axis=1)
    x[0, 128:256] = 0.0                          # one all-zero tile
    t_new = torch.from_numpy(x).to(torch.bfloat16)
    bits = t_new.view(torch.int16).numpy().view(np.uint16)
    q = torch.zeros((1, 128, 576), dtype=torch.bfloat16, device=dev)
    cache0 = rng.integers(0, 256, (wl.cache_rows, 656)).astype(np.uint8)
    cache = torch.from_numpy(cache0.copy()).to(dev)
    mla = dsa.Mla(q=q, kv_cache=cache, d_latent=512, d_rope=64, softmax_scale=1.0, dtype=dsa.DSA_E4M3_T128)
    dsa.latent_cache_append(_seq(wl, dev), mla, t_new.to(dev))
    assert dsa.last_plan() == "latent_append<fp8_tile128>"
    dsa.check_status()
    want = O.latent_cache_append(wl.block_table, wl.page_size, wl.q_seq, wl.q_pos, bits, cache0, fp8_rows=True,
                                 tile128=True)
    assert np.array_equal(cache.cpu().numpy(), want)
