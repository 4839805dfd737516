"""Shared helpers of the GPU parity tests: run each stage through the C ABI and
compare with the CPU oracle using the tolerances of the method statement:

* indexer scores: within 1e-3 relative in fp32.  Read here as
  |gpu - oracle| <= 1e-3 * max(|oracle|, 1e-3 * rowmax|oracle|) per causal entry
  (the floor keeps the test meaningful for scores that cancel to ~0, since the
  head weights can be negative);
* Top-K on the oracle's own scores: bit-exact index sets;
* end to end: every selected index has an oracle score >= the oracle's K-th
  score - 1e-3 * max|score| of that query, the selection has min(K, n) distinct
  causal positions;
* attention: max-abs <= 2e-2 and mean-abs <= 2e-3 against the fp64 oracle for
  bf16 rows (3e-2 / 4e-3 for the FP8 latent cache, oracle on dequantised
  values); lse within 2e-3 absolute (fp32 online softmax with bf16 P).
"""
import numpy as np
import torch

import dsa_indexed_sparse_gb300 as dsa
import dsa_workloads as W
from oracle import dsa_oracle as O

ATTN_TOL = {"bf16": (2e-2, 2e-3), "e4m3": (3e-2, 4e-3), "e4m3_t128": (3e-2, 4e-3), "f32": (2e-5, 2e-6)}
LSE_TOL = {"bf16": 2e-3, "e4m3": 2e-3, "e4m3_t128": 2e-3, "f32": 1e-5}


class Run:
    """A workload on the device plus output buffers."""

    def __init__(self, wl, dev):
        self.wl, self.dev = wl, dev
        d = W.device_tensors(wl, dev)
        self.seq = dsa.Seq(**d["seq"])
        self.idxr = dsa.Indexer(**d["indexer"])
        self.mla = dsa.Mla(**d["mla"])
        self.ld = (wl.max_ctx + 3) // 4 * 4
        self.out_dtype = torch.float32 if wl.mla_dtype == "f32" else torch.bfloat16

    def scores(self):
        s = torch.full((self.wl.T, self.ld), float("nan"), dtype=torch.float32, device=self.dev)
        dsa.indexer_scores(self.seq, self.idxr, s)
        plan = dsa.last_plan()
        dsa.check_status()
        return s.cpu().numpy(), plan

    def topk(self, scores_np, K=None):
        K = K or self.wl.K
        pad = np.full((scores_np.shape[0], self.ld), -np.inf, dtype=np.float32)
        pad[:, :min(self.ld, scores_np.shape[1])] = scores_np[:, :self.ld]
        s = torch.from_numpy(pad).to(self.dev)
        idx = torch.full((self.wl.T, K), -7, dtype=torch.int32, device=self.dev)
        dsa.topk(self.seq, s, K, idx)
        plan = dsa.last_plan()
        dsa.check_status()
        return idx.cpu().numpy(), plan

    def attn(self, idx_np, K=None, workspace=True):
        wl = self.wl
        K = K or idx_np.shape[1]
        idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).to(self.dev)
        out = torch.full((wl.T, wl.H, wl.d_v), float("nan"), dtype=self.out_dtype, device=self.dev)
        lse = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=self.dev)
        ws = None
        if workspace:
            n = dsa.sparse_mla_attn_workspace_size(self.seq, self.mla, K)
            ws = torch.empty(max(n, 16), dtype=torch.uint8, device=self.dev)
        dsa.sparse_mla_attn(self.seq, self.mla, idx, K, out, lse=lse, workspace=ws)
        plan = dsa.last_plan()
        dsa.check_status()
        return out.float().cpu().numpy(), lse.cpu().numpy(), plan

    def chained_indices(self):
        """The chained plan's selection made from the separate calls: the GPU's
        own scores (dsa_indexer_scores), then dsa_topk on them."""
        s = torch.full((self.wl.T, self.ld), float("-inf"), dtype=torch.float32, device=self.dev)
        dsa.indexer_scores(self.seq, self.idxr, s)
        idx = torch.full((self.wl.T, self.wl.K), -7, dtype=torch.int32, device=self.dev)
        dsa.topk(self.seq, s, self.wl.K, idx)
        dsa.check_status()
        return idx.cpu().numpy()

    def decode_step(self):
        wl = self.wl
        out = torch.full((wl.T, wl.H, wl.d_v), float("nan"), dtype=self.out_dtype, device=self.dev)
        lse = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=self.dev)
        sel = torch.full((wl.T, wl.K), -7, dtype=torch.int32, device=self.dev)
        n = dsa.decode_workspace_size(self.seq, self.idxr, self.mla, wl.K)
        ws = torch.empty(n, dtype=torch.uint8, device=self.dev)
        dsa.decode_step(self.seq, self.idxr, self.mla, wl.K, out, ws, lse=lse, idx_out=sel)
        plan = dsa.last_plan()
        dsa.check_status()
        return out.float().cpu().numpy(), lse.cpu().numpy(), sel.cpu().numpy(), plan


def check_scores(g, o, q_pos, ts=None):
    """g, o: [len(ts), L] score rows; only causal entries are compared."""
    ts = range(g.shape[0]) if ts is None else ts
    worst = 0.0
    for i, t in enumerate(ts):
        n = int(q_pos[t]) + 1
        gr, orow = g[i, :n].astype(np.float64), o[i, :n].astype(np.float64)
        assert np.all(np.isfinite(gr)), f"non-finite GPU score in row {t}"
        rowmax = np.abs(orow).max()
        bound = 1e-3 * np.maximum(np.abs(orow), 1e-3 * rowmax)
        err = np.abs(gr - orow)
        bad = np.nonzero(err > bound)[0]
        assert bad.size == 0, f"row {t}: {bad.size} scores off, e.g. s={bad[0]} gpu={gr[bad[0]]} oracle={orow[bad[0]]}"
        worst = max(worst, float((err / np.maximum(bound, 1e-30)).max()) * 1e-3)
    return worst


def as_sets(idx):
    return [sorted(int(x) for x in r if x >= 0) for r in idx]


def check_topk_exact(g_idx, o_idx, q_pos, K):
    for t in range(g_idx.shape[0]):
        n = int(q_pos[t]) + 1
        m = min(K, n)
        valid = g_idx[t][:m]
        assert np.all(g_idx[t][m:] == -1), f"row {t}: padding is not -1"
        assert sorted(valid.tolist()) == as_sets(o_idx[t:t + 1])[0], f"row {t}: index set differs"
        assert np.all(np.diff(valid) > 0), f"row {t}: not ascending"


def check_selection(g_idx, o_scores, q_pos, K, ts=None):
    ts = range(g_idx.shape[0]) if ts is None else ts
    for i, t in enumerate(ts):
        n = int(q_pos[t]) + 1
        row = o_scores[i, :n].astype(np.float64)
        chosen = g_idx[i][g_idx[i] >= 0]
        assert len(chosen) == min(K, n) and len(set(chosen.tolist())) == len(chosen)
        assert chosen.max() <= q_pos[t]
        kth = np.sort(row)[::-1][min(K, n) - 1]
        assert np.all(row[chosen] >= kth - 1e-3 * np.abs(row).max()), f"row {t}: selection below the K-th score"


def step_plan_ok(plan):
    """The decode step ran the tensor-core kernels: the fused indexer + Top-K
    kernel, or the chained indexer and Top-K kernels; then the attention."""
    fused = "indexer_topk_fused" in plan
    chained = "indexer_tc" in plan and "topk_radix" in plan
    return (fused or chained) and "attn_tc" in plan


def check_attn(g_out, g_lse, o_out, o_lse, dtype):
    mx, mean = ATTN_TOL[dtype]
    err = np.abs(g_out - o_out)
    assert np.all(np.isfinite(g_out)), "non-finite attention output"
    assert err.max() <= mx and err.mean() <= mean, f"attention error max {err.max():.3g} mean {err.mean():.3g}"
    fin = np.isfinite(o_lse)
    assert np.array_equal(fin, np.isfinite(g_lse)), "lse finiteness differs"
    lerr = np.abs(g_lse[fin] - o_lse[fin]).max() if fin.any() else 0.0
    assert lerr <= LSE_TOL[dtype], f"lse error {lerr:.3g}"
    return float(err.max()), float(err.mean())
