"""dsa_decode_step_static_ws: the decode step for callers that cannot allocate
device memory (for example a plugin inside an engine that owns all device memory
and gives plugins no allocator, or a service whose memory pool is fixed at
start-up).  Its scratch lives in a device array the library reserves, so the
call takes no workspace.

These tests call it through the C ABI and compare it with dsa_decode_step (the
entry point that takes a caller-provided workspace) within the parity
tolerances, on two calls in a row, since every call reuses the same array; one
case is also held against the CPU oracle directly, and the device's free memory
and torch's allocator are checked to be untouched by a call.  The file is named
so that pytest collects it after every other test."""
import numpy as np
import pytest
import torch

import dsa_indexed_sparse_gb300 as dsa
import dsa_workloads as W
from oracle import dsa_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu


def _static_call(run, wl, dev):
    out = torch.full((wl.T, wl.H, wl.d_v), float("nan"), dtype=run.out_dtype, device=dev)
    lse = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=dev)
    sel = torch.full((wl.T, wl.K), -7, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    dsa.decode_step_static_ws(run.seq, run.idxr, run.mla, wl.K, out, lse=lse, idx_out=sel)
    plan = dsa.last_plan()
    dsa.check_status()
    free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    return out, lse, sel, plan, (free0, alloc0, free1, alloc1)


@pytest.mark.parametrize("name,over,vs_oracle", [
    ("decode_b1", dict(ctx=[5000], K=2048), True),                               # split rows: partials in scratch
    ("decode_b64", dict(ctx_range=(300, 3000), B=6, K=256), False),              # shuffled pages, one slice per query
    ("decode_b4_long", dict(ctx=[2500, 4100], B=2, K=2048), False),              # FP8 latent rows
])
def test_static_workspace_step_matches_workspace_step(dev, name, over, vs_oracle):
    wl = W.make(name, seed=11, **over)
    run = P.Run(wl, dev)
    ref_out, ref_lse, ref_idx, ref_plan = run.decode_step()       # caller-provided workspace
    for call in range(2):                                         # the array keeps the last call's data
        out, lse, sel, plan, mem = _static_call(run, wl, dev)
        assert plan == ref_plan
        if call == 1:   # after a first call (which may load the module's code): nothing allocated
            free0, alloc0, free1, alloc1 = mem
            assert alloc1 == alloc0, "torch's allocator grew during the call"
            assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
        g_idx = sel.cpu().numpy()
        assert P.as_sets(g_idx) == P.as_sets(ref_idx), f"call {call}: selection differs"
        g_out, g_lse = out.float().cpu().numpy(), lse.cpu().numpy()
        P.check_attn(g_out, g_lse, ref_out, ref_lse, wl.mla_dtype)
        if vs_oracle:
            P.check_selection(g_idx, O.indexer_scores(wl), wl.q_pos, wl.K)
            o_out, o_lse = O.sparse_mla_attn(wl, g_idx)
            P.check_attn(g_out, g_lse, o_out, o_lse, wl.mla_dtype)


def test_static_workspace_rejects_steps_larger_than_the_array(dev):
    wl = W.make("decode_b1", seed=12, ctx=[600], K=64)
    run = P.Run(wl, dev)
    # a context bound whose score rows alone need more than the reserved array
    big_ctx = (dsa.STATIC_WORKSPACE_BYTES // 4) + 4096
    stride = (big_ctx + 63) // 64
    bt = torch.zeros((1, stride), dtype=torch.int32, device=dev)
    seq = dsa.Seq(q_seq=run.seq.q_seq, q_pos=run.seq.q_pos, block_table=bt, max_ctx=big_ctx,
                  cache_rows=run.seq.cache_rows, page_size=64, q_per_seq=1)
    assert dsa.decode_workspace_size(seq, run.idxr, run.mla, wl.K) > dsa.STATIC_WORKSPACE_BYTES
    out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_step_static_ws(seq, run.idxr, run.mla, wl.K, out)
    assert e.value.status == 3 and "static workspace too small" in str(e.value)


def test_static_workspace_gives_the_same_status_as_the_workspace_step(dev):
    """A descriptor both calls reject gets the same status from both (K = 0 has
    no kernel: DSA_ERR_UNSUPPORTED)."""
    wl = W.make("decode_b1", seed=12, ctx=[600], K=64)
    run = P.Run(wl, dev)
    out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(dsa.DSAError) as e1:
        dsa.decode_step(run.seq, run.idxr, run.mla, 0, out, ws)
    with pytest.raises(dsa.DSAError) as e2:
        dsa.decode_step_static_ws(run.seq, run.idxr, run.mla, 0, out)
    assert e1.value.status == e2.value.status == 2, (str(e1.value), str(e2.value))
