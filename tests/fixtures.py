"""Workloads built from the stored fixtures under tests/golden/."""
import json
import os

import numpy as np

import dsa_workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def hand_example():
    """The hand-worked example as a 1-query fp32 workload (page size 64, one page)."""
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        fx = json.load(f)
    inp = fx["inputs"]
    n = len(inp["k_I"])
    rows = 64
    k_i = np.zeros((rows, 2), np.float32); k_i[:n] = inp["k_I"]
    kv = np.zeros((rows, 3), np.float32); kv[:n] = inp["latent"]
    wl = W.Workload(
        name="hand_example", B=1, T=1, K=inp["K"], page_size=64, max_ctx=inp["q_pos"] + 1,
        q_per_seq=1, q_seq=np.zeros(1, np.int32), q_pos=np.array([inp["q_pos"]], np.int32),
        seq_lens=np.array([inp["q_pos"] + 1], np.int32), block_table=np.zeros((1, 1), np.int32),
        cache_rows=rows, idx_dtype="f32", H_I=2, D_I=2,
        q_i=np.array([inp["q_I"]], np.float32), q_i_scale=np.ones((1, 2), np.float32),
        w=np.array([inp["w"]], np.float32), k_i=k_i, k_i_scale=np.ones(rows, np.float32),
        mla_dtype="f32", H=1, d_latent=inp["d_latent"], d_rope=inp["d_rope"],
        q=np.array([[inp["q"]]], np.float32), kv=kv, row_bytes=12,
        softmax_scale=inp["softmax_scale"])
    return wl, fx["expected"]
