"""GPU parity of MiniMax block selection against the oracle: bit-exact block
indices (the page's sequential f32 dot), through the C ABI."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import block_select as obs
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "block_select_examples.json")))


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _gpu_select(B, q, k, pos, bs, top, init, local, width=None):
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    Q, n_kv, D = q.shape
    L = k.shape[0]
    cfg = B.block_sparse_config(bs, top, init, local)
    W = width or max(top, init + local, 1)
    out = torch.empty((Q, n_kv, W), dtype=torch.int32, device="cuda")
    cnt = torch.empty((Q, n_kv), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(1, B.block_select_workspace_size(Q, n_kv, max(L, 1), cfg)), dtype=torch.uint8, device="cuda")
    B.block_select(torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda() if L else torch.empty((0, D), device="cuda"),
                   torch.from_numpy(np.asarray(pos, dtype=np.int32)).cuda(), cfg, out, cnt, ws)
    o, c = out.cpu().numpy(), cnt.cpu().numpy()
    res = []
    for i in range(Q):
        row = []
        for h in range(n_kv):
            sel = o[i, h, :c[i, h]].tolist()
            assert (o[i, h, c[i, h]:] == -1).all()
            row.append(sel)
        res.append(row)
    return res


def _keys(case):
    n = case["n"]
    if "all" in case:
        return np.tile(np.array(case["all"], dtype=np.float32), (n, 1))
    if "set" in case:
        k = np.zeros((n, 2), dtype=np.float32)
        for p, v in case["set"].items():
            k[int(p)] = v
        return k
    k = np.tile(np.array([0.0, 0.01], dtype=np.float32), (n, 1))
    for p in case["hot"]:
        k[p] = [1.0, 0.0]
    return k


def test_printed_cases_on_gpu(B):
    for c in GOLD["cases"] + [GOLD["per_head"]]:
        q = np.array(c["q"], dtype=np.float32)[None]
        sel = _gpu_select(B, q, _keys(c), [c["pos"]], *c["cfg"])[0]
        ref = obs.block_sparse_select(q[0], _keys(c), c["pos"], *c["cfg"])
        assert sel == ref, c["name"]
        if "expected" in c:
            assert sel == c["expected"], c["name"]
    c = GOLD["never_empty"]
    for pos in c["positions"]:
        sel = _gpu_select(B, np.array(c["q"], np.float32)[None], _keys(c), [pos], *c["cfg"])[0]
        assert sel[0]


@pytest.mark.parametrize("seed,Q,n_kv,D,L,bs,top,init,local", [
    (1, 20, 3, 128, 3000, 128, 8, 1, 2), (2, 17, 2, 128, 1000, 16, 12, 2, 3), (3, 9, 4, 64, 777, 32, 5, 0, 0),
    (4, 12, 2, 5, 300, 7, 6, 1, 1), (5, 30, 1, 128, 2048, 128, 32, 1, 2), (6, 8, 2, 128, 500, 1, 40, 3, 3)])
def test_random_against_oracle(B, seed, Q, n_kv, D, L, bs, top, init, local):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((Q, n_kv, D)).astype(np.float32)
    k = rng.standard_normal((L, D)).astype(np.float32)
    k[rng.integers(0, L, L // 10)] = k[0]           # exact ties between blocks
    pos = rng.integers(0, L + 200, Q).astype(np.int32)
    pos[0] = 0
    got = _gpu_select(B, q, k, pos, bs, top, init, local)
    for i in range(Q):
        assert got[i] == obs.block_sparse_select(q[i], k, int(pos[i]), bs, top, init, local), i
    assert B.device_error() == 0


def test_minimax_workload_every_selection(B):
    """1024 queries x 8 KV heads over 131072 keys (block 128, top 32, init 1,
    local 2): every (query, KV head) selection bit for bit against the oracle
    (run on every host core)."""
    from helpers import block_select_task, oracle_pool
    bp = wl.block_select()
    got = _gpu_select(B, bp.index_q, bp.index_k, bp.query_pos, bp.block_size, bp.top_blocks, bp.init_blocks,
                      bp.local_blocks)
    pool = oracle_pool(bp)
    try:
        # the late (long) queries first so the pool stays busy to the end
        refs = pool.map(block_select_task, list(range(1023, -1, -1)), chunksize=1)
    finally:
        pool.close()
        pool.join()
    assert len(refs) == 1024
    for i, ref in refs:
        assert got[i] == ref, i
    for i in range(1024):
        for h in range(8):
            assert len(got[i][h]) == min(32, i + 1)
    assert B.device_error() == 0
