"""Tensor-core score path: parity with the fp64 oracle on every (H, key
layout, dtype) instantiation, bit-identity of a (query, key) score across
launch shapes, and rows with a bad extent."""
import numpy as np
import pytest
import torch

from helpers import EPS, check_scores
from oracle import dsa as odsa
from sparse_attention_indexer_idx_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_idx_gb300 import binding
    binding.lib()
    return binding


def _score(B, p, M, ld):
    out = torch.full((M, ld), float("nan"), dtype=torch.float32, device="cuda")
    B.idx_score(p, out, ld)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check_all(B, wp):
    p = B.problem_to_device(wp)
    got = _score(B, p, wp.M, max(1, p.max_key_len))
    assert B.device_error() == 0
    for m in range(wp.M):
        L = int(wp.key_len[m])
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_scores(got[m, :L], s_ref, a_ref, EPS[wp.dtype])
        assert np.isnan(got[m, L:]).all(), "wrote beyond key_len"


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_per_row_bf16(B, H):
    _check_all(B, wl.decode_bf16(seed=H, M=5, H=H, D=128, L=700, K=16))


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_shared_bf16(B, H):
    _check_all(B, wl.prefill_bf16(seed=H, n_queries=37, H=H, D=128, L=900, K=16))


@pytest.mark.parametrize("H", [32, 64])
def test_per_row_fp8(B, H):
    _check_all(B, wl.ragged_fp8(seed=H, M=6, H=H, D=128, L_min=1, L_max=1300, K=16))


def test_shared_fp8(B):
    wp = wl.ragged_fp8(seed=3, M=9, H=64, D=128, L_min=500, L_max=900, K=16)
    # one shared key sequence: rows read keys from 0 with causal lengths
    wp.key_off = None
    wp.key_len = np.arange(wp.n_keys - wp.M, wp.n_keys, dtype=np.int32)[:wp.M] // 3 + 1
    _check_all(B, wp)


def test_score_bits_do_not_depend_on_the_launch_shape(B):
    """The same (query, key) pair scored inside a 4-query N=256 tile (shared
    keys) and inside a 1-query N=64 tile (per-row keys, key_off = 0) must give
    identical bits: the pruned and unpruned paths rely on it."""
    wp = wl.prefill_bf16(seed=5, n_queries=12, H=64, D=128, L=1000, K=16)
    p = B.problem_to_device(wp)
    a = _score(B, p, wp.M, 1000)
    p.key_off = torch.zeros(wp.M, dtype=torch.int64, device="cuda")
    b = _score(B, p, wp.M, 1000)
    for m in range(wp.M):
        L = int(wp.key_len[m])
        assert np.array_equal(a[m, :L].view(np.uint32), b[m, :L].view(np.uint32)), m
    # and inside a tile whose keys start at a different offset (keys shifted by 37 rows)
    keys2 = torch.cat([torch.zeros((37, 128), dtype=p.keys.dtype, device="cuda"), p.keys])
    p2 = B.Problem(p.q, p.w, keys2, p.key_len, p.max_key_len, torch.full((wp.M,), 37, dtype=torch.int64, device="cuda"))
    c = _score(B, p2, wp.M, 1000)
    for m in range(wp.M):
        L = int(wp.key_len[m])
        assert np.array_equal(a[m, :L].view(np.uint32), c[m, :L].view(np.uint32)), m


def test_bad_rows_are_empty_and_reported(B):
    wp = wl.decode_bf16(seed=7, M=4, H=32, D=128, L=300, K=16)
    p = B.problem_to_device(wp)
    kl = p.key_len.clone()
    kl[1] = 301                       # above max_key_len
    ko = p.key_off.clone()
    ko[2] = wp.n_keys - 100           # runs past the key buffer
    p.key_len, p.key_off = kl, ko
    got = _score(B, p, wp.M, 300)
    assert B.device_error() & B.DEVERR_BAD_ROW
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all()
    for m in (0, 3):
        s_ref, a_ref = odsa.row_scores(wp, m)
        check_scores(got[m], s_ref, a_ref, EPS["bf16"])
