"""Seeded synthetic inputs for the indexer hot path.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests.  It holds no arithmetic of the method itself: it only draws
random numbers, rounds them once to the stored dtype (bf16 or FP8 e4m3 with a
per-token scale) and lays them out the way the C-ABI expects.  Both sides
therefore see the very same bytes.

Storage formats:
  * bf16 values are kept as ``uint16`` bit patterns (numpy has no bf16).
  * FP8 e4m3 (the ``fn`` variant: no infinities, max 448) is kept as ``uint8``.
  * Keys are row-major ``[n_keys, D]``; queries ``[M, H, D]``; weights
    ``[M, H]`` float32; ``key_off`` int64 ``[M]`` (or ``None`` = every row reads
    the shared key sequence from key 0); ``key_len`` int32 ``[M]``.

Workloads (names follow the shapes on the pages: H32/H64, D128, K2048,
128-token blocks):
  tiny_fp32      8 rows, H4, D16, L512, K32, fp32, then witnesses S=4
  decode_bf16    64 rows each with its own 32768 bf16 keys, H32, K2048, S=16
  prefill_bf16   4096 causal queries over 65536 shared bf16 keys, H64, K2048
  block_select   MiniMax block select: 1024 queries, 8 KV heads, L131072
  ragged_fp8     128 rows, L_r ~ U{4096..131072}, FP8 keys + scale, H64, S=32
Every generator takes size overrides so the tests can run scaled-down
instances with the same value distributions.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_table() -> np.ndarray:
    t = np.zeros(256, dtype=np.float64)
    for b in range(256):
        s = -1.0 if b & 0x80 else 1.0
        e = (b >> 3) & 0xF
        m = b & 0x7
        if e == 0xF and m == 0x7:
            t[b] = np.nan
        elif e == 0:
            t[b] = s * m * 2.0 ** -9
        else:
            t[b] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


E4M3_VALUES = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact decode of FP8 e4m3 bit patterns."""
    return E4M3_VALUES[np.asarray(b, dtype=np.uint8)].astype(np.float32)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Encode to FP8 e4m3 (round to nearest even, saturate to +-448)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(a)                      # a = f * 2**ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)               # unbiased exponent, subnormals at -6
    quantum = np.ldexp(1.0, e - 3)
    y = np.rint(a / quantum) * quantum       # exact scaling, ties to even
    y = np.minimum(y, E4M3_MAX)
    _, ey = np.frexp(y)
    ey = ey - 1
    normal = y >= 2.0 ** -6
    E = np.where(normal, ey + 7, 0)
    mant = np.where(normal, y / np.ldexp(1.0, np.where(normal, ey, 0)) * 8.0 - 8.0, y / 2.0 ** -9)
    bits = (E.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    bits = np.where(y == 0, 0, bits)
    bits = bits | np.where(sign, 0x80, 0)
    return bits.astype(np.uint8)


def _bulk_bf16(x: np.ndarray) -> np.ndarray:
    """f32_to_bf16_bits for large arrays (torch's cast: same round-to-nearest-even,
    checked equal by the generator tests)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bulk_e4m3(x: np.ndarray) -> np.ndarray:
    """f32_to_e4m3_bits for large arrays with |x| <= 448 (torch's cast, checked
    equal by the generator tests)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ----------------------------------------------------------------------------
# problem containers
# ----------------------------------------------------------------------------


@dataclass
class IndexerProblem:
    """One batch of indexer rows.

    dtype is "f32", "bf16" or "fp8".  For "bf16" q and keys hold uint16 bit
    patterns; for "fp8" keys hold uint8 e4m3 bits and key_scale the per-token
    float32 scale while q is bf16; for "f32" both are float32.
    """

    name: str
    dtype: str
    q: np.ndarray                  # [M, H, D]
    w: np.ndarray                  # [M, H] float32
    keys: np.ndarray               # [n_keys, D]
    key_len: np.ndarray            # [M] int32
    key_off: Optional[np.ndarray]  # [M] int64, or None for one shared sequence
    K: int
    key_scale: Optional[np.ndarray] = None  # [n_keys] float32 (fp8 only)
    extras: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.q.shape[0])

    @property
    def H(self) -> int:
        return int(self.q.shape[1])

    @property
    def D(self) -> int:
        return int(self.q.shape[2])

    @property
    def n_keys(self) -> int:
        return int(self.keys.shape[0])

    def q_f32(self) -> np.ndarray:
        return self.q if self.dtype == "f32" else bf16_bits_to_f32(self.q)

    def keys_f32(self, start: int = 0, stop: Optional[int] = None) -> np.ndarray:
        """Stored keys [start, stop) widened exactly to float32 (codes only for FP8)."""
        k = self.keys[start:stop]
        if self.dtype == "f32":
            return k
        if self.dtype == "bf16":
            return bf16_bits_to_f32(k)
        return e4m3_bits_to_f32(k)

    def row_offset(self, m: int) -> int:
        return 0 if self.key_off is None else int(self.key_off[m])

    def pairs(self) -> int:
        return int(np.asarray(self.key_len, dtype=np.int64).sum())


@dataclass
class BlockSelectProblem:
    name: str
    index_q: np.ndarray     # [Q, n_kv, D] float32
    index_k: np.ndarray     # [L, D] float32
    query_pos: np.ndarray   # [Q] int32
    block_size: int
    top_blocks: int
    init_blocks: int
    local_blocks: int


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def tiny_fp32(seed: int = 0, M: int = 8, H: int = 4, D: int = 16, L: int = 512,
              K: int = 32, S: int = 4) -> IndexerProblem:
    """8 query rows, H4, D16, 512 shared keys, fp32; witnesses S=4 after top-K."""
    rng = np.random.default_rng(seed)
    q = _normal(rng, (M, H, D))
    keys = _normal(rng, (L, D))
    w = rng.uniform(-1.0, 1.0, (M, H)).astype(np.float32)
    key_len = np.full(M, L, dtype=np.int32)
    return IndexerProblem("tiny_fp32", "f32", q, w, keys, key_len, None, K,
                          extras=dict(S=S, keep=K - S, max_repl=S))


def decode_bf16(seed: int = 2, M: int = 64, H: int = 32, D: int = 128, L: int = 32768,
                K: int = 2048, S: int = 16, pad_frac: float = 0.05) -> IndexerProblem:
    """Decode batch: every row owns L bf16 keys; w ~ N(0, 1/H) (variance 1/H)."""
    rng = np.random.default_rng(seed)
    q = _bulk_bf16(_normal(rng, (M, H, D)))
    keys = np.empty((M * L, D), dtype=np.uint16)
    chunk = max(1, (1 << 22) // D)
    for s in range(0, M * L, chunk):
        e = min(M * L, s + chunk)
        keys[s:e] = _bulk_bf16(_normal(rng, (e - s, D)))
    w = _normal(rng, (M, H), std=float(np.sqrt(1.0 / H)))
    key_len = np.full(M, L, dtype=np.int32)
    key_off = (np.arange(M, dtype=np.int64) * L)
    pad_mask = rng.random((M, K)) < pad_frac
    return IndexerProblem("decode_bf16", "bf16", q, w, keys, key_len, key_off, K,
                          extras=dict(S=S, keep=K - S, max_repl=S, pad_mask=pad_mask))


def prefill_bf16(seed: int = 3, n_queries: int = 4096, H: int = 64, D: int = 128,
                 L: int = 65536, K: int = 2048, n_centres: int = 64, sigma: float = 0.3,
                 n_seed: int = 12288, R: int = 16, q_noise: Optional[float] = None,
                 q_run: int = 1, positive_w: bool = False) -> IndexerProblem:
    """Causal prefill: queries at positions L-n..L-1 over one shared key sequence.

    Keys: with probability 1/2 a cluster key c_z + sigma*eps (z uniform over
    n_centres centres c ~ N(0, I)), otherwise N(0, I) noise.  w ~ N(0, 1/H).
    Queries: q ~ N(0, 1) when q_noise is None; otherwise the heads of query m
    share one direction, q_{m,h} = a_{m,h} c_{z_m} + q_noise * eps with
    a = |N(0, 1)| and z_m uniform over the centres (heads of a trained indexer
    are strongly correlated; this is the structure the anchor bound uses).
    q_run > 1: runs of q_run consecutive queries share their centre (neighbouring
    positions of a prompt look for the same content).  positive_w: w = |w|.
    """
    rng = np.random.default_rng(seed)
    centres = _normal(rng, (n_centres, D))
    is_cluster = rng.random(L) < 0.5
    z = rng.integers(0, n_centres, L)
    eps = _normal(rng, (L, D))
    kf = np.where(is_cluster[:, None], centres[z] + np.float32(sigma) * eps, eps).astype(np.float32)
    keys = _bulk_bf16(kf)
    if q_noise is None:
        q = _bulk_bf16(_normal(rng, (n_queries, H, D)))
    else:
        if q_run > 1:
            zq = np.repeat(rng.integers(0, n_centres, -(-n_queries // q_run)), q_run)[:n_queries]
        else:
            zq = rng.integers(0, n_centres, n_queries)
        amp = np.abs(_normal(rng, (n_queries, H)))
        qf = amp[:, :, None] * centres[zq][:, None, :] + np.float32(q_noise) * _normal(rng, (n_queries, H, D))
        q = _bulk_bf16(qf.astype(np.float32))
    w = _normal(rng, (n_queries, H), std=float(np.sqrt(1.0 / H)))
    if positive_w:
        w = np.abs(w)
    pos = np.arange(L - n_queries, L, dtype=np.int64)
    key_len = (pos + 1).astype(np.int32)
    return IndexerProblem("prefill_bf16", "bf16", q, w, keys, key_len, None, K,
                          extras=dict(n_seed=n_seed, R=R, pos=pos, q_noise=q_noise))


def ragged_fp8(seed: int = 5, M: int = 128, H: int = 64, D: int = 128, L_min: int = 4096,
               L_max: int = 131072, K: int = 2048, S: int = 32, R: int = 20,
               seed_cap: int = 8192) -> IndexerProblem:
    """Ragged decode batch with FP8 e4m3 keys and a per-token float32 scale.

    L_r ~ U{L_min..L_max}.  Keys k ~ N(0,1) are quantised per token:
    scale = amax/448 (1 when amax = 0), stored code = e4m3(k / scale).
    Queries are bf16, w ~ N(0, 1/H).
    """
    rng = np.random.default_rng(seed)
    key_len = rng.integers(L_min, L_max + 1, M).astype(np.int32)
    key_off = np.concatenate([[0], np.cumsum(key_len.astype(np.int64))[:-1]]).astype(np.int64)
    n_keys = int(key_len.astype(np.int64).sum())
    keys = np.empty((n_keys, D), dtype=np.uint8)
    scale = np.empty(n_keys, dtype=np.float32)
    chunk = max(1, (1 << 23) // D)
    for s in range(0, n_keys, chunk):
        e = min(n_keys, s + chunk)
        k = _normal(rng, (e - s, D))
        amax = np.abs(k).max(axis=1)
        sc = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        k /= sc[:, None]
        np.clip(k, -E4M3_MAX, E4M3_MAX, out=k)
        keys[s:e] = _bulk_e4m3(k)
        scale[s:e] = sc
    q = _bulk_bf16(_normal(rng, (M, H, D)))
    w = _normal(rng, (M, H), std=float(np.sqrt(1.0 / H)))
    return IndexerProblem("ragged_fp8", "fp8", q, w, keys, key_len, key_off, K,
                          key_scale=scale,
                          extras=dict(S=S, keep=K - S, max_repl=S, R=R, seed_cap=seed_cap))


def block_select(seed: int = 4, Q: int = 1024, n_kv: int = 8, D: int = 128, L: int = 131072,
                 block_size: int = 128, top_blocks: int = 32, init_blocks: int = 1,
                 local_blocks: int = 2, pos=None) -> BlockSelectProblem:
    """MiniMax block select; query i sits at position 128*i + 64 (mid-block)."""
    rng = np.random.default_rng(seed)
    index_k = _normal(rng, (L, D))
    index_q = _normal(rng, (Q, n_kv, D))
    if pos is None:
        pos = (np.arange(Q, dtype=np.int64) * max(1, L // Q) + max(1, L // Q) // 2).astype(np.int32)
    return BlockSelectProblem("block_select", index_q, index_k, np.asarray(pos, dtype=np.int32),
                              block_size, top_blocks, init_blocks, local_blocks)


def previous_step(wp: IndexerProblem, seed: int = 11, noise: float = 0.3) -> IndexerProblem:
    """The decode step before `wp`: every row saw one key fewer and its query
    was q + noise * N(0, 1) (rounded as q is stored); keys, offsets and
    weights are shared.  Its top-K is the prior of the step `wp`."""
    rng = np.random.default_rng(seed)
    qf = wp.q_f32() + np.float32(noise) * _normal(rng, wp.q.shape)
    q = qf.astype(np.float32) if wp.dtype == "f32" else _bulk_bf16(qf.astype(np.float32))
    key_len = np.maximum(np.asarray(wp.key_len, dtype=np.int32) - 1, 0).astype(np.int32)
    return IndexerProblem(wp.name + "_previous", wp.dtype, q, wp.w, wp.keys, key_len, wp.key_off, wp.K,
                          key_scale=wp.key_scale, extras=dict(wp.extras))


def witness_rows(seed: int, rows: int, topk: int, L_min: int = 1, L_max: int = 4096,
                 pad_frac: float = 0.1, oob_frac: float = 0.01):
    """Random learned rows for the witness merge: distinct in-range offsets with
    some -1 padding and a few out-of-range entries (x >= L_r)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(L_min, L_max + 1, rows).astype(np.int32)
    out = np.full((rows, topk), -1, dtype=np.int32)
    for r in range(rows):
        L = int(ctx[r])
        n = min(topk, L)
        if n > 0:
            out[r, :n] = rng.choice(L, size=n, replace=False).astype(np.int32)
        pad = rng.random(topk) < pad_frac
        out[r, pad] = -1
        oob = rng.random(topk) < oob_frac
        out[r, oob] = L + rng.integers(0, 1000, int(oob.sum()))
    return out, ctx


def score_rows(seed: int, M: int, L_max: int, ties: bool = False, ragged: bool = True):
    """Random float32 score rows [M, L_max] with row lengths in [0, L_max];
    `ties` draws small integers (many exact ties, signed zeros)."""
    rng = np.random.default_rng(seed)
    if ties:
        s = rng.integers(-4, 5, (M, L_max)).astype(np.float32)
        s[rng.random((M, L_max)) < 0.1] = np.float32(-0.0)
    else:
        s = rng.standard_normal((M, L_max), dtype=np.float32)
    lens = rng.integers(0, L_max + 1, M).astype(np.int32) if ragged else np.full(M, L_max, dtype=np.int32)
    return s, lens
