"""ctypes wrappers around the C oracle (``fs_oracle.c``).

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Every function takes
and returns numpy arrays.  bf16 tensors are passed as their raw uint16 words.

Citations are to "FlashSampling: Fast and Memory-Efficient Exact Sampling"
(arXiv 2603.15854): the Gumbel-max rule and its single-pass online form (method
section, Algorithm I.1 in the Appendix), the exactness statement (a tiled
argmax returns the same maximizer as a full Gumbel-max pass, Appendix C), and
the LM-head GEMM of the IO-model section.
"""
import ctypes
import os

import numpy as np

from . import build as _build

NO_NOISE = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u64, i64, u32, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32, ctypes.c_int
        vp = ctypes.c_void_p
        lib.oracle_philox4x64_10.argtypes = [vp, vp, vp]
        lib.oracle_philox4x64_10.restype = None
        lib.oracle_noise_word.argtypes = [u64, u64, i64, i64]
        lib.oracle_noise_word.restype = u32
        lib.oracle_uniform.argtypes = [u32]
        lib.oracle_uniform.restype = ctypes.c_double
        lib.oracle_gumbel_from_word.argtypes = [u32]
        lib.oracle_gumbel_from_word.restype = ctypes.c_float
        lib.oracle_gumbel.argtypes = [u64, u64, i64, i64]
        lib.oracle_gumbel.restype = ctypes.c_float
        lib.oracle_noise_block.argtypes = [u64, u64, i64, i64, i64, i64, vp, vp, i32]
        lib.oracle_noise_block.restype = None
        lib.oracle_uniform_block.argtypes = [vp, i64, vp]
        lib.oracle_uniform_block.restype = None
        lib.oracle_gumbel_block.argtypes = [vp, i64, vp, i32]
        lib.oracle_gumbel_block.restype = None
        lib.oracle_logits.argtypes = [vp, vp, i64, i64, i64, vp, i32]
        lib.oracle_logits.restype = None
        lib.oracle_logits64.argtypes = [vp, vp, i64, i64, i64, vp, i32]
        lib.oracle_logits64.restype = None
        lib.oracle_sample_from_logits.argtypes = [vp, i64, i64, vp, vp, u64, u64, u32,
                                                  vp, vp, vp, vp, i32]
        lib.oracle_sample_from_logits.restype = None
        lib.oracle_sample.argtypes = [vp, vp, i64, i64, i64, vp, vp, u64, u64, u32,
                                      vp, vp, vp, vp, i32]
        lib.oracle_sample.restype = None
        lib.oracle_logprob.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.oracle_logprob.restype = None
        lib.oracle_transform_logits.argtypes = [vp, i64, i64, vp, ctypes.c_float, vp, i64]
        lib.oracle_transform_logits.restype = None
        lib.oracle_group_gumbel.argtypes = [u64, u64, i64, i64]
        lib.oracle_group_gumbel.restype = ctypes.c_float
        lib.oracle_sample_shard.argtypes = [vp, vp, i64, i64, i64, i64, vp, u64, u64, vp, vp, vp,
                                            vp, i32]
        lib.oracle_sample_shard.restype = None
        lib.oracle_combine_groups.argtypes = [i64, i64, vp, vp, u64, u64, vp, vp, vp, vp]
        lib.oracle_combine_groups.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().oracle_num_threads())


def philox4x64_10(counter, key):
    """One Philox4x64-10 block (SC'11): counter [4] uint64, key [2] uint64."""
    c = _c(counter, np.uint64)
    k = _c(key, np.uint64)
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def noise_word(seed, offset, b, v) -> int:
    return int(_load().oracle_noise_word(seed, offset, b, v))


def uniform(x) -> float:
    return float(_load().oracle_uniform(x))


def gumbel_from_word(x) -> float:
    return float(_load().oracle_gumbel_from_word(x))


def gumbel(seed, offset, b, v) -> float:
    return float(_load().oracle_gumbel(seed, offset, b, v))


def uniform_block(words):
    """u for each 32-bit word (float64, exact)."""
    x = _c(words, np.uint32)
    u = np.zeros(x.shape, dtype=np.float64)
    _load().oracle_uniform_block(_ptr(x), x.size, _ptr(u))
    return u


def gumbel_block(words, nthreads=0):
    """g for each 32-bit word (f32)."""
    x = _c(words, np.uint32)
    g = np.zeros(x.shape, dtype=np.float32)
    _load().oracle_gumbel_block(_ptr(x), x.size, _ptr(g), nthreads)
    return g


def noise_block(seed, offset, b0, nb, v0, nv, nthreads=0):
    """Random words and Gumbels for rows [b0, b0+nb) x vocab [v0, v0+nv)."""
    words = np.zeros((nb, nv), dtype=np.uint32)
    g = np.zeros((nb, nv), dtype=np.float32)
    _load().oracle_noise_block(seed, offset, b0, nb, v0, nv, _ptr(words), _ptr(g),
                               nthreads)
    return words, g


def logits(H_bits, W_bits, nthreads=0):
    """The oracle's logits H W^T (f32 [B, V]) from raw bf16 words H [B, D] and
    W [V, D]: exact f32 products summed in f32 in index order k = 0..D-1."""
    H = _c(H_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    B, D = H.shape
    V, D2 = W.shape
    assert D == D2
    out = np.zeros((B, V), dtype=np.float32)
    _load().oracle_logits(_ptr(H), _ptr(W), B, V, D, _ptr(out), nthreads)
    return out


def logits64(H_bits, W_bits, nthreads=0):
    """Diagnostic: the same products summed in fp64 (float64 [B, V])."""
    H = _c(H_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    B, D = H.shape
    V, D2 = W.shape
    assert D == D2
    out = np.zeros((B, V), dtype=np.float64)
    _load().oracle_logits64(_ptr(H), _ptr(W), B, V, D, _ptr(out), nthreads)
    return out


def _temps(T, B):
    T = np.asarray(T, dtype=np.float32)
    if T.ndim == 0:
        T = np.full(B, T, dtype=np.float32)
    assert T.shape == (B,)
    return np.ascontiguousarray(T)


def _rows(row_ids, B):
    if row_ids is None:
        return None
    r = np.ascontiguousarray(row_ids, dtype=np.int64)
    assert r.shape == (B,)
    return r


def sample_from_logits(l32, T, seed, offset, flags=0, want_scores=False, nthreads=0,
                       row_ids=None):
    """Full Gumbel-max pass over given f32 logits [B, V].

    row_ids: optional row index (in the full batch) of each given row; it keys
    the noise counter.  Default 0..B-1.
    Returns (idx int64 [B], best f32 [B], second f32 [B], scores or None).
    """
    L = _c(l32, np.float32)
    B, V = L.shape
    Tv = _temps(T, B)
    rows = _rows(row_ids, B)
    idx = np.zeros(B, dtype=np.int64)
    best = np.zeros(B, dtype=np.float32)
    second = np.zeros(B, dtype=np.float32)
    scores = np.zeros((B, V), dtype=np.float32) if want_scores else None
    _load().oracle_sample_from_logits(_ptr(L), B, V, _ptr(Tv), _ptr(rows), seed, offset, flags,
                                      _ptr(idx), _ptr(best), _ptr(second),
                                      _ptr(scores), nthreads)
    return idx, best, second, scores


def sample(H_bits, W_bits, T, seed, offset, flags=0, want_logits=False, nthreads=0,
           row_ids=None):
    """The whole path from bf16 H [B, D] and W [V, D].

    row_ids: optional row index (in the full batch) of each given row of H.
    Returns (idx int64 [B], best f32 [B], second f32 [B], logits or None),
    the logits being the f32 [B, V] the pass sampled from.
    """
    H = _c(H_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    B, D = H.shape
    V, D2 = W.shape
    assert D == D2
    Tv = _temps(T, B)
    rows = _rows(row_ids, B)
    idx = np.zeros(B, dtype=np.int64)
    best = np.zeros(B, dtype=np.float32)
    second = np.zeros(B, dtype=np.float32)
    l32 = np.zeros((B, V), dtype=np.float32) if want_logits else None
    _load().oracle_sample(_ptr(H), _ptr(W), B, V, D, _ptr(Tv), _ptr(rows), seed, offset, flags,
                          _ptr(idx), _ptr(best), _ptr(second), _ptr(l32), nthreads)
    return idx, best, second, l32


def group_gumbel(seed, offset, b, g) -> float:
    """The Gumbel of group g of row b in the grouped sampler (counter word 3 = 1)."""
    return float(_load().oracle_group_gumbel(seed, offset, b, g))


def sample_shard(H_bits, W_shard_bits, vocab_offset, T, seed, offset, nthreads=0):
    """Local sample (global index), its score and the local log-mass of a
    vocabulary slice.  Returns (idx int64 [B], score f32 [B], logmass f64 [B],
    second f32 [B]) -- second: the slice's runner-up score."""
    H = _c(H_bits, np.uint16)
    Ws = _c(W_shard_bits, np.uint16)
    B, D = H.shape
    Vs = Ws.shape[0]
    Tv = _temps(T, B)
    idx = np.zeros(B, dtype=np.int64)
    score = np.zeros(B, dtype=np.float32)
    second = np.zeros(B, dtype=np.float32)
    lm = np.zeros(B, dtype=np.float64)
    _load().oracle_sample_shard(_ptr(H), _ptr(Ws), B, Vs, D, int(vocab_offset), _ptr(Tv), seed,
                                offset, _ptr(idx), _ptr(score), _ptr(second), _ptr(lm), nthreads)
    return idx, score, lm, second


def combine_groups(group_idx, group_logmass, seed, offset, want_scores=False):
    """Grouped sampler: draw a group by Gumbel-max over the log-masses [G, B]
    (rounded to f32, the kernel's precision) and return (idx [B], group [B])
    [, best f32 [B], second f32 [B]]."""
    gi = _c(group_idx, np.int64)
    gl = _c(group_logmass, np.float32)
    G, B = gi.shape
    out = np.zeros(B, dtype=np.int64)
    grp = np.zeros(B, dtype=np.int64)
    best = np.zeros(B, dtype=np.float32)
    second = np.zeros(B, dtype=np.float32)
    _load().oracle_combine_groups(G, B, _ptr(gi), _ptr(gl), seed, offset, _ptr(out), _ptr(grp),
                                  _ptr(best), _ptr(second))
    if want_scores:
        return out, grp, best, second
    return out, grp


def transform_logits(l32, bias=None, softcap=0.0, mask=None):
    """Bias, soft-cap and allowed-token mask applied to f32 logits [B, V] (a copy).

    mask: uint32 [B, words] (bit v & 31 of word v >> 5 allows token v) or None.
    """
    L = np.array(l32, dtype=np.float32, order="C", copy=True)
    B, V = L.shape
    bv = None if bias is None else _c(bias, np.float32)
    mk = None if mask is None else _c(mask, np.uint32)
    words = 0 if mk is None else mk.shape[1]
    _load().oracle_transform_logits(_ptr(L), B, V, _ptr(bv), float(softcap), _ptr(mk), words)
    return L


def logprob(l32, T, idx):
    """log softmax(l~)[idx] per row in fp64, l~ = fl(l * fl(1/T)) (f32 logits [B, V])."""
    L = _c(l32, np.float32)
    B, V = L.shape
    Tv = _temps(T, B)
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.zeros(B, dtype=np.float64)
    _load().oracle_logprob(_ptr(L), B, V, _ptr(Tv), _ptr(ix), _ptr(out))
    return out


__all__ = ["group_gumbel", "sample_shard", "combine_groups", "transform_logits", "logprob", "NO_NOISE", "num_threads", "philox4x64_10", "noise_word", "uniform",
           "gumbel_from_word", "gumbel", "uniform_block", "gumbel_block", "noise_block", "logits",
           "logits64", "sample_from_logits", "sample"]
