"""fp64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, index-order
compensated sums); this module compiles it with gcc and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to the sources (-O2, no fast-math, OpenMP)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_verify_sample.argtypes = [P, P, P, P, ctypes.c_double, I, I, I, P, P, P, P, P, I]
            lib.oracle_verify_sample.restype = I
            lib.oracle_verify_greedy.argtypes = [P, P, I, I, I, P, P, P, I]
            lib.oracle_verify_greedy.restype = I
            lib.oracle_verify_tree_greedy.argtypes = [P, P, P, I, I, I, P, P, P, I]
            lib.oracle_verify_tree_greedy.restype = I
            lib.oracle_topk_exclude.argtypes = [P, P, I, I, I, P, P, I]
            lib.oracle_topk_exclude.restype = I
            lib.oracle_ngram_retrieve.argtypes = [P, P, I, I, I, I, I, P, P, P, I]
            lib.oracle_ngram_retrieve.restype = I
            _lib = lib
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def verify_sample(target, draft, tokens, uniforms, T, *, want_logprob=False, want_ratio=False,
                  want_cdf=False, nthreads=0):
    """Stochastic verification.  target [B, g+1, V], draft [B, g, V] float32
    (bf16 inputs as exact float32), tokens [B, g], uniforms [B, g+1].
    Returns a dict with tokens, accepted, bad and the optional diagnostics."""
    lib = _load()
    target = _f32(target)
    B, g1, V = target.shape
    g = g1 - 1
    draft = _f32(draft) if g > 0 else None
    tokens = _i32(tokens) if g > 0 else None
    uniforms = _f32(uniforms)
    assert uniforms.shape == (B, g + 1)
    if g > 0:
        assert draft.shape == (B, g, V) and tokens.shape == (B, g)
    out_t = np.empty((B, g + 1), np.int32)
    out_a = np.empty((B,), np.int32)
    lp = np.empty((B, g, 2), np.float64) if want_logprob else None
    ra = np.empty((B, g), np.float64) if want_ratio else None
    cdf = np.empty((B, V), np.float64) if want_cdf else None
    bad = lib.oracle_verify_sample(_ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms),
                                   float(T), B, g, V, _ptr(out_t), _ptr(out_a), _ptr(lp),
                                   _ptr(ra), _ptr(cdf), int(nthreads))
    if bad < 0:
        raise ValueError("oracle_verify_sample: invalid arguments")
    return {"tokens": out_t, "accepted": out_a, "bad": bad, "logprob": lp, "ratio": ra, "cdf": cdf}


def verify_greedy(target, tokens, *, nthreads=0):
    lib = _load()
    target = _f32(target)
    B, g1, V = target.shape
    g = g1 - 1
    tokens = _i32(tokens) if g > 0 else None
    out_t = np.empty((B, g + 1), np.int32)
    out_a = np.empty((B,), np.int32)
    amax = np.empty((B, g + 1), np.int32)
    bad = lib.oracle_verify_greedy(_ptr(target), _ptr(tokens), B, g, V, _ptr(out_t), _ptr(out_a),
                                   _ptr(amax), int(nthreads))
    if bad < 0:
        raise ValueError("oracle_verify_greedy: invalid arguments")
    return {"tokens": out_t, "accepted": out_a, "argmax": amax, "bad": bad}


def verify_tree_greedy(target, node_tokens, parents, *, nthreads=0):
    lib = _load()
    target = _f32(target)
    B, N, V = target.shape
    node_tokens = _i32(node_tokens)
    parents = _i32(parents)
    out_n = np.empty((B, N), np.int32)
    out_t = np.empty((B, N), np.int32)
    out_a = np.empty((B,), np.int32)
    bad = lib.oracle_verify_tree_greedy(_ptr(target), _ptr(node_tokens), _ptr(parents), B, N, V,
                                        _ptr(out_n), _ptr(out_t), _ptr(out_a), int(nthreads))
    if bad < 0:
        raise ValueError("oracle_verify_tree_greedy: invalid arguments")
    return {"nodes": out_n, "tokens": out_t, "accepted": out_a, "bad": bad}


def topk_exclude(logits, K, exclude=None, *, nthreads=0):
    """Top-K tokens of each row of logits [R, V] (larger logit first, lower
    index on ties), with exclude[r] removed and -1 padding."""
    lib = _load()
    logits = _f32(logits)
    R, V = logits.shape
    ex = None if exclude is None else _i32(exclude)
    out_i = np.empty((R, K), np.int32)
    out_v = np.empty((R, K), np.float32)
    rc = lib.oracle_topk_exclude(_ptr(logits), _ptr(ex), R, V, int(K), _ptr(out_i), _ptr(out_v),
                                 int(nthreads))
    if rc < 0:
        raise ValueError("oracle_topk_exclude: invalid arguments")
    return {"idx": out_i, "val": out_v}


def ngram_retrieve(tokens, lengths, w, L, max_matches, *, nthreads=0):
    """Lexical retrieval per sequence: match count, the first max_matches match
    positions (ascending, -1 padded) and the draft after the last match."""
    lib = _load()
    tokens = _i32(tokens)
    B, n_max = tokens.shape
    lengths = _i32(lengths)
    cnt = np.empty((B,), np.int32)
    mat = np.empty((B, max_matches), np.int32)
    dr = np.empty((B, L), np.int32)
    bad = lib.oracle_ngram_retrieve(_ptr(tokens), _ptr(lengths), B, n_max, int(w), int(L),
                                    int(max_matches), _ptr(cnt), _ptr(mat), _ptr(dr),
                                    int(nthreads))
    if bad < 0:
        raise ValueError("oracle_ngram_retrieve: invalid arguments")
    return {"count": cnt, "matches": mat, "draft": dr, "bad": bad}


def cosine_topk(hidden, query, delta, positions=None):
    """Semantic fallback of AdaPLD (section 3.2, "semantic fallback stage";
    Algorithm 1, SemanticFallback): score(j) = h_current . h_j /
    (|h_current| |h_j|) over the window rows h_j of each sequence, in fp64
    (0 when either norm is 0), then the delta largest scores, larger first,
    lower window index first among equal scores.  hidden [B, W, d], query
    [B, d] (float32 arrays holding the exact input values); positions [B, W]
    maps window rows to context positions (None: the window index itself).
    Returns idx [B, delta] (window rows), pos [B, delta], score [B, delta]
    and all scores [B, W]."""
    H = np.asarray(hidden, dtype=np.float64)
    q = np.asarray(query, dtype=np.float64)
    B, W, d = H.shape
    dots = np.einsum("bwd,bd->bw", H, q)
    nh = np.sqrt(np.einsum("bwd,bwd->bw", H, H))
    nq = np.sqrt(np.einsum("bd,bd->b", q, q))
    den = nh * nq[:, None]
    scores = np.where(den > 0, dots / np.where(den > 0, den, 1.0), 0.0)
    idx = np.full((B, delta), -1, np.int32)
    sc = np.full((B, delta), -np.inf)
    for b in range(B):
        order = np.lexsort((np.arange(W), -scores[b]))[:delta]
        idx[b, :len(order)] = order
        sc[b, :len(order)] = scores[b, order]
    if positions is None:
        pos = idx.copy()
    else:
        P = np.asarray(positions, dtype=np.int32)
        pos = np.where(idx >= 0, np.take_along_axis(P, np.maximum(idx, 0), axis=1), -1)
    return {"idx": idx, "pos": pos.astype(np.int32), "score": sc, "scores": scores}

