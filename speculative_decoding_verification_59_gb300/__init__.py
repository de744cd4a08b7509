"""GB300 (sm_103a) speculative-decoding verification.

A thin ctypes binding over the C ABI of libspecverify.so (declared in
include/spec_verify.h).  The functions named ``spec_verify_*`` take raw device
pointers and sizes exactly like the C calls; the ``verify_*`` helpers only
marshal torch CUDA tensors into those calls (pointers, current stream,
output allocation).  Every step of the verification runs in the library's
CUDA kernels: there is no CPU or PyTorch fallback, and using the package
without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "SPEC_OK", "SPEC_DTYPE_F32", "SPEC_DTYPE_BF16", "SpecVerifyError", "lib_path", "load_library",
    "spec_verify_workspace_size", "spec_verify_workspace_init", "spec_verify_sample",
    "spec_verify_sample_stats", "spec_verify_sample_finish", "spec_verify_sample_noalloc",
    "spec_verify_greedy", "spec_verify_tree_greedy", "spec_verify_read_error",
    "spec_verify_status_string", "Workspace", "verify_sample", "verify_greedy", "verify_tree_greedy",
]

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED_DTYPE = 2
SPEC_ERR_MISALIGNED = 3
SPEC_ERR_WORKSPACE_TOO_SMALL = 4
SPEC_ERR_CUDA = 5
SPEC_ERR_DEVICE_INPUT = 6
SPEC_ERR_EXCEEDS_STATIC_SCRATCH = 7
SPEC_VERIFY_NOALLOC_SCRATCH_BYTES = 8 << 20
SPEC_DTYPE_F32 = 0
SPEC_DTYPE_BF16 = 1
SPEC_DEVERR_TOKEN_RANGE = 1
SPEC_DEVERR_EMPTY_ROW = 2
SPEC_DEVERR_TREE_PARENT = 4
SPEC_DEVERR_TIMEOUT = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libspecverify.so")
_lib = None

# name -> (argtypes, restype); pointers travel as c_void_p, the stream as c_void_p
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "spec_verify_workspace_size": ([_I, _I, _I], _S),
    "spec_verify_workspace_init": ([_P, _S, _P], _I),
    "spec_verify_sample": ([_P, _P, _I, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P, _P, _S,
                            _P], _I),
    "spec_verify_sample_lazy": ([_P, _P, _I, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P, _P, _S,
                                 _P], _I),
    "spec_verify_lazy_groups": ([_I, _I, _I, _I, _P], _I),
    "spec_verify_sample_stats": ([_P, _P, _I, ctypes.c_float, _I, _I, _I, _P, _S, _P], _I),
    "spec_verify_sample_finish": ([_P, _P, _I, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P, _P,
                                   _S, _P], _I),
    "spec_verify_sample_noalloc": ([_P, _P, _I, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P,
                                    _P], _I),
    "spec_verify_greedy": ([_P, _I, _P, _I, _I, _I, _P, _P, _P, _S, _P], _I),
    "spec_verify_tree_greedy": ([_P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P, _S, _P], _I),
    "spec_topk_workspace_size": ([_I, _I, _I], _S),
    "spec_topk_exclude": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P], _I),
    "spec_ngram_workspace_size": ([_I, _I, _I], _S),
    "spec_ngram_retrieve": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P], _I),
    "spec_cosine_workspace_size": ([_I, _I], _S),
    "spec_cosine_topk": ([_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P], _I),
    "spec_verify_read_error": ([_P, _P, _P], _I),
    "spec_verify_status_string": ([_I], ctypes.c_char_p),
    "spec_verify_set_wait_limit": ([ctypes.c_uint32], None),
    "spec_verify_set_lazy_split_bytes": ([ctypes.c_double], None),
    "spec_verify_default_wait_limit": ([], ctypes.c_uint32),
}


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {spec_verify_status_string(status)} (status {status})")


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libspecverify.so (built in-tree by __graft_entry__.build() or
    speculative_decoding_verification_59_gb300._build).  Raises if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is not built; run __graft_entry__.build() first")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (argt, rest) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = lib
    return _lib


# ---- raw C-ABI calls (pointers are ints, stream is an int handle or 0) ------
def spec_verify_workspace_size(B: int, gamma_or_nodes: int, V: int) -> int:
    return load_library().spec_verify_workspace_size(B, gamma_or_nodes, V)


def spec_topk_workspace_size(rows: int, V: int, K: int) -> int:
    return load_library().spec_topk_workspace_size(rows, V, K)


def spec_topk_exclude(logits, dtype, rows, V, K, exclude, out_idx, out_val, ws, ws_bytes,
                      stream) -> int:
    return load_library().spec_topk_exclude(logits, dtype, rows, V, K, exclude, out_idx, out_val,
                                            ws, ws_bytes, stream)


def spec_ngram_workspace_size(B: int, n_max: int, max_matches: int) -> int:
    return load_library().spec_ngram_workspace_size(B, n_max, max_matches)


def spec_ngram_retrieve(tokens, lengths, B, n_max, w, L, max_matches, out_count, out_matches,
                        out_draft, ws, ws_bytes, stream) -> int:
    return load_library().spec_ngram_retrieve(tokens, lengths, B, n_max, w, L, max_matches,
                                              out_count, out_matches, out_draft, ws, ws_bytes,
                                              stream)


def spec_cosine_workspace_size(B: int, W: int) -> int:
    return load_library().spec_cosine_workspace_size(B, W)


def spec_cosine_topk(hidden, query, dtype, B, W, d, delta, positions, out_idx, out_pos, out_score,
                     ws, ws_bytes, stream) -> int:
    return load_library().spec_cosine_topk(hidden, query, dtype, B, W, d, delta, positions,
                                           out_idx, out_pos, out_score, ws, ws_bytes, stream)


def spec_verify_workspace_init(ws: int, nbytes: int, stream: int = 0) -> int:
    return load_library().spec_verify_workspace_init(ws, nbytes, stream)


def spec_verify_sample(target, draft, dtype, draft_tokens, uniforms, temperature, B, gamma, V,
                       out_tokens, out_num_accepted, out_logprobs, ws, ws_bytes, stream) -> int:
    return load_library().spec_verify_sample(target, draft, dtype, draft_tokens, uniforms,
                                             temperature, B, gamma, V, out_tokens,
                                             out_num_accepted, out_logprobs, ws, ws_bytes, stream)


def spec_verify_sample_lazy(target, draft, dtype, draft_tokens, uniforms, temperature, B, gamma,
                            V, out_tokens, out_num_accepted, out_logprobs, ws, ws_bytes,
                            stream) -> int:
    return load_library().spec_verify_sample_lazy(target, draft, dtype, draft_tokens, uniforms,
                                                  temperature, B, gamma, V, out_tokens,
                                                  out_num_accepted, out_logprobs, ws, ws_bytes,
                                                  stream)


def spec_verify_lazy_groups(B, gamma, V, dtype, ends) -> int:
    return load_library().spec_verify_lazy_groups(B, gamma, V, dtype, ends)


def lazy_groups(B: int, gamma: int, V: int, dtype: int):
    """Position groups of spec_verify_sample_lazy as [(lo, hi), ...] (host only,
    no GPU needed); raises for invalid arguments."""
    ends = (ctypes.c_int32 * 8)()
    n = spec_verify_lazy_groups(B, gamma, V, dtype, ctypes.addressof(ends))
    if n < 1:
        raise ValueError(f"spec_verify_lazy_groups: invalid arguments {(B, gamma, V, dtype)}")
    out, lo = [], 0
    for g in range(n):
        out.append((lo, int(ends[g])))
        lo = int(ends[g])
    return out


def spec_verify_sample_stats(target, draft, dtype, temperature, B, gamma, V, ws, ws_bytes,
                             stream) -> int:
    return load_library().spec_verify_sample_stats(target, draft, dtype, temperature, B, gamma, V,
                                                   ws, ws_bytes, stream)


def spec_verify_sample_finish(target, draft, dtype, draft_tokens, uniforms, temperature, B, gamma,
                              V, out_tokens, out_num_accepted, out_logprobs, ws, ws_bytes,
                              stream) -> int:
    return load_library().spec_verify_sample_finish(target, draft, dtype, draft_tokens, uniforms,
                                                    temperature, B, gamma, V, out_tokens,
                                                    out_num_accepted, out_logprobs, ws, ws_bytes,
                                                    stream)


def spec_verify_sample_noalloc(target, draft, dtype, draft_tokens, uniforms, temperature, B, gamma,
                               V, out_tokens, out_num_accepted, out_logprobs, stream) -> int:
    """spec_verify_sample without a workspace, for callers that cannot
    allocate device memory (see include/spec_verify.h)."""
    return load_library().spec_verify_sample_noalloc(target, draft, dtype, draft_tokens, uniforms,
                                                     temperature, B, gamma, V, out_tokens,
                                                     out_num_accepted, out_logprobs, stream)


def spec_verify_greedy(target, dtype, draft_tokens, B, gamma, V, out_tokens, out_num_accepted,
                       ws, ws_bytes, stream) -> int:
    return load_library().spec_verify_greedy(target, dtype, draft_tokens, B, gamma, V, out_tokens,
                                             out_num_accepted, ws, ws_bytes, stream)


def spec_verify_tree_greedy(target, dtype, node_tokens, parents, B, N, V, out_path_nodes,
                            out_tokens, out_num_accepted, ws, ws_bytes, stream) -> int:
    return load_library().spec_verify_tree_greedy(target, dtype, node_tokens, parents, B, N, V,
                                                  out_path_nodes, out_tokens, out_num_accepted,
                                                  ws, ws_bytes, stream)


def spec_verify_read_error(ws: int, stream: int = 0):
    code = ctypes.c_int32(0)
    st = load_library().spec_verify_read_error(ws, stream, ctypes.addressof(code))
    return st, code.value


def spec_verify_set_lazy_split_bytes(nbytes: float) -> None:
    load_library().spec_verify_set_lazy_split_bytes(float(nbytes))


def spec_verify_set_wait_limit(polls: int) -> None:
    load_library().spec_verify_set_wait_limit(polls)


def spec_verify_default_wait_limit() -> int:
    return load_library().spec_verify_default_wait_limit()


def spec_verify_status_string(status: int) -> str:
    try:
        return load_library().spec_verify_status_string(status).decode()
    except ImportError:
        return "status %d" % status


# ---- torch marshalling ----------------------------------------------------------
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SPEC_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return SPEC_DTYPE_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_tensor(t, name: str, shape, dtypes, device=None):
    """Raises unless t is a contiguous CUDA tensor of one of dtypes, of the
    given shape (None entries match anything) and, when given, on device: the
    C ABI reads raw device memory, so a strided, host-resident or mistyped
    tensor would be read as garbage rather than rejected."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor, got {type(t).__name__}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got device {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other arguments on {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if len(t.shape) != len(shape) or any(w is not None and w != h for w, h in zip(shape, t.shape)):
        raise ValueError(f"{name} must have shape {tuple('*' if w is None else w for w in shape)}, "
                         f"got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _logits_dtypes():
    torch = _torch()
    return (torch.float32, torch.bfloat16)


def _stream(stream) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, what: str):
    if status != SPEC_OK:
        raise SpecVerifyError(status, what)


class Workspace:
    """Device scratch for the verification calls, zero-filled when it is
    (re)allocated so the error word starts clear.  Grows on demand."""

    def __init__(self, device=None):
        torch = _torch()
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = None

    def get(self, B: int, g: int, V: int, stream=None):
        return self.get_bytes(spec_verify_workspace_size(B, g, V), stream)

    def get_bytes(self, need: int, stream=None):
        torch = _torch()
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.empty(max(need, 256), dtype=torch.uint8, device=self.device)
            _check(spec_verify_workspace_init(self.buf.data_ptr(), self.buf.numel(), _stream(stream)),
                   "spec_verify_workspace_init")
        return self.buf.data_ptr(), self.buf.numel()

    def read_error(self, stream=None) -> int:
        st, code = spec_verify_read_error(self.buf.data_ptr(), _stream(stream))
        _check(st, "spec_verify_read_error")
        return code


_default_ws = {}


def _ws(workspace, device):
    if workspace is not None:
        return workspace
    key = str(device)
    if key not in _default_ws:
        _default_ws[key] = Workspace(device)
    return _default_ws[key]


def verify_sample(target, draft, draft_tokens, uniforms, temperature: float, *, logprobs=False,
                  workspace: Optional[Workspace] = None, out=None, stream=None, lazy=False):
    """Stochastic verification (see spec_verify_sample).  target [B, g+1, V],
    draft [B, g, V] (same dtype), draft_tokens [B, g] int32, uniforms
    [B, g+1] float32, all contiguous CUDA tensors.  Returns (tokens [B, g+1],
    num_accepted [B]) or, with logprobs=True, also [B, g, 2] log-probabilities.
    lazy=True: spec_verify_sample_lazy (same tokens and counts; the rows of the
    position groups after the one holding a sequence's first rejection are not
    read, and the log-probabilities of positions after the rejection are NaN)."""
    torch = _torch()
    _check_tensor(target, "target", (None, None, None), _logits_dtypes())
    B, g1, V = target.shape
    g = g1 - 1
    dev = target.device
    if g > 0:
        _check_tensor(draft, "draft", (B, g, V), (target.dtype,), dev)
        _check_tensor(draft_tokens, "draft_tokens", (B, g), (torch.int32,), dev)
    _check_tensor(uniforms, "uniforms", (B, g1), (torch.float32,), dev)
    if out is None:
        tok = torch.empty((B, g1), dtype=torch.int32, device=dev)
        acc = torch.empty((B,), dtype=torch.int32, device=dev)
        lp = torch.empty((B, g, 2), dtype=torch.float32, device=dev) if logprobs else None
    else:
        tok, acc, lp = out
        _check_tensor(tok, "out tokens", (B, g1), (torch.int32,), dev)
        _check_tensor(acc, "out num_accepted", (B,), (torch.int32,), dev)
        if lp is not None:
            _check_tensor(lp, "out logprobs", (B, g, 2), (torch.float32,), dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get(B, g, V, stream)
    fn = spec_verify_sample_lazy if lazy else spec_verify_sample
    st = fn(_ptr(target), _ptr(draft) if g > 0 else None, _dtype_code(target),
            _ptr(draft_tokens) if g > 0 else None, _ptr(uniforms), float(temperature), B, g, V,
            _ptr(tok), _ptr(acc), _ptr(lp), wp, wb, _stream(stream))
    _check(st, "spec_verify_sample_lazy" if lazy else "spec_verify_sample")
    return (tok, acc, lp) if logprobs else (tok, acc)


def topk_exclude(logits, K: int, exclude=None, *, values=False,
                 workspace: Optional[Workspace] = None, out=None, stream=None):
    """Top-K branch tokens (see spec_topk_exclude).  logits [..., V] contiguous
    CUDA tensor (bf16 or fp32), exclude int32 with one entry per row or None.
    Returns idx [..., K] int32 (and, with values=True, the logits [..., K])."""
    torch = _torch()
    _check_tensor(logits, "logits", (None,) * max(logits.dim(), 1), _logits_dtypes())
    V = logits.shape[-1]
    rows = logits.numel() // V
    dev = logits.device
    if exclude is not None:
        _check_tensor(exclude, "exclude", tuple(logits.shape[:-1]), (torch.int32,), dev)
    if out is None:
        idx = torch.empty((*logits.shape[:-1], K), dtype=torch.int32, device=dev)
        val = torch.empty((*logits.shape[:-1], K), dtype=torch.float32, device=dev) if values else None
    else:
        idx, val = out
        _check_tensor(idx, "out idx", (*logits.shape[:-1], K), (torch.int32,), dev)
        if val is not None:
            _check_tensor(val, "out values", (*logits.shape[:-1], K), (torch.float32,), dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get_bytes(spec_topk_workspace_size(rows, V, K), stream)
    st = spec_topk_exclude(_ptr(logits), _dtype_code(logits), rows, V, K, _ptr(exclude), _ptr(idx),
                           _ptr(val), wp, wb, _stream(stream))
    _check(st, "spec_topk_exclude")
    return (idx, val) if values else idx


def ngram_retrieve(tokens, lengths, w: int, L: int, max_matches: int, *,
                   workspace: Optional[Workspace] = None, stream=None):
    """Lexical retrieval (see spec_ngram_retrieve).  tokens [B, n_max] int32
    (n_max a multiple of 4), lengths [B] int32, CUDA tensors.  Returns
    (count [B], matches [B, max_matches], draft [B, L])."""
    torch = _torch()
    _check_tensor(tokens, "tokens", (None, None), (torch.int32,))
    B, n_max = tokens.shape
    dev = tokens.device
    _check_tensor(lengths, "lengths", (B,), (torch.int32,), dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    mat = torch.empty((B, max_matches), dtype=torch.int32, device=dev)
    dr = torch.empty((B, max(L, 1)), dtype=torch.int32, device=dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get_bytes(spec_ngram_workspace_size(B, n_max, max_matches), stream)
    st = spec_ngram_retrieve(_ptr(tokens), _ptr(lengths), B, n_max, w, L, max_matches, _ptr(cnt),
                             _ptr(mat), _ptr(dr), wp, wb, _stream(stream))
    _check(st, "spec_ngram_retrieve")
    return cnt, mat, dr[:, :L]


def cosine_topk(hidden, query, delta: int, positions=None, *,
                workspace: Optional[Workspace] = None, stream=None):
    """Semantic fallback (see spec_cosine_topk).  hidden [B, W, d], query
    [B, d] (same dtype, bf16 or fp32), positions [B, W] int32 or None, CUDA
    tensors.  Returns (idx [B, delta], pos [B, delta], score [B, delta])."""
    torch = _torch()
    _check_tensor(hidden, "hidden", (None, None, None), _logits_dtypes())
    B, W, d = hidden.shape
    dev = hidden.device
    _check_tensor(query, "query", (B, d), (hidden.dtype,), dev)
    if positions is not None:
        _check_tensor(positions, "positions", (B, W), (torch.int32,), dev)
    idx = torch.empty((B, delta), dtype=torch.int32, device=dev)
    pos = torch.empty((B, delta), dtype=torch.int32, device=dev)
    sc = torch.empty((B, delta), dtype=torch.float32, device=dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get_bytes(spec_cosine_workspace_size(B, W), stream)
    st = spec_cosine_topk(_ptr(hidden), _ptr(query), _dtype_code(hidden), B, W, d, delta,
                          _ptr(positions), _ptr(idx), _ptr(pos), _ptr(sc), wp, wb, _stream(stream))
    _check(st, "spec_cosine_topk")
    return idx, pos, sc


def verify_greedy(target, draft_tokens, *, workspace: Optional[Workspace] = None, out=None,
                  stream=None):
    """Greedy verification (see spec_verify_greedy).  Returns (tokens, num_accepted)."""
    torch = _torch()
    _check_tensor(target, "target", (None, None, None), _logits_dtypes())
    B, g1, V = target.shape
    g = g1 - 1
    dev = target.device
    if g > 0:
        _check_tensor(draft_tokens, "draft_tokens", (B, g), (torch.int32,), dev)
    if out is None:
        tok = torch.empty((B, g1), dtype=torch.int32, device=dev)
        acc = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        tok, acc = out
        _check_tensor(tok, "out tokens", (B, g1), (torch.int32,), dev)
        _check_tensor(acc, "out num_accepted", (B,), (torch.int32,), dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get(B, g, V, stream)
    st = spec_verify_greedy(_ptr(target), _dtype_code(target), _ptr(draft_tokens) if g > 0 else None,
                            B, g, V, _ptr(tok), _ptr(acc), wp, wb, _stream(stream))
    _check(st, "spec_verify_greedy")
    return tok, acc


def verify_tree_greedy(target, node_tokens, parents, *, workspace: Optional[Workspace] = None,
                       out=None, stream=None):
    """Greedy tree verification (see spec_verify_tree_greedy).  Returns
    (path_nodes [B, N], tokens [B, N], num_accepted [B])."""
    torch = _torch()
    _check_tensor(target, "target", (None, None, None), _logits_dtypes())
    B, N, V = target.shape
    dev = target.device
    _check_tensor(node_tokens, "node_tokens", (B, N), (torch.int32,), dev)
    _check_tensor(parents, "parents", (B, N), (torch.int32,), dev)
    if out is None:
        nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
        tok = torch.empty((B, N), dtype=torch.int32, device=dev)
        acc = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        nodes, tok, acc = out
        _check_tensor(nodes, "out path_nodes", (B, N), (torch.int32,), dev)
        _check_tensor(tok, "out tokens", (B, N), (torch.int32,), dev)
        _check_tensor(acc, "out num_accepted", (B,), (torch.int32,), dev)
    ws = _ws(workspace, dev)
    wp, wb = ws.get(B, N, V, stream)
    st = spec_verify_tree_greedy(_ptr(target), _dtype_code(target), _ptr(node_tokens),
                                 _ptr(parents), B, N, V, _ptr(nodes), _ptr(tok), _ptr(acc), wp, wb,
                                 _stream(stream))
    _check(st, "spec_verify_tree_greedy")
    return nodes, tok, acc
