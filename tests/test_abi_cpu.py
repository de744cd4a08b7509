"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/spec_verify.h declares, sizes workspaces, and rejects
bad arguments before touching the device (no kernel is launched here)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_59_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sv.lib_path()):
        import __graft_entry__
        __graft_entry__.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(spec_[a-z_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7, names
    for n in names:
        assert hasattr(lib, n), n
        assert n in sv.SIGNATURES, n


@pytest.fixture
def split_bytes():
    """Sets the lazy pass's split figure for one test, restoring the built-in
    one afterwards."""
    yield sv.spec_verify_set_lazy_split_bytes
    sv.spec_verify_set_lazy_split_bytes(-1.0)


def test_lazy_groups_schedule(lib, split_bytes):
    """The lazy pass's position groups, from the host-only schedule call: the
    benchmark workloads' groups, the doubling schedule with every boundary
    taken, and its invariants for every gamma."""
    split_bytes(-1.0)
    bf16, f32 = sv.SPEC_DTYPE_BF16, sv.SPEC_DTYPE_F32
    assert sv.lazy_groups(64, 7, 151936, bf16) == [(0, 2), (2, 8)]        # 58 MB after [2, 6)
    assert sv.lazy_groups(8, 7, 151936, bf16) == [(0, 8)]                 # 32 MB after [0, 2)
    assert sv.lazy_groups(256, 4, 128256, f32) == [(0, 2), (2, 5)]
    assert sv.lazy_groups(1, 0, 1000, f32) == [(0, 1)]
    split_bytes(0)
    assert sv.lazy_groups(1, 7, 1000, f32) == [(0, 2), (2, 6), (6, 8)]
    assert sv.lazy_groups(1, 256, 1000, f32) == [(0, 2), (2, 6), (6, 14), (14, 30), (30, 62),
                                                 (62, 126), (126, 254), (254, 257)]
    for split in (0, 1e11):
        split_bytes(split)
        for gamma in range(0, 257):
            gr = sv.lazy_groups(3, gamma, 4096, bf16)
            assert gr[0][0] == 0 and gr[-1][1] == gamma + 1 and len(gr) <= 8
            for (lo, hi), (lo2, _) in zip(gr, gr[1:]):
                assert hi == lo2
            for g, (lo, hi) in enumerate(gr):
                assert 0 < hi - lo <= 128
                assert hi - lo >= min(2 << g, gamma + 1 - lo, 128)
    with pytest.raises(ValueError):
        sv.lazy_groups(0, 7, 1000, f32)
    assert sv.spec_verify_lazy_groups(1, 257, 1000, f32, ctypes.addressof((ctypes.c_int32 * 8)())) == 0


def test_workspace_size_monotone_and_invalid(lib):
    a = sv.spec_verify_workspace_size(8, 7, 151936)
    b = sv.spec_verify_workspace_size(64, 7, 151936)
    c = sv.spec_verify_workspace_size(64, 7, 128256)
    assert 0 < a < b and c <= b and a % 256 == 0
    assert sv.spec_verify_workspace_size(-1, 7, 10) == 0
    assert sv.spec_verify_workspace_size(1, 7, 0) == 0
    assert sv.spec_verify_workspace_size(0, 7, 10) > 0


def test_status_strings(lib):
    for s in range(7):
        assert sv.spec_verify_status_string(s)
    assert "unknown" in sv.spec_verify_status_string(99)


FAKE = 1 << 20          # an aligned address that is never dereferenced
WS = 1 << 24


def call_sample(**kw):
    a = dict(target=FAKE, draft=FAKE, dtype=sv.SPEC_DTYPE_BF16, draft_tokens=FAKE, uniforms=FAKE,
             temperature=1.0, B=2, gamma=3, V=100, out_tokens=FAKE, out_num_accepted=FAKE,
             out_logprobs=None, ws=WS, ws_bytes=0, stream=None)
    a.update(kw)
    return sv.spec_verify_sample(a["target"], a["draft"], a["dtype"], a["draft_tokens"],
                                 a["uniforms"], a["temperature"], a["B"], a["gamma"], a["V"],
                                 a["out_tokens"], a["out_num_accepted"], a["out_logprobs"], a["ws"],
                                 a["ws_bytes"], a["stream"])


def test_sample_argument_checks(lib):
    assert call_sample(dtype=7) == sv.SPEC_ERR_UNSUPPORTED_DTYPE
    assert call_sample(B=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(gamma=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(gamma=257) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(V=0) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(temperature=0.0) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(temperature=-1.0) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(temperature=float("inf")) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(temperature=float("nan")) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(B=0) == sv.SPEC_OK                    # empty batch: nothing launched
    assert call_sample(target=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(draft=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(draft_tokens=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(uniforms=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(out_tokens=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(target=FAKE + 8) == sv.SPEC_ERR_MISALIGNED
    assert call_sample(draft=FAKE + 2) == sv.SPEC_ERR_MISALIGNED
    assert call_sample(ws=None) == sv.SPEC_ERR_INVALID_ARG
    assert call_sample(ws=WS + 16) == sv.SPEC_ERR_MISALIGNED
    need = sv.spec_verify_workspace_size(2, 3, 100)
    assert call_sample(ws_bytes=need - 1) == sv.SPEC_ERR_WORKSPACE_TOO_SMALL


def test_lazy_sample_shares_the_argument_checks(lib):
    f = sv.spec_verify_sample_lazy
    ok = dict(t=FAKE, d=FAKE, dt=sv.SPEC_DTYPE_BF16, x=FAKE, u=FAKE, T=1.0, B=2, g=3, V=100,
              tok=FAKE, acc=FAKE, lp=None, ws=WS, wb=1 << 24)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["t"], a["d"], a["dt"], a["x"], a["u"], a["T"], a["B"], a["g"], a["V"], a["tok"],
                 a["acc"], a["lp"], a["ws"], a["wb"], None)
    assert call(dt=3) == sv.SPEC_ERR_UNSUPPORTED_DTYPE
    assert call(g=300) == sv.SPEC_ERR_INVALID_ARG
    assert call(T=0.0) == sv.SPEC_ERR_INVALID_ARG
    assert call(u=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(x=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(t=FAKE + 2) == sv.SPEC_ERR_MISALIGNED
    assert call(wb=16) == sv.SPEC_ERR_WORKSPACE_TOO_SMALL
    assert call(B=0) == sv.SPEC_OK


def test_topk_argument_checks(lib):
    k = sv.spec_topk_exclude
    need = sv.spec_topk_workspace_size(3, 100, 4)
    assert need > 256
    assert sv.spec_topk_workspace_size(3, 100, 9) == 0            # K outside 1..8
    assert sv.spec_topk_workspace_size(3, 100, 8) >= sv.spec_topk_workspace_size(3, 100, 4)
    assert k(FAKE, 9, 3, 100, 4, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_UNSUPPORTED_DTYPE
    assert k(FAKE, 0, 3, 100, 0, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE, 0, 3, 100, 9, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE, 0, -1, 100, 4, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE, 0, 3, 0, 4, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE, 0, 0, 100, 4, None, FAKE, None, WS, need, None) == sv.SPEC_OK
    assert k(None, 0, 3, 100, 4, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE, 0, 3, 100, 4, None, None, None, WS, need, None) == sv.SPEC_ERR_INVALID_ARG
    assert k(FAKE + 4, 0, 3, 100, 4, None, FAKE, None, WS, need, None) == sv.SPEC_ERR_MISALIGNED
    assert k(FAKE, 0, 3, 100, 4, None, FAKE, None, WS + 64, need, None) == sv.SPEC_ERR_MISALIGNED
    assert k(FAKE, 0, 3, 100, 4, None, FAKE, None, WS, need - 1, None) == \
        sv.SPEC_ERR_WORKSPACE_TOO_SMALL


def test_greedy_and_tree_argument_checks(lib):
    g = sv.spec_verify_greedy
    assert g(FAKE, 5, FAKE, 1, 1, 10, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_UNSUPPORTED_DTYPE
    assert g(FAKE, 0, FAKE, 1, -1, 10, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert g(FAKE, 0, None, 1, 2, 10, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert g(FAKE + 4, 0, FAKE, 1, 2, 10, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_MISALIGNED
    assert g(FAKE, 0, FAKE, 1, 2, 10, FAKE, FAKE, WS, 16, None) == sv.SPEC_ERR_WORKSPACE_TOO_SMALL
    assert g(FAKE, 0, FAKE, 0, 2, 10, FAKE, FAKE, WS, 16, None) == sv.SPEC_OK
    t = sv.spec_verify_tree_greedy
    assert t(FAKE, 1, FAKE, FAKE, 1, 0, 10, FAKE, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 1, FAKE, FAKE, 1, 1025, 10, FAKE, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 1, None, FAKE, 1, 4, 10, FAKE, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 1, FAKE, FAKE, 1, 4, 10, None, FAKE, FAKE, WS, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 1, FAKE, FAKE, 1, 4, 10, FAKE, FAKE, FAKE, WS, 8, None) == sv.SPEC_ERR_WORKSPACE_TOO_SMALL
    assert sv.spec_verify_workspace_init(None, 10, None) == sv.SPEC_ERR_INVALID_ARG
    st, _ = sv.spec_verify_read_error(None, None)
    assert st == sv.SPEC_ERR_INVALID_ARG


def test_product_package_does_not_reach_the_oracle():
    """The product path never imports the oracle (test infrastructure)."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_59_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle.h" not in src, f


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(sv, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(ImportError):
        sv.load_library()


def test_tensor_helpers_reject_bad_tensors():
    """The tensor-level helpers check device, dtype, shape and contiguity
    before anything reaches the C ABI (which would read raw memory)."""
    torch = pytest.importorskip("torch")
    z = torch.zeros((2, 4, 64))
    x = torch.zeros((2, 3), dtype=torch.int32)
    u = torch.zeros((2, 4))
    with pytest.raises(ValueError, match="CUDA"):
        sv.verify_sample(z, z[:, :3], x, u, 1.0)
    with pytest.raises(TypeError, match="torch tensor"):
        sv.verify_greedy(z.numpy(), x)
    with pytest.raises(ValueError, match="CUDA"):
        sv.verify_tree_greedy(z, x, x)
    with pytest.raises(ValueError, match="CUDA"):
        sv.topk_exclude(z.reshape(8, 64), 4)
    with pytest.raises(ValueError, match="CUDA"):
        sv.ngram_retrieve(torch.zeros((2, 8), dtype=torch.int32), torch.zeros(2, dtype=torch.int32),
                          3, 7, 16)
    with pytest.raises(ValueError, match="CUDA"):
        sv.cosine_topk(z, z[:, 0], 4)
    # dtype and shape are checked the same way (on the first, CUDA-independent, failing
    # property): a mistyped logits tensor is a TypeError
    with pytest.raises((TypeError, ValueError)):
        sv.verify_sample(z.to(torch.float64), z[:, :3], x, u, 1.0)
