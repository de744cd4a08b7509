"""spec_verify_sample_noalloc: the entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns all
device memory, or a decode loop that must not call cudaMalloc mid-step).  It
takes no workspace; its scratch is a fixed array inside the library.

Checked through the C ABI against spec_verify_sample (the workspace entry
point) on two calls in a row, which share that one array.  Collected last so
that a failure here cannot hide the other tests' results; passes on its own
in a fresh process as well."""
import numpy as np
import pytest

from speculative_decoding_verification_59_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def _inputs(x):
    dt = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    zt = torch.from_numpy(x.target).cuda().to(dt)
    zd = torch.from_numpy(x.draft).cuda().to(dt)
    xt = torch.from_numpy(x.draft_tokens).cuda()
    u = torch.from_numpy(x.uniforms).cuda()
    return zt, zd, xt, u


def _outputs(x):
    tok = torch.full((x.B, x.gamma + 1), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((x.B,), -7, dtype=torch.int32, device="cuda")
    lp = torch.zeros((x.B, x.gamma, 2), dtype=torch.float32, device="cuda")
    return tok, acc, lp


def _code(sv, x):
    return sv.SPEC_DTYPE_BF16 if x.dtype == "bf16" else sv.SPEC_DTYPE_F32


def test_noalloc_matches_workspace_entry_point_twice(sv):
    """Two consecutive calls with different shapes and dtypes: tokens and
    accept counts equal, log-probabilities within the 1e-5 relative bar of
    the parity tests (the same kernels run, so they are in fact identical)."""
    stream = torch.cuda.current_stream().cuda_stream
    cases = [W.make_chain("chain-b64", B=8, V=151936), W.make_chain("chain-b256", B=256, V=128256)]
    for x in cases:
        zt, zd, xt, u = _inputs(x)
        need = sv.spec_verify_workspace_size(x.B, x.gamma, x.V)
        assert need <= sv.SPEC_VERIFY_NOALLOC_SCRATCH_BYTES
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        ref_tok, ref_acc, ref_lp = _outputs(x)
        st = sv.spec_verify_sample(zt.data_ptr(), zd.data_ptr(), _code(sv, x), xt.data_ptr(),
                                   u.data_ptr(), x.T, x.B, x.gamma, x.V, ref_tok.data_ptr(),
                                   ref_acc.data_ptr(), ref_lp.data_ptr(), ws.data_ptr(), need,
                                   stream)
        assert st == sv.SPEC_OK
        tok, acc, lp = _outputs(x)
        st = sv.spec_verify_sample_noalloc(zt.data_ptr(), zd.data_ptr(), _code(sv, x),
                                           xt.data_ptr(), u.data_ptr(), x.T, x.B, x.gamma, x.V,
                                           tok.data_ptr(), acc.data_ptr(), lp.data_ptr(), stream)
        assert st == sv.SPEC_OK
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok)
        assert torch.equal(acc, ref_acc)
        assert (acc >= 0).all() and (tok[:, 0] >= 0).all()
        rel = ((lp.double().exp() - ref_lp.double().exp()).abs() /
               ref_lp.double().exp().clamp_min(1e-300))
        assert float(rel.max()) <= 1e-5


def test_noalloc_rejects_problems_beyond_its_scratch(sv):
    """A problem whose scratch need exceeds the fixed array is refused on the
    host with SPEC_ERR_EXCEEDS_STATIC_SCRATCH; nothing is launched."""
    B, gamma, V = 4096, 7, 151936
    assert sv.spec_verify_workspace_size(B, gamma, V) > sv.SPEC_VERIFY_NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    st = sv.spec_verify_sample_noalloc(fake, fake, sv.SPEC_DTYPE_BF16, fake, fake, 1.0, B, gamma,
                                       V, fake, fake, None, None)
    assert st == sv.SPEC_ERR_EXCEEDS_STATIC_SCRATCH
    assert "scratch" in sv.spec_verify_status_string(st)


def test_noalloc_bad_sequence_then_valid_call(sv):
    """A draft token outside [0, V) marks only its own sequence (-1 count and
    tokens); the shared array keeps the device error bits this entry point
    never reads, and the next valid call on the same stream still equals
    spec_verify_sample bit for bit."""
    stream = torch.cuda.current_stream().cuda_stream
    x = W.make_chain("chain-b64", B=6, V=20000)
    x.draft_tokens = x.draft_tokens.copy()
    x.draft_tokens[2, 3] = x.V
    zt, zd, xt, u = _inputs(x)
    tok, acc, lp = _outputs(x)
    st = sv.spec_verify_sample_noalloc(zt.data_ptr(), zd.data_ptr(), _code(sv, x), xt.data_ptr(),
                                       u.data_ptr(), x.T, x.B, x.gamma, x.V, tok.data_ptr(),
                                       acc.data_ptr(), lp.data_ptr(), stream)
    assert st == sv.SPEC_OK
    torch.cuda.synchronize()
    a = acc.cpu().numpy()
    assert a[2] == -1 and (tok[2] == -1).all()
    assert (np.delete(a, 2) >= 0).all()

    y = W.make_chain("chain-b64", B=6, V=20000, seed=77)
    zt, zd, xt, u = _inputs(y)
    need = sv.spec_verify_workspace_size(y.B, y.gamma, y.V)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ref_tok, ref_acc, ref_lp = _outputs(y)
    assert sv.spec_verify_sample(zt.data_ptr(), zd.data_ptr(), _code(sv, y), xt.data_ptr(),
                                 u.data_ptr(), y.T, y.B, y.gamma, y.V, ref_tok.data_ptr(),
                                 ref_acc.data_ptr(), ref_lp.data_ptr(), ws.data_ptr(), need,
                                 stream) == sv.SPEC_OK
    tok, acc, lp = _outputs(y)
    assert sv.spec_verify_sample_noalloc(zt.data_ptr(), zd.data_ptr(), _code(sv, y),
                                         xt.data_ptr(), u.data_ptr(), y.T, y.B, y.gamma, y.V,
                                         tok.data_ptr(), acc.data_ptr(), lp.data_ptr(),
                                         stream) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert torch.equal(tok, ref_tok) and torch.equal(acc, ref_acc) and torch.equal(lp, ref_lp)
