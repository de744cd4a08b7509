"""The bounded waits' timeout path, driven without breaking a kernel.

spec_verify_set_wait_limit(0) makes every wait of the streaming kernels on
their bulk-copy ring give up without polling: the consumers skip their work,
the producer stops issuing copies and waits for those in flight, and the call
returns with SPEC_DEVERR_TIMEOUT in the workspace error word.  With the
default limit restored, the same workspace gives the oracle's results again
and a clear error word.  One row of 32 KB per position keeps the calls tiny.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_59_gb300 import workloads as W

from parity import compare_exact, compare_sample

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def test_wait_limit_zero_times_out_then_recovers(sv):
    default = sv.spec_verify_default_wait_limit()
    assert default > 0
    x = W.make_chain("chain-b8", B=2, gamma=1, V=16384)
    zt = torch.from_numpy(x.target).cuda().to(torch.bfloat16)
    zd = torch.from_numpy(x.draft).cuda().to(torch.bfloat16)
    xt = torch.from_numpy(x.draft_tokens).cuda()
    u = torch.from_numpy(x.uniforms).cuda()
    ws = sv.Workspace()
    ws.get(x.B, x.gamma + 1, x.V)
    sv.spec_verify_set_wait_limit(0)
    try:
        sv.verify_greedy(zt, xt, workspace=ws)
        torch.cuda.synchronize()
        assert ws.read_error() & sv.SPEC_DEVERR_TIMEOUT
        sv.verify_sample(zt, zd, xt, u, x.T, workspace=ws)
        torch.cuda.synchronize()
        assert ws.read_error() & sv.SPEC_DEVERR_TIMEOUT
    finally:
        sv.spec_verify_set_wait_limit(default)
    tok, acc = sv.verify_greedy(zt, xt, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(x.target, x.draft_tokens)
    assert not compare_exact("tokens", tok.cpu().numpy(), ref["tokens"])
    assert not compare_exact("accepted", acc.cpu().numpy(), ref["accepted"])
    tok, acc, lp = sv.verify_sample(zt, zd, xt, u, x.T, logprobs=True, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.verify_sample(x.target, x.draft, x.draft_tokens, x.uniforms, x.T,
                               want_logprob=True, want_ratio=True, want_cdf=True)
    res = compare_sample(tok.cpu().numpy(), acc.cpu().numpy(), ref, x.draft_tokens, x.uniforms,
                         gpu_lp=lp.cpu().numpy())
    assert not res["failures"], res["failures"]
    assert ws.read_error() == 0
