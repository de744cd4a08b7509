"""Logits rewritten in place by a kernel on the same CUDA stream right before
each call, with no host synchronisation anywhere between the rewrites and the
calls: every call must return the oracle's results for the logits of its own
rewrite.

The streaming kernels prefetch their first chunks into L2 before they wait on
the kernel before them (on streams of 1024 chunks or more, which every call
here is: 2400 sampling chunks, 1280 for greedy, tree and top-K), and they copy
the logits only after that wait.  The rewriting kernels here do not release
their dependents early, so this checks the ordering of the copies behind the
rewrite, for every kind of call, and that a prefetch of the old values never
reaches a result."""
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


def chain_tree(x):
    """The drafts as a chain-shaped tree: node 0 the root, node i + 1 carrying
    draft x_i under node i."""
    B, g = x.draft_tokens.shape
    par = np.tile(np.arange(-1, g, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.full((B, 1), -1, np.int32), x.draft_tokens], axis=1)
    return np.ascontiguousarray(tok), np.ascontiguousarray(par)


def test_logits_rewritten_before_each_call(sv):
    xs = [W.make_chain("chain-b8", B=16, seed=s) for s in (101, 202)]
    zt_src = [torch.from_numpy(x.target).cuda().to(torch.bfloat16) for x in xs]
    zd_src = [torch.from_numpy(x.draft).cuda().to(torch.bfloat16) for x in xs]
    zt = torch.empty_like(zt_src[0])
    zd = torch.empty_like(zd_src[0])
    one = torch.ones((), dtype=torch.bfloat16, device="cuda")
    ws = sv.Workspace()
    order = (0, 1, 0, 1)

    def rewrite(i):
        torch.mul(zt_src[i], one, out=zt)          # elementwise kernels, same stream
        torch.mul(zd_src[i], one, out=zd)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    inputs = []
    for x in xs:
        tt, tp = chain_tree(x)
        rows = x.B * (x.gamma + 1)
        ex = np.concatenate([x.draft_tokens, np.full((x.B, 1), -1, np.int32)], axis=1).reshape(rows)
        inputs.append(dict(xt=dev(x.draft_tokens), u=dev(x.uniforms), gt=dev(x.greedy_tokens),
                           tt=dev(tt), tp=dev(tp), ex=dev(ex), tt_np=tt, tp_np=tp, ex_np=ex))
    torch.cuda.synchronize()

    outs = []
    for i in order:
        x, d = xs[i], inputs[i]
        rewrite(i)
        s = sv.verify_sample(zt, zd, d["xt"], d["u"], x.T, logprobs=True, workspace=ws)
        rewrite(1 - i)
        rewrite(i)
        g = sv.verify_greedy(zt, d["gt"], workspace=ws)
        rewrite(1 - i)
        rewrite(i)
        t = sv.verify_tree_greedy(zt, d["tt"], d["tp"], workspace=ws)
        rewrite(1 - i)
        rewrite(i)
        k = sv.topk_exclude(zt.reshape(-1, x.V), 4, d["ex"], values=True, workspace=ws)
        outs.append((i, s, g, t, k))
    torch.cuda.synchronize()

    refs = {}
    for i, (x, d) in enumerate(zip(xs, inputs)):
        refs[i] = dict(
            sample=oracle.verify_sample(x.target, x.draft, x.draft_tokens, x.uniforms, x.T,
                                        want_logprob=True, want_ratio=True, want_cdf=True),
            greedy=oracle.verify_greedy(x.target, x.greedy_tokens),
            tree=oracle.verify_tree_greedy(x.target, d["tt_np"], d["tp_np"]),
            topk=oracle.topk_exclude(x.target.reshape(-1, x.V), 4, d["ex_np"]))
    for i, s, g, t, k in outs:
        x, r = xs[i], refs[i]
        tok, acc, lp = (a.cpu().numpy() for a in s)
        res = compare_sample(tok, acc, r["sample"], x.draft_tokens, x.uniforms, gpu_lp=lp)
        assert not res["failures"], (i, res["failures"][:5])
        f = compare_exact("greedy tokens", g[0].cpu().numpy(), r["greedy"]["tokens"]) + \
            compare_exact("greedy accepted", g[1].cpu().numpy(), r["greedy"]["accepted"]) + \
            compare_exact("tree nodes", t[0].cpu().numpy(), r["tree"]["nodes"]) + \
            compare_exact("tree tokens", t[1].cpu().numpy(), r["tree"]["tokens"]) + \
            compare_exact("tree accepted", t[2].cpu().numpy(), r["tree"]["accepted"]) + \
            compare_exact("top-K tokens", k[0].cpu().numpy(), r["topk"]["idx"])
        assert not f, (i, f)
        assert np.array_equal(k[1].cpu().numpy(), r["topk"]["val"]), i
    assert ws.read_error() == 0
