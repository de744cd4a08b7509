"""Whatever a workspace holds before a call -- an earlier call of another
shape, an aborted call, or bytes that were never written by the library --
the call's results are those of a freshly zeroed workspace, bit for bit.

The sampling path reads its partials, SampleDescs and segment sums as tagged
words while their writers may still run, and every stream claims chunks from
a tagged counter; a workspace filled with all-ones bytes holds the largest
possible tag in every counter, which no launch can raise, so the calls must
install their own tags by compare-and-swap (the path otherwise taken only when
the process's launch-tag count wraps)."""
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


def dev_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def sample(sv, x, ws, lazy=False):
    out = sv.verify_sample(dev_logits(x.target, x.dtype), dev_logits(x.draft, x.dtype),
                           dev(x.draft_tokens), dev(x.uniforms), x.T, logprobs=True,
                           workspace=ws, lazy=lazy)
    torch.cuda.synchronize()
    return [t.cpu() for t in out]


def greedy(sv, x, ws):
    out = sv.verify_greedy(dev_logits(x.target, x.dtype), dev(x.draft_tokens), workspace=ws)
    torch.cuda.synchronize()
    return [t.cpu() for t in out]


def spoil(ws, fill, seed=7):
    """Overwrite everything but the error word with fill (a byte value or
    'random')."""
    buf = ws.buf
    if fill == "random":
        g = torch.Generator(device="cpu").manual_seed(seed)
        buf[4:] = torch.randint(0, 256, (buf.numel() - 4,), generator=g, dtype=torch.uint8).cuda()
    else:
        buf[4:] = fill
    torch.cuda.synchronize()


def same(a, b):
    """Bit-equal tensors (NaN log-probabilities of unread positions included)."""
    def bits(t):
        return t.view(torch.int32) if t.dtype == torch.float32 else t
    return all(torch.equal(bits(p), bits(q)) for p, q in zip(a, b))


SHAPES = [("chain-b64", dict(B=6, V=30000)), ("chain-b8", dict(B=3, gamma=2, V=151936)),
          ("chain-b256", dict(B=9, V=4096)), ("chain-small", dict())]


@pytest.mark.parametrize("fill", [0xFF, 0x00, 0x5A, "random"])
@pytest.mark.parametrize("lazy", [False, True])
def test_sample_after_spoiled_workspace(sv, fill, lazy):
    for name, kw in SHAPES:
        x = W.make_chain(name, **kw)
        ref = sample(sv, x, sv.Workspace(), lazy=lazy)
        ws = sv.Workspace()
        ws.get(x.B, x.gamma, x.V)
        spoil(ws, fill)
        got = sample(sv, x, ws, lazy=lazy)
        assert same(ref, got), (name, fill, lazy)
        assert ws.read_error() == 0, (name, fill)
        got2 = sample(sv, x, ws, lazy=lazy)            # and the call after it
        assert same(ref, got2), (name, fill, lazy)


@pytest.mark.parametrize("fill", [0xFF, "random"])
def test_greedy_after_spoiled_workspace(sv, fill):
    for name, kw in SHAPES:
        x = W.make_chain(name, **kw)
        ref = greedy(sv, x, sv.Workspace())
        ws = sv.Workspace()
        ws.get(x.B, x.gamma, x.V)
        spoil(ws, fill)
        assert same(ref, greedy(sv, x, ws)), (name, fill)
        assert ws.read_error() == 0


def tree(sv, t, ws):
    out = sv.verify_tree_greedy(dev_logits(t.target, t.dtype), dev(t.node_tokens), dev(t.parents),
                                workspace=ws)
    torch.cuda.synchronize()
    return [q.cpu() for q in out]


@pytest.mark.parametrize("fill", [0xFF, "random"])
def test_tree_after_spoiled_workspace(sv, fill):
    """Trees decided beside the stream (up to 32 nodes) and after it (more)."""
    for kw in (dict(B=6, V=30000, depth=3, branches=1), dict(B=4, V=30000),
               dict(B=3, V=151936, depth=2, branches=0)):
        t = W.make_tree("tree-b32", **kw)
        ref = tree(sv, t, sv.Workspace())
        ws = sv.Workspace()
        ws.get(t.B, t.N, t.V)
        spoil(ws, fill)
        assert same(ref, tree(sv, t, ws)), (kw, fill)
        assert ws.read_error() == 0


def test_one_workspace_across_shapes_and_modes(sv):
    """One workspace, calls of changing shape and mode in turn: each result
    equals the same call on a fresh workspace."""
    ws = sv.Workspace()
    ws.get(64, 7, 151936)
    order = [("chain-b64", dict(B=20, V=151936), "sample"), ("chain-b8", dict(B=2, V=30000), "greedy"),
             ("chain-b64", dict(B=7, gamma=3, V=50000), "sample"), ("chain-b256", dict(B=40, V=2048), "lazy"),
             ("chain-b64", dict(B=20, V=151936), "sample"), ("chain-small", dict(), "sample"),
             ("chain-b8", dict(B=8, V=151936), "lazy"), ("chain-b64", dict(B=1, gamma=1, V=3000), "greedy")]
    for i, (name, kw, mode) in enumerate(order):
        x = W.make_chain(name, seed=100 + i, **kw)
        if mode == "greedy":
            ref, got = greedy(sv, x, sv.Workspace()), greedy(sv, x, ws)
        else:
            ref, got = sample(sv, x, sv.Workspace(), lazy=mode == "lazy"), sample(sv, x, ws, lazy=mode == "lazy")
        assert same(ref, got), (i, name, kw, mode)
    assert ws.read_error() == 0
