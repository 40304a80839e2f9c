"""Element scans inside PyTorch graphs: gradients through
``element_scan_recurrences_gb300.autograd.element_scan`` (forward and
backward in the library's kernels) against the gradient oracles.

"Precision and gradients": gradients flow to `initial` and every sequence;
a broadcast parameter's gradient sums its contributions across time and the
other broadcast axes; repeated sequence arguments accumulate."""
import numpy as np
import pytest
import torch

from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300.autograd import element_scan
from oracle.body import scan_body
from oracle.body_grad import scan_body_backward

pytestmark = pytest.mark.gpu

RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()


def close(got, want, what, exact=False):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if exact:
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), what
        return
    err = np.abs(got.astype(np.float64) - want) / (1.0 + np.abs(want.astype(np.float64)))
    assert float(err.max()) <= RTOL, "%s: max scaled error %.3g" % (what, float(err.max()))


def _leaf(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda().requires_grad_(True)


def test_builtin_body_gradients():
    """TANH_DECAY through autograd equals the fixed-body gradient oracle."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 40, 64)).astype(np.float32)
    a = rng.uniform(0.5, 0.99, (2, 40, 64)).astype(np.float32)
    h0 = rng.standard_normal((2, 64)).astype(np.float32)
    G = rng.standard_normal((2, 40, 64)).astype(np.float32)
    ti, tx, ta = _leaf(h0), _leaf(x), _leaf(a)
    out = element_scan("tanh_decay", ti, [tx, ta], axis=1)
    (out * torch.from_numpy(G).cuda()).sum().backward()
    st = oracle.scan(es.TANH_DECAY, h0, [x, a], axis=1)
    wi, (wx, wa) = oracle.scan_backward(es.TANH_DECAY, h0, [x, a], st, G, axis=1)
    # the library's forward states (CUDA tanhf) feed its backward: within tolerance
    close(ti.grad.cpu(), wi, "initial")
    close(tx.grad.cpu(), wx, "x")
    close(ta.grad.cpu(), wa, "a")


@pytest.mark.parametrize("reverse", [False, True])
def test_body_program_gradients(reverse):
    text = "(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))"
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 50, 40)).astype(np.float32)
    a = rng.uniform(0.5, 0.99, x.shape).astype(np.float32)
    g = rng.uniform(0, 1, x.shape).astype(np.float32)
    h0 = rng.standard_normal((3, 40)).astype(np.float32)
    G = rng.standard_normal(x.shape).astype(np.float32)
    leaves = [_leaf(v) for v in (h0, x, a, g)]
    out = element_scan(text, leaves[0], leaves[1:], axis=1, reverse=reverse)
    (out * torch.from_numpy(G).cuda()).sum().backward()
    st = scan_body(text, h0, [x, a, g], axis=1, reverse=reverse)
    close(out.detach().cpu(), st, "states")
    wi, ws = scan_body_backward(text, h0, [x, a, g], st, G, axis=1, reverse=reverse)
    for t, w, nm in zip(leaves, [wi] + ws, ["initial", "x", "a", "g"]):
        close(t.grad.cpu(), w, nm)


def test_broadcast_parameter_sums_over_time_and_lanes():
    """A decay shared by every trip and lane, broadcast before the call: its
    gradient is the sequence gradient summed over time and lanes."""
    text = "(lambda (h x a) (+ (* a h) x))"
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 30, 36)).astype(np.float32)
    h0 = rng.standard_normal((2, 36)).astype(np.float32)
    G = rng.standard_normal(x.shape).astype(np.float32)
    decay = torch.tensor([0.9], device="cuda", requires_grad=True)
    tx, ti = _leaf(x), _leaf(h0)
    a_full = decay.expand(x.shape)            # the broadcast before the call
    out = element_scan(text, ti, [tx, a_full], axis=1)
    (out * torch.from_numpy(G).cuda()).sum().backward()
    a = np.full(x.shape, 0.9, np.float32)
    st = scan_body(text, h0, [x, a], axis=1)
    wi, (wx, wa) = scan_body_backward(text, h0, [x, a], st, G, axis=1)
    close(tx.grad.cpu(), wx, "x", exact=True)
    got = float(decay.grad.cpu()[0])
    want = float(np.sum(wa.astype(np.float64)))
    assert abs(got - want) <= 1e-4 * (1 + abs(want)), (got, want)


def test_repeated_sequence_argument_accumulates():
    text = "(lambda (h x y) (+ (* 0.5 h) (* x y)))"
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 20, 32)).astype(np.float32)
    h0 = rng.standard_normal((2, 32)).astype(np.float32)
    G = rng.standard_normal(x.shape).astype(np.float32)
    tx, ti = _leaf(x), _leaf(h0)
    out = element_scan(text, ti, [tx, tx], axis=1)
    (out * torch.from_numpy(G).cuda()).sum().backward()
    st = scan_body(text, h0, [x, x], axis=1)
    _, (g1, g2) = scan_body_backward(text, h0, [x, x], st, G, axis=1)
    close(tx.grad.cpu(), g1 + g2, "x read twice")


def test_vector_state_and_upstream_graph():
    """A NORMCAP body over a projection of the inputs: gradients reach the
    projection's weight through the scan."""
    text = ("(lambda (h x a) (let ((y (+ (* a h) x))) "
            "(/ y (maximum 1.0 (sqrt (sum (* y y) :axes [-1]))))))")
    torch.manual_seed(4)
    z = torch.randn(2, 24, 16, 8, device="cuda")
    Wt = torch.randn(8, 16, device="cuda", requires_grad=True)
    gate = torch.rand(2, 24, 16, 1, device="cuda") * 0.5 + 0.5
    h0 = torch.zeros(2, 16, 16, device="cuda")
    x = z @ Wt                                  # [2, 24, 16, 16]
    out = element_scan(text, h0, [x, gate], axis=1, state_axis=True)
    G = torch.randn_like(out)
    (out * G).sum().backward()
    xs = x.detach().cpu().numpy()
    st = scan_body(text, h0.cpu().numpy(), [xs, gate.cpu().numpy()], axis=1, state_axis=True)
    _, (gx, _) = scan_body_backward(text, h0.cpu().numpy(), [xs, gate.cpu().numpy()], st, G.cpu().numpy(),
                                    axis=1, state_axis=True)
    want = np.einsum("otjk,otjn->kn", z.cpu().numpy().astype(np.float64), gx.astype(np.float64))
    err = np.abs(Wt.grad.cpu().numpy() - want) / (1 + np.abs(want))
    assert float(err.max()) <= 1e-4, float(err.max())
