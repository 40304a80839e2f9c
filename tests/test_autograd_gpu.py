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


def test_matrix_scan_gradients_and_shared_operand():
    """matrix-scan through autograd: the delta rule's a and b built from
    k, v, beta; gradients reach k, v and beta (checked against an f64 torch
    loop), and a shared `a` (broadcast over the batch) sums its gradient."""
    from element_scan_recurrences_gb300.autograd import matrix_scan
    torch.manual_seed(6)
    B, T, n, m = 2, 33, 8, 4
    k = torch.nn.functional.normalize(torch.randn(B, T, n, device="cuda"), dim=-1).requires_grad_(True)
    v = torch.randn(B, T, m, device="cuda", requires_grad=True)
    beta = torch.rand(B, T, 1, 1, device="cuda", requires_grad=True)
    eye = torch.eye(n, device="cuda")
    a = eye - beta * k.unsqueeze(-1) * k.unsqueeze(-2)
    b = beta * k.unsqueeze(-1) * v.unsqueeze(-2)
    S = matrix_scan(a, b, axis=1)
    G = torch.randn_like(S)
    (S * G).sum().backward()
    # the same in f64 with torch.matmul
    k64, v64, b64 = (t.detach().double().requires_grad_(True) for t in (k, v, beta))
    a64 = torch.eye(n, dtype=torch.float64, device="cuda") - b64 * k64.unsqueeze(-1) * k64.unsqueeze(-2)
    bb64 = b64 * k64.unsqueeze(-1) * v64.unsqueeze(-2)
    h = torch.zeros(B, n, m, dtype=torch.float64, device="cuda")
    outs = []
    for t in range(T):
        h = a64[:, t] @ h + bb64[:, t]
        outs.append(h)
    (torch.stack(outs, 1) * G.double()).sum().backward()
    for got, want, nm in ((k.grad, k64.grad, "k"), (v.grad, v64.grad, "v"), (beta.grad, b64.grad, "beta")):
        err = (got.double() - want).abs() / (1 + want.abs())
        assert float(err.max()) < 1e-4, (nm, float(err.max()))
    # a shared by both sequences: its gradient is the sum of theirs
    a1 = (torch.randn(1, T, n, n, device="cuda") * 0.3).requires_grad_(True)
    bb = torch.randn(B, T, n, m, device="cuda")
    out = matrix_scan(a1, bb, axis=1)
    Gs = torch.randn_like(out)
    (out * Gs).sum().backward()
    A = a1.detach().expand(B, T, n, n).contiguous()
    ga, _ = es.matrix_scan_backward(A, bb, es.matrix_scan(A, bb, axis=1), Gs.contiguous(), axis=1)
    assert torch.allclose(a1.grad[0], ga.sum(0), rtol=1e-5, atol=1e-5)
    # a projective scan has no gradient
    ap = a1.detach().expand(B, T, n, n).contiguous().requires_grad_(True)
    outp = matrix_scan(ap, bb, axis=1, projective=True)
    with pytest.raises(es.EsError):
        outp.sum().backward()


def test_linear_scan_gradients():
    from element_scan_recurrences_gb300.autograd import linear_scan
    import oracle.matrix as M
    rng = np.random.default_rng(7)
    a = rng.uniform(0.5, 0.99, (3, 50, 40)).astype(np.float32)
    b = rng.standard_normal((3, 50, 40)).astype(np.float32)
    G = rng.standard_normal((3, 50, 40)).astype(np.float32)
    ta, tb = _leaf(a), _leaf(b)
    out = linear_scan(ta, tb, axis=1)
    (out * torch.from_numpy(G).cuda()).sum().backward()
    st = M.linear_scan(a, b, axis=1)
    wa, wb = M.linear_scan_backward(a, b, st, G, axis=1)
    close(ta.grad.cpu(), wa, "a", exact=True)
    close(tb.grad.cpu(), wb, "b", exact=True)


def test_matrix_scan_chunked_gradients():
    """matrix-scan through autograd with ``chunked=True`` on few long lanes:
    the delta rule's k, v, beta gradients within tolerance of the sequential
    autograd gradients (the chunked forward and gradient reassociate the
    chains), with the chunked paths actually taken."""
    from element_scan_recurrences_gb300.autograd import matrix_scan
    torch.manual_seed(7)
    B, T, n, m = 2, 3000, 16, 16
    assert es.matrix_scan_workspace((B, T, n, n), (B, T, n, m), 1) > 0
    k0 = torch.nn.functional.normalize(torch.randn(B, T, n, device="cuda"), dim=-1)
    v0 = torch.randn(B, T, m, device="cuda")
    beta0 = torch.rand(B, T, 1, 1, device="cuda")
    G = torch.randn(B, T, n, m, device="cuda")
    grads = []
    for chunked in (False, True):
        k, v, beta = (t.clone().requires_grad_(True) for t in (k0, v0, beta0))
        a = torch.eye(n, device="cuda") - beta * k.unsqueeze(-1) * k.unsqueeze(-2)
        b = beta * k.unsqueeze(-1) * v.unsqueeze(-2)
        n0 = es.launch_count()
        S = matrix_scan(a, b, axis=1, chunked=chunked)
        (S * G).sum().backward()
        es.device_status()
        launches = es.launch_count() - n0
        # the sequential gradient runs in min(8, T // 128) windows of a scan
        # and a grad_a launch each
        windows = min(8, T // 128)
        assert launches == (3 + 4 if chunked else 1 + 2 * windows), launches
        grads.append((S.detach().cpu().numpy(), k.grad.cpu().numpy(), v.grad.cpu().numpy(),
                      beta.grad.cpu().numpy()))
    for seq, chk, nm in zip(grads[0], grads[1], ("states", "k", "v", "beta")):
        close(chk, seq, "chunked %s" % nm)
