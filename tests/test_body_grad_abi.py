"""Body-program gradients through the C ABI without a GPU: every backward
kernel compiles for sm_103a (NVRTC on the host), the plan validates the
gradient buffers, and the generated vector-Jacobian product has the
documented derivative rules."""
import re

import pytest

import body_cases
import body_grad_pins
from element_scan_recurrences_gb300 import binding as es


# scalar and vector states, width-one sequences, the most sequences, `max`
# over the state and most operations of the body language
COMPILE_IDS = ["identities", "angle", "eight_seqs", "normcap_w16", "row_max_w8"]


@pytest.mark.parametrize("cid", COMPILE_IDS)
def test_backward_kernel_compiles(cid):
    """NVRTC compiles every backward kernel variant of the signature."""
    c = body_cases.case(cid)
    es.Body(c[1]).prepare_backward(c[2], c[3])


def test_backward_source_for_every_test_body():
    for c in body_cases.CASES:
        assert "static void vjp(" in es.Body(c[1]).source_backward(c[2], c[3])
    for case in body_grad_pins.AUTOGRAD_CASES:
        assert "static void vjp(" in es.Body(case[0]).source_backward(case[2], case[3])


def _ptrs(n):
    return [(k + 1) << 44 for k in range(2 * n + 4)]


def test_backward_plan():
    b = es.Body("(lambda (h x a) (tanh (+ x (* a h))))")
    p = b.plan_backward([3, 100, 64], 1)
    assert p["path"] == "lane_tma" and (p["O"], p["T"], p["J"], p["W"]) == (3, 100, 64, 1)
    # lanes innermost need 32 or more lanes in rows of 16 bytes, 16-byte aligned TMA-read buffers
    assert b.plan_backward([3, 100, 66], 1)["path"] == "generic"
    assert b.plan_backward([3, 100, 16], 1)["path"] == "generic"
    assert b.plan_backward([64, 100], 0)["path"] == "lane_tma"
    assert b.plan_backward([100, 64], -1)["path"] == "time_tma"     # the sequence axis last
    assert b.plan_backward([100, 32], -1)["path"] == "generic"      # one tile of trips only
    assert b.plan_backward([100, 66], -1)["path"] == "generic"      # rows of 16 bytes
    for k in (1, 3, 4):                                   # a sequence, the states, grad_out
        ptrs = _ptrs(2)
        ptrs[k] += 4
        assert b.plan_backward([3, 100, 64], 1, ptrs=ptrs)["path"] == "generic"
    ptrs = _ptrs(2)
    ptrs[6] += 4                                          # a gradient: written by TMA tensor stores
    assert b.plan_backward([3, 100, 64], 1, ptrs=ptrs)["path"] == "generic"
    ptrs = _ptrs(2)
    ptrs[5] += 4                                          # grad_initial: plain stores
    assert b.plan_backward([3, 100, 64], 1, ptrs=ptrs)["path"] == "lane_tma"
    assert b.plan_backward([3, 100, 64], 1, reverse=True)["reverse"]
    v = es.Body(body_cases.NORMCAP_TEXT)
    p = v.plan_backward([2, 10, 5, 16], 1, 16, [16, 1])
    assert p["path"] == "generic" and p["W"] == 16 and p["seq_width"] == (16, 1)
    # no lanes: nothing to do
    assert b.plan_backward([0, 100, 64], 1)["path"] == "empty"


def test_backward_plan_rejects_bad_buffers():
    b = es.Body("(lambda (h x a) (tanh (+ x (* a h))))")
    shape = [3, 100, 64]
    n = 2
    for k in range(n + 3, 2 * n + 4):           # each written buffer onto `states`
        ptrs = _ptrs(n)
        ptrs[k] = ptrs[n + 1] + 64
        with pytest.raises(es.EsError) as e:
            b.plan_backward(shape, 1, ptrs=ptrs)
        assert e.value.status == 3 and "overlaps" in str(e.value)
    ptrs = _ptrs(n)
    ptrs[n + 4] = ptrs[n + 5]                     # two gradients on one buffer
    with pytest.raises(es.EsError) as e:
        b.plan_backward(shape, 1, ptrs=ptrs)
    assert e.value.status == 3
    for k in (n + 2, n + 3, n + 4):               # grad_out, grad_initial, a gradient: null
        ptrs = _ptrs(n)
        ptrs[k] = 0
        with pytest.raises(es.EsError) as e:
            b.plan_backward(shape, 1, ptrs=ptrs)
        assert e.value.status == 3
    ptrs = _ptrs(n)
    ptrs[n + 5] += 2                              # misaligned gradient
    with pytest.raises(es.EsError) as e:
        b.plan_backward(shape, 1, ptrs=ptrs)
    assert e.value.status == 3 and "aligned" in str(e.value)


def test_backward_forced_path():
    b = es.Body("(lambda (h x a) (tanh (+ x (* a h))))")
    for path, shape, status in (("time_tma", [3, 100, 64], 4), ("vec_tma", [3, 100, 64], 4),
                                ("lane_tma", [3, 100, 66], 4), ("mat_tma", [3, 100, 64], 4)):
        es.set_path_override(path)
        try:
            with pytest.raises(es.EsError) as e:
                b.plan_backward(shape, 1)
            assert e.value.status == status
        finally:
            es.set_path_override("auto")
    for path in ("generic", "lane_tma"):
        es.set_path_override(path)
        try:
            assert b.plan_backward([3, 100, 64], 1)["path"] == path
        finally:
            es.set_path_override("auto")


def test_backward_rejects_what_the_forward_rejects():
    with pytest.raises(es.EsError) as e:
        es.Body("(lambda (h x) (+ h (sum x)))").plan_backward([2, 5, 3], 1)
    assert e.value.status == 7 and "reduce" in str(e.value)


def test_vjp_source_has_the_derivative_rules():
    src = es.Body("(lambda (h x a) (tanh (+ x (* a h))))").source_backward()
    assert "static void vjp(" in src
    # tanh: g * (1 - out * out), the trip's result read from the saved states;
    # the product's operands swap
    assert "__fmul_rn(g_v2[e], __fsub_rn(1.0f, __fmul_rn(res[e], res[e])))" in src
    assert "g_sw1[e] = __fmul_rn(g_v0[e], h[e])" in src and "g_h[e] = __fmul_rn(g_v0[e], sw[1][e])" in src
    # nothing of the body is computed again, and x is never read
    vjp = src[src.index("static void vjp("):]
    assert "tanhf" not in vjp and not re.search(r"(?<!d)sw\[0\]", vjp)
    assert "kVjpSeqs = 0x2u" in src and "kVjpRes = true" in src
    # linear-scan's body: the gradient never reads b
    src = es.Body("(lambda (h a b) (+ (* a h) b))").source_backward()
    assert "kVjpSeqs = 0x1u" in src and "kVjpRes = false" in src
    # a body whose derivatives read an intermediate recomputes it (and what it needs)
    src = es.Body("(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))").source_backward()
    vjp = src[src.index("static void vjp("):]
    assert "tanhf" in vjp and "kVjpSeqs = 0x7u" in src
    # a width-one gate of a vector state takes the sum over the state
    src = es.Body("(lambda (h g) (* h g))").source_backward(8, [1])
    assert "es::group_sum<E, G>(c0, mask)" in src and "dsn[0] = g_sn0" in src
    # maximum: the winner takes g, a tie splits it
    src = es.Body("(lambda (h x c) (maximum (- h c) x))").source_backward()
    assert "__fmul_rn(g_v1[e], 0.5f)" in src
    # comparisons and casts carry no gradient; a constant result none at all
    src = es.Body("(lambda (h x) (+ h (cast (> x 0.5) :f32)))").source_backward()
    assert "dsw[0][e] = 0.0f" in src
    src = es.Body("(lambda (h x) 3.0)").source_backward()
    assert "dp[e] = 0.0f" in src


def test_autograd_refuses_cpu_tensors():
    """No CPU fallback: the differentiable scan wants CUDA tensors."""
    torch = pytest.importorskip("torch")
    from element_scan_recurrences_gb300.autograd import element_scan
    x = torch.zeros(2, 5, 3)
    with pytest.raises(TypeError):
        element_scan("(lambda (h x) (+ h x))", torch.zeros(2, 3), [x], axis=1)
    with pytest.raises(TypeError):
        element_scan("tanh_decay", torch.zeros(2, 3), [x, x], axis=1)
