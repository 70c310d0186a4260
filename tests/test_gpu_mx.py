"""MXFP8 Q and K through the C ABI against the oracle's MX format
(``oracle/mx.py``) and GDPA (``oracle/ref.py``).

* gdpa_mx_quantise: E4M3 codes and E8M0 scale bytes bit for bit equal to the
  oracle's quantisation of the same bf16 values, with the format's corner
  cases planted: all-zero blocks, negative zeros, block maxima that saturate
  at 448, exact ties, elements that become E4M3 subnormals or underflow to a
  signed zero, bf16 subnormals and values near bf16's largest.
* gdpa_mx_dequantise: every finite code under scales across the E8M0 range,
  bit for bit equal to the oracle's value rounded to bf16.
* gdpa_fwd_mx / gdpa_bwd_mx: GDPA on the values the MXFP8 tensors stand for,
  i.e. the oracle's GDPA on mx_round_trip(Q) and mx_round_trip(K).
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL, check, max_rel, to_dev
from oracle import mx, ref
from oracle import rmsnorm as rn
from workloads import get_config, make_inputs, offsets_from_lengths

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import recommender_model_attention_gb300 as g
    g.build()
    return g


def _codes(values):
    """E4M3 codes of float64 E4M3 values (the oracle's table, read back)."""
    table = {}
    for c in range(0x7F):                       # positive finite codes
        table[mx.e4m3_value(c)] = c
    v = np.asarray(values, dtype=np.float64)
    mag = np.vectorize(lambda a: table[a], otypes=[np.int64])(np.abs(v).ravel()).reshape(v.shape)
    return (mag | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def _corner_blocks():
    """[n, 32] float32 blocks (exact bf16 values) covering the format's cases."""
    rows = []
    z = np.zeros(32, np.float32)
    rows.append(z.copy())                        # all zero
    nz = z.copy()
    nz[3] = -0.0
    rows.append(nz)                              # negative zero only
    s = np.full(32, 1.0, np.float32)
    s[0] = 1.90625                               # 1.90625 * 2^8 / 2^0 -> past 448: saturates
    s[1] = -1.96875
    rows.append(s)
    t = np.full(32, 0.5, np.float32)             # block max 256 -> E = 0
    t[:8] = [256.0, 1.0625, 1.1875, -1.0625, 2.125, 17.0, 19.0, 0.0]   # ties to even
    t[8:12] = [2.0 ** -8, 3 * 2.0 ** -10, 2.0 ** -11, -2.0 ** -10]      # subnormal / underflow
    rows.append(t)
    u = np.full(32, 3.0e38, np.float32)          # near bf16's largest
    u[1] = -2.5e38
    rows.append(u)
    tiny = np.full(32, 2.0 ** -133, np.float32)  # bf16 subnormals
    tiny[0] = 2.0 ** -126
    tiny[1] = -3 * 2.0 ** -131
    rows.append(tiny)
    mixed = np.full(32, 2.0 ** 100, np.float32)  # tiny elements beside a huge maximum
    mixed[5:10] = [2.0 ** -120, -1e-30, 1.0, -2.0 ** 91, 2.0 ** 90 * 1.0625]
    rows.append(mixed)
    out = np.stack(rows)
    return torch.from_numpy(out).to(torch.bfloat16).float().numpy()


def _random_blocks(seed, n):
    g = np.random.default_rng(seed)
    x = g.standard_normal((n, 32)) * np.exp2(g.integers(-30, 31, size=(n, 1)))
    x[g.random((n, 32)) < 0.05] = 0.0
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()


def test_mx_quantise_bit_exact(gd):
    x = np.concatenate([_corner_blocks(), _random_blocks(1, 4000)])
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), x)   # every input is a bf16 value
    m = gd.mx_quantise(xb.cuda().contiguous())
    torch.cuda.synchronize()
    el, ex = mx.quantise(x.astype(np.float64))
    assert np.array_equal(m.scales.cpu().numpy().reshape(-1), (ex.reshape(-1) + 127).astype(np.uint8))
    got = m.elements.cpu().numpy()
    want = _codes(el)
    bad = np.argwhere(got != want)
    assert bad.size == 0, "first mismatches (block, index): %s got %s want %s" % (
        bad[:5].tolist(), got[tuple(bad[:5].T)], want[tuple(bad[:5].T)])


def test_mx_quantise_tensor_layout(gd):
    # a [T, H, d] tensor: one scale byte per 32 values along d, row by row
    g = np.random.default_rng(2)
    T, H, d = 37, 3, 128
    x = torch.from_numpy(g.standard_normal((T, H, d)).astype(np.float32)).to(torch.bfloat16)
    m = gd.mx_quantise(x.cuda())
    assert tuple(m.elements.shape) == (T, H, d) and tuple(m.scales.shape) == (T, H, d // 32)
    el, ex = mx.quantise(x.float().numpy().astype(np.float64))
    assert np.array_equal(m.scales.cpu().numpy(), (ex + 127).astype(np.uint8))
    assert np.array_equal(m.elements.cpu().numpy(), _codes(el))


def test_mx_dequantise_bit_exact(gd):
    g = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    nb = 2048
    codes = np.concatenate([np.tile(finite, (nb * 32) // finite.size + 1)[:nb * 32]])
    g.shuffle(codes)
    codes = codes.reshape(nb, 32)
    e = g.integers(-127, 120, size=nb).astype(np.int32)
    e[:4] = [-127, -126, 119, 0]
    vals = np.vectorize(mx.e4m3_value)(codes.astype(np.int64))
    want = torch.from_numpy(mx.dequantise(vals, e[:, None])).to(torch.bfloat16)
    m = gd.MX(torch.from_numpy(codes).cuda(), torch.from_numpy((e + 127).astype(np.uint8)[:, None]).cuda())
    got = gd.mx_dequantise(m).cpu()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_mx_round_trip_on_device(gd):
    x = _random_blocks(4, 3000)
    m = gd.mx_quantise(torch.from_numpy(x).to(torch.bfloat16).cuda())
    got = gd.mx_dequantise(m).cpu()
    want = torch.from_numpy(mx.mx_round_trip(x.astype(np.float64))).to(torch.bfloat16)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def _mx_case(seed, lq, lkv, H, d, spread=True):
    g = np.random.default_rng(seed)
    qo, ko = offsets_from_lengths(np.asarray(lq)), offsets_from_lengths(np.asarray(lkv))

    def rows(n):
        x = g.standard_normal((int(n), H, d))
        if spread:   # per-block magnitudes over several binades
            x *= np.exp2(g.integers(-3, 4, size=(int(n), H, d // 32))).repeat(32, axis=-1)
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)

    return to_dev({"q_off": qo, "kv_off": ko, "q": rows(qo[-1]), "k": rows(ko[-1]),
                   "v": rows(ko[-1]), "do": rows(qo[-1])})


def _oracle_inputs(x):
    rq = mx.mx_round_trip(ref.to_f64(x["q"]))
    rk = mx.mx_round_trip(ref.to_f64(x["k"]))
    return rq, rk


def _run_mx(gd, x, H, d, act, alpha=None, kernel="auto", backward=True, mask="none", window=0):
    alpha = d ** -0.5 if alpha is None else alpha
    plan = gd.Plan(x["q_off"], x["kv_off"], H, d, mask=mask, window=window)
    plan.set_kernel(kernel)
    qm, km = gd.mx_quantise(x["q"]), gd.mx_quantise(x["k"])
    o = gd.gdpa_fwd_mx(plan, qm, km, x["v"], alpha=alpha, act=act)
    grads = gd.gdpa_bwd_mx(plan, qm, km, x["v"], x["do"], alpha=alpha, act=act) if backward else None
    plan.check()
    rq, rk = _oracle_inputs(x)
    args = (x["q_off"], x["kv_off"], rq, rk, x["v"])
    errs = {"o": max_rel(ref.to_f64(o), ref.fwd(*args, alpha, act, mask, window))}
    if backward:
        want = ref.bwd(*args, x["do"], alpha, act, mask, window)
        for n, gt, w in zip(("dq", "dk", "dv"), grads, want):
            errs[n] = max_rel(ref.to_f64(gt), w)
    plan.destroy()
    return errs


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("act", ["gelu_erf", "silu", "gelu_taylor6"])
def test_mx_fwd_bwd_tensor_cores(gd, d, act):
    x = _mx_case(5, [300, 5, 129, 64, 1], [70, 300, 1, 257, 40], 2, d)
    check(_run_mx(gd, x, 2, d, act), TOL["bf16"])


def test_mx_softmax_forward(gd):
    x = _mx_case(6, [200, 17], [300, 129], 2, 128)
    check(_run_mx(gd, x, 2, 128, "softmax", backward=False), TOL["bf16"])


def test_mx_causal_window(gd):
    lens = [300, 129, 7]
    x = _mx_case(7, lens, lens, 2, 128)
    check(_run_mx(gd, x, 2, 128, "gelu_tanh", mask="causal_window", window=77), TOL["bf16"])


def test_mx_cuda_core_path(gd):
    # d = 32: the CUDA-core kernels run on the expanded rows
    x = _mx_case(8, [40, 3], [20, 70], 3, 32)
    check(_run_mx(gd, x, 3, 32, "silu"), TOL["bf16"])


def test_mx_with_fused_rmsnorm(gd):
    x = _mx_case(9, [150, 33], [90, 260], 2, 128)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    plan.set_qk_norm(1.0, 1e-6)
    qm, km = gd.mx_quantise(x["q"]), gd.mx_quantise(x["k"])
    a = 128 ** -0.5
    o = gd.gdpa_fwd_mx(plan, qm, km, x["v"], alpha=a, act="gelu_erf")
    dq, dk, dv = gd.gdpa_bwd_mx(plan, qm, km, x["v"], x["do"], alpha=a, act="gelu_erf")
    plan.check()
    rq, rk = _oracle_inputs(x)
    args = (x["q_off"], x["kv_off"], rq, rk, x["v"])
    want = rn.bwd(*args, x["do"], a, "gelu_erf", 1.0, 1e-6)
    errs = {"o": max_rel(ref.to_f64(o), rn.fwd(*args, a, "gelu_erf", 1.0, 1e-6))}
    for n, gt, w in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        errs[n] = max_rel(ref.to_f64(gt), w)
    check(errs, TOL["bf16"])
    plan.destroy()


def test_mx_shared_seeds(gd):
    g = np.random.default_rng(10)
    H, d, n = 2, 128, 32
    lkv = [300, 17, 140]
    qo, ko = offsets_from_lengths(np.full(3, n)), offsets_from_lengths(np.asarray(lkv))

    def t(*shape):
        return torch.from_numpy(g.standard_normal(shape).astype(np.float32)).to(torch.bfloat16).cuda()

    seeds, k, v, do = t(n, H, d), t(ko[-1], H, d), t(ko[-1], H, d), t(qo[-1], H, d)
    plan = gd.Plan(qo, ko, H, d)
    plan.set_shared_q(n)
    sm, km = gd.mx_quantise(seeds), gd.mx_quantise(k)
    o = gd.gdpa_fwd_mx(plan, sm, km, v, act="silu")
    dq, dk, dv = gd.gdpa_bwd_mx(plan, sm, km, v, do, act="silu")
    plan.check()
    rs = mx.mx_round_trip(ref.to_f64(seeds))
    rk = mx.mx_round_trip(ref.to_f64(k))
    qt = ref.shared_q_tokens(rs, qo)
    a = d ** -0.5
    wdq, wdk, wdv = ref.bwd(qo, ko, qt, rk, v, do, a, "silu")
    check({"o": max_rel(ref.to_f64(o), ref.fwd(qo, ko, qt, rk, v, a, "silu")),
           "dq": max_rel(ref.to_f64(dq), ref.shared_q_grad(wdq, qo, n)),
           "dk": max_rel(ref.to_f64(dk), wdk), "dv": max_rel(ref.to_f64(dv), wdv)}, TOL["bf16"])
    plan.destroy()


def test_mx_training_workload_full_size(gd):
    # the training workload at full size: the quantiser's codes on sampled
    # rows against the oracle, and the MXFP8 forward equal, bit for bit, to
    # the bf16 forward on the dequantised rows (the same kernels and values)
    w = get_config("training_cross_fwd_bwd")
    x = to_dev(make_inputs(w, device="cpu", seed=31))
    plan = gd.Plan(x["q_off"], x["kv_off"], w.H, w.d)
    qm, km = gd.mx_quantise(x["q"]), gd.mx_quantise(x["k"])
    o = gd.gdpa_fwd_mx(plan, qm, km, x["v"], alpha=w.alpha, act=w.act)
    o_ref = gd.gdpa_fwd(plan, gd.mx_dequantise(qm), gd.mx_dequantise(km), x["v"], alpha=w.alpha,
                        act=w.act)
    plan.check()
    assert torch.equal(o, o_ref)
    g = np.random.default_rng(32)
    for t, m in ((x["q"], qm), (x["k"], km)):
        rows = np.sort(g.choice(t.shape[0], size=256, replace=False))
        idx = torch.from_numpy(rows).cuda()
        el, ex = mx.quantise(ref.to_f64(t.index_select(0, idx)))
        assert np.array_equal(m.scales.index_select(0, idx).cpu().numpy(), (ex + 127).astype(np.uint8))
        assert np.array_equal(m.elements.index_select(0, idx).cpu().numpy(), _codes(el))
    plan.destroy()


def test_mx_backward_reuses_forward_expansion(gd):
    # gdpa_bwd_mx with no MXFP8 pointers takes the forward's expansion: the
    # gradients equal those of a backward given Q and K again
    x = _mx_case(12, [200, 40, 3], [90, 130, 257], 2, 128)
    plan = gd.Plan(x["q_off"], x["kv_off"], 2, 128)
    qm, km = gd.mx_quantise(x["q"]), gd.mx_quantise(x["k"])
    with pytest.raises(gd.GdpaError) as e:    # nothing expanded yet
        gd.gdpa_bwd_mx(plan, None, None, x["v"], x["do"], act="silu")
    assert e.value.status == 1
    gd.gdpa_fwd_mx(plan, qm, km, x["v"], act="silu")
    reused = gd.gdpa_bwd_mx(plan, None, None, x["v"], x["do"], act="silu")
    given = gd.gdpa_bwd_mx(plan, qm, km, x["v"], x["do"], act="silu")
    plan.check()
    rq, rk = _oracle_inputs(x)
    want = ref.bwd(x["q_off"], x["kv_off"], rq, rk, x["v"], x["do"], 128 ** -0.5, "silu")
    check({n: max_rel(ref.to_f64(g), w) for n, g, w in zip(("dq", "dk", "dv"), reused, want)},
          TOL["bf16"])
    for a, b in zip(reused, given):
        assert torch.allclose(a, b, rtol=0, atol=1e-6 * float(b.abs().max()))
    plan.destroy()


def test_mx_argument_errors(gd):
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    el = torch.empty(64, dtype=torch.uint8, device="cuda")
    sc = torch.empty(2, dtype=torch.uint8, device="cuda")
    L = gd.lib()
    import ctypes
    vp = ctypes.c_void_p
    assert L.gdpa_mx_quantise(vp(x.data_ptr()), 48, vp(el.data_ptr()), vp(sc.data_ptr()), None) == 1
    assert L.gdpa_mx_quantise(vp(x.data_ptr() + 2), 32, vp(el.data_ptr()), vp(sc.data_ptr()),
                              None) == 1
    assert L.gdpa_mx_dequantise(vp(el.data_ptr() + 1), vp(sc.data_ptr()), 32, vp(x.data_ptr()),
                                None) == 1
    assert L.gdpa_mx_quantise(None, 0, None, None, None) == 0
    # a head dim that is not a multiple of 32, and the softmax backward
    case = _mx_case(11, [8], [8], 1, 64, spread=False)
    plan = gd.Plan(case["q_off"], case["kv_off"], 1, 48)
    b = torch.zeros(8, 1, 48, dtype=torch.uint8, device="cuda")
    s = torch.zeros(8, 1, 48 // 16, dtype=torch.uint8, device="cuda")
    v = torch.zeros(8, 1, 48, dtype=torch.bfloat16, device="cuda")
    st = L.gdpa_fwd_mx(plan.handle, vp(b.data_ptr()), vp(s.data_ptr()), vp(b.data_ptr()),
                       vp(s.data_ptr()), vp(v.data_ptr()), vp(v.data_ptr()), ctypes.c_float(1.0),
                       0, None)
    assert st == 1
    plan.destroy()
    plan = gd.Plan(case["q_off"], case["kv_off"], 1, 64)
    qm, km = gd.mx_quantise(case["q"]), gd.mx_quantise(case["k"])
    with pytest.raises(gd.GdpaError) as e:
        gd.gdpa_bwd_mx(plan, qm, km, case["v"], case["do"], act="softmax")
    assert e.value.status == 2
    plan.check()
    plan.destroy()
