"""Parity at the full sizes of the five decode workloads, in the launch
configuration the benchmark times (same entry points, same shapes, device-
resident inputs). The oracle computes every output row of every workload here
(a few seconds of plain C each), and the integer block sums are compared bit for
bit on sampled rows through the debug entry point.
"""
import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    Z.lib()
    Z.device_status(clear=True)
    yield
    assert Z.device_status() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(y, y_ref, e_ref):
    yh = y.double().cpu().numpy().reshape(np.shape(y_ref))
    assert not np.isnan(yh).any()
    ok, worst = oracle.within_tolerance(yh, y_ref, e_ref)
    assert ok, f"worst |dy|/bound = {worst:.3g}"


def sampled_sums(cfg, w, xq_ref, wd, xqd, n=64):
    """Bit-exact int32 block sums on n sampled rows (plus first/last)."""
    rows, cols = cfg.rows, cfg.cols
    rb = cfg.nb * synth.BLOCK_BYTES[cfg.fmt]
    g = np.random.default_rng(cfg.seed)
    pick = np.unique(np.concatenate([[0, rows - 1], g.integers(0, rows, n)]))
    w_rows = w.reshape(rows, rb)[pick].reshape(-1)
    ref = oracle.block_sums(cfg.fmt, w_rows, len(pick), cols, xq_ref)
    got = Z.debug_block_sums(cfg.fmt, dev(w_rows), len(pick), cols, xqd)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("cfg", [synth.SSM_ALPHA_BETA, synth.DENSE_Q4_0, synth.LM_HEAD_Q4_0],
                         ids=lambda c: c.name)
def test_dense_workload_full_size(cfg):
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    wd = dev(w)
    xqd = Z.quantize_act_q8_0(dev(x))
    y = torch.full((cfg.rows,), float("nan"), device="cuda")
    Z.dmmv(cfg.fmt, wd, cfg.rows, cfg.cols, xqd, y=y)
    torch.cuda.synchronize()
    xq_ref = oracle.quantize_q8_0(x)
    assert np.array_equal(xqd.cpu().numpy(), xq_ref)
    y_ref, e_ref = oracle.dmmv(cfg.fmt, w, cfg.rows, cfg.cols, xq_ref)
    check(y, y_ref, e_ref)
    sampled_sums(cfg, w, xq_ref, wd, xqd)
    # the headline step's fused entry point (quantization inside the DMMV launch): the same bits
    yf = torch.full((cfg.rows,), float("nan"), device="cuda")
    Z.dmmv_f32(cfg.fmt, wd, cfg.rows, cfg.cols, dev(x), y=yf)
    torch.cuda.synchronize()
    assert torch.equal(yf, y)
    # the greedy pick with the fused argmax epilogue: the first index of the
    # kernel's own logits' maximum, and a valid argmax of the oracle's
    i = int(Z.dmmv_argmax(cfg.fmt, wd, cfg.rows, cfg.cols, xqd).item())
    yh = y.cpu().numpy()
    assert i == int(np.argmax(yh))
    j, _ = oracle.argmax(y_ref)
    assert y_ref[i] >= y_ref[j] - 1e-5 * (e_ref[i] + e_ref[j]) - 2e-6


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_batched_workload_full_size(batch):
    cfg = synth.BATCHED_Q8_0[batch]
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, batch=batch)
    wd = dev(w)
    xqd = Z.quantize_act_q8_0(dev(x))
    y = torch.full((batch, cfg.rows), float("nan"), device="cuda")
    Z.dmmv_batched(cfg.fmt, wd, cfg.rows, cfg.cols, xqd, batch, y=y)
    torch.cuda.synchronize()
    xq_ref = oracle.quantize_q8_0(x)
    assert np.array_equal(xqd.cpu().numpy(), xq_ref)
    y_ref, e_ref = oracle.dmmv_batched(cfg.fmt, w, cfg.rows, cfg.cols, xq_ref, batch)
    check(y, y_ref, e_ref)


def test_moe_workload_full_size():
    m = synth.MOE
    gate = synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed, stream=synth.S_WEIGHT)
    up = synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed, stream=synth.S_WEIGHT2)
    down = synth.weight_blocks(synth.Q8_0, m.n_slots * m.hidden, m.ffn, seed=m.seed, stream=synth.S_WEIGHT3)
    idx = synth.expert_indices(m.seed, m.n_routed, m.top_k)
    x = synth.activations(m.hidden, seed=m.seed)
    xd = synth.activations(m.ffn, seed=m.seed, stream=synth.S_ACT2, batch=m.n_sel)
    gu_per, dn_per = m.gate_up_bytes(), m.down_bytes()
    idx_d = dev(idx)
    xq = Z.quantize_act_q8_0(dev(x))
    xqd = Z.quantize_act_q8_0(dev(xd))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    yg = torch.full((m.n_sel, m.ffn), float("nan"), device="cuda")
    yu = torch.full((m.n_sel, m.ffn), float("nan"), device="cuda")
    yd = torch.full((m.n_sel, m.hidden), float("nan"), device="cuda")
    Z.expert_gather(Z.Q4_0, dev(gate), gu_per, m.ffn, m.hidden, idx_d, m.n_slots, xq, 0, y=yg, status=st)
    Z.expert_gather(Z.Q4_0, dev(up), gu_per, m.ffn, m.hidden, idx_d, m.n_slots, xq, 0, y=yu, status=st)
    Z.expert_gather(Z.Q8_0, dev(down), dn_per, m.hidden, m.ffn, idx_d, m.n_slots, xqd,
                    (m.ffn // 32) * 34, y=yd, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    xq_ref = oracle.quantize_q8_0(x)
    xqd_ref = oracle.quantize_q8_0(xd)
    for y, stack, per, fmt, rows, cols, xr, xs in [
            (yg, gate, gu_per, synth.Q4_0, m.ffn, m.hidden, xq_ref, 0),
            (yu, up, gu_per, synth.Q4_0, m.ffn, m.hidden, xq_ref, 0),
            (yd, down, dn_per, synth.Q8_0, m.hidden, m.ffn, xqd_ref, (m.ffn // 32) * 34)]:
        y_ref, e_ref, s = oracle.expert_gather(fmt, stack, per, rows, cols, idx, m.n_slots, xr, xs)
        assert s == 0
        check(y, y_ref, e_ref)


def test_large_matrix_sampled_rows():
    """A matrix larger than anything above (604 MB of Q4_0 weights, 2^19 rows):
    sampled rows against the oracle, computed row by row."""
    rows, cols = 1 << 19, 2048
    rb = cols // 32 * 18
    w = synth.weight_blocks(synth.Q4_0, rows, cols, seed=123)
    x = synth.activations(cols, seed=124)
    xqd = Z.quantize_act_q8_0(dev(x))
    wd = dev(w)
    y = torch.full((rows,), float("nan"), device="cuda")
    Z.q4_0(wd, rows, cols, xqd, y=y)
    torch.cuda.synchronize()
    yh = y.double().cpu().numpy()
    assert not np.isnan(yh).any()
    xq_ref = oracle.quantize_q8_0(x)
    pick = np.unique(np.concatenate([[0, 1, rows - 1], np.random.default_rng(0).integers(0, rows, 4000)]))
    y_ref, e_ref = oracle.dmmv(synth.Q4_0, w.reshape(rows, rb)[pick].reshape(-1), len(pick), cols, xq_ref)
    ok, worst = oracle.within_tolerance(yh[pick], y_ref, e_ref)
    assert ok, worst


def _swiglu_bound(g_ref, u_ref, e_g, e_u, h_ref):
    tg, tu = 1e-5 * e_g + 1e-6, 1e-5 * e_u + 1e-6
    silu = g_ref / (1.0 + np.exp(-g_ref))
    return 1.1 * tg * np.abs(u_ref) + np.abs(silu) * tu + 1.1 * tg * tu + 16 * 2.0 ** -24 * np.abs(h_ref) + 1e-12


def test_moe_gate_up_swiglu_full_size():
    """The MoE workload's gate and up projections with the SwiGLU epilogue, in the
    launch the benchmark times: h = silu(G x) * (U x) for the 9 selected experts."""
    m = synth.MOE
    gate = synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed, stream=synth.S_WEIGHT)
    up = synth.weight_blocks(synth.Q4_0, m.n_slots * m.ffn, m.hidden, seed=m.seed, stream=synth.S_WEIGHT2)
    idx = synth.expert_indices(m.seed, m.n_routed, m.top_k)
    x = synth.activations(m.hidden, seed=m.seed)
    gu_per = m.gate_up_bytes()
    gd, ud, idx_d = dev(gate), dev(up), dev(idx)
    xq = Z.quantize_act_q8_0(dev(x))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h = torch.full((m.n_sel, m.ffn), float("nan"), device="cuda")
    Z.expert_swiglu(Z.Q4_0, gd, ud, m.ffn, m.hidden, xq, idx=idx_d, expert_stride=gu_per, n_experts=m.n_slots,
                    h=h, status=st)
    ga, ua = Z.expert_gather2(Z.Q4_0, gd, ud, gu_per, m.ffn, m.hidden, idx_d, m.n_slots, xq, 0)
    torch.cuda.synchronize()
    assert st.item() == 0
    hh = h.double().cpu().numpy()
    assert not np.isnan(hh).any()
    g32, u32 = ga.double().cpu().numpy(), ua.double().cpu().numpy()
    h64 = g32 / (1.0 + np.exp(-g32)) * u32
    assert np.all(np.abs(hh - h64) <= 16 * 2.0 ** -24 * np.abs(h64) + 1e-30)
    xq_ref = oracle.quantize_q8_0(x)
    g_ref, e_g, _ = oracle.expert_gather(synth.Q4_0, gate, gu_per, m.ffn, m.hidden, idx, m.n_slots, xq_ref, 0)
    u_ref, e_u, _ = oracle.expert_gather(synth.Q4_0, up, gu_per, m.ffn, m.hidden, idx, m.n_slots, xq_ref, 0)
    h_ref = oracle.swiglu(g_ref.ravel(), u_ref.ravel()).reshape(g_ref.shape)
    assert np.all(np.abs(hh - h_ref) <= _swiglu_bound(g_ref, u_ref, e_g, e_u, h_ref))


def test_shared_expert_sigmoid_scale_acc_full_size():
    """The shared expert's down projection (Q8_0 2048 x 512) accumulated into a
    residual with the sigmoid gate, and the gate-less accumulate mode."""
    m = synth.MOE
    rows, cols = m.hidden, m.ffn
    w = synth.weight_blocks(synth.Q8_0, rows, cols, seed=m.seed, stream=synth.S_WEIGHT3)
    xq = synth.activation_blocks(cols // 32, seed=m.seed)
    y0 = synth.activations(rows, seed=m.seed + 1, scale=0.05)
    wd, xqd = dev(w), dev(xq)
    d_ref, _ = oracle.dmmv(synth.Q8_0, w, rows, cols, xq)
    for gate in (None, -0.7):
        y = dev(y0.copy())
        g = None if gate is None else torch.tensor([gate], dtype=torch.float32, device="cuda")
        Z.dmmv_acc(synth.Q8_0, wd, rows, cols, xqd, y, gate=g)
        torch.cuda.synchronize()
        y_ref, e_ref = oracle.dmmv_acc(synth.Q8_0, w, rows, cols, xq, y0.astype(np.float64), gate=gate)
        yh = y.double().cpu().numpy()
        bound = 1e-5 * e_ref + 1e-6 + 4 * 2.0 ** -24 * np.abs(d_ref) + 2.0 ** -24 * np.abs(y_ref)
        assert np.all(np.abs(yh - y_ref) <= bound)


@pytest.mark.parametrize("cfg", [synth.DENSE_Q4_0, synth.LM_HEAD_Q4_0, synth.BATCHED_Q8_0[1]],
                         ids=lambda c: c.name)
def test_xf32_activation_full_size(cfg):
    """The fp32-activation product at the workloads' full sizes (all rows)."""
    w = synth.weight_blocks(cfg.fmt, cfg.rows, cfg.cols, seed=cfg.seed)
    x = synth.activations(cfg.cols, seed=cfg.seed, scale=cfg.x_scale)
    y = torch.full((cfg.rows,), float("nan"), device="cuda")
    Z.dmmv_xf32(cfg.fmt, dev(w), cfg.rows, cfg.cols, dev(x), y=y)
    torch.cuda.synchronize()
    y_ref, e_ref = oracle.dmmv_xf32(cfg.fmt, w, cfg.rows, cfg.cols, x)
    check(y, y_ref, e_ref)
