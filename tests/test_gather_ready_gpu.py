"""zdmmv_expert_gather_ready: the expert gather that reads its index list as soon
as its kernel starts, for a list an earlier expert call on the stream has read
(the down projections after the gate/up launch of the same experts); and
zdmmv_expert_gather_f32, the gather over fp32 activations quantized in the
launch (the down projection of the SwiGLU output without a quantizer launch),
which reads its list either way.

Its results must be those of zdmmv_expert_gather bit for bit (same kernel
arithmetic), NaN rows and the status word for an out-of-range index included;
and, in a decode-like loop where a kernel rewrites ONE index buffer before every
layer's gate/up call, each layer's ready gather must see that layer's list (a
stale or half-written list would give another layer's experts).
"""
import numpy as np
import pytest
import torch

import oracle
from gguf_block_quant_gb300 import synth
from gguf_block_quant_gb300 import zdmmv as Z

pytestmark = pytest.mark.gpu

Q4_0, Q8_0 = Z.Q4_0, Z.Q8_0


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    Z.lib()
    Z.device_status(clear=True)
    yield
    assert Z.device_status() == 0, "a kernel reported a device fault"


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def nan_out(*shape) -> torch.Tensor:
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def _stack(fmt, rows, cols, n_exp, seed, layout, stream=synth.S_WEIGHT):
    bb = 18 if fmt == Q4_0 else 34
    per = rows * cols // 32 * bb
    s = synth.weight_blocks(fmt, n_exp * rows, cols, seed=seed, stream=stream)
    d = dev(s)
    if layout == Z.REPACKED:
        d = torch.cat([Z.repack(fmt, d[e * per:(e + 1) * per], rows, cols) for e in range(n_exp)])
    return s, d, per


@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols", [(Q8_0, 2048, 512), (Q4_0, 512, 2048), (Q8_0, 300, 4096),
                                           (Q4_0, 40, 96)])
def test_ready_gather_equals_gather_bitwise(fmt, rows, cols, layout):
    """After a gate/up-like gather2 of the same list: the ready gather's rows equal
    zdmmv_expert_gather's bit for bit, an out-of-range index gives NaN rows and
    status 1, and the good rows meet the oracle's tolerance. (40 x 96 runs off the
    pipelined path.)"""
    n_exp = 9
    s_gu, d_gu, per_gu = _stack(fmt, rows, cols, n_exp, seed=61, layout=layout)
    s_dn, d_dn, per_dn = _stack(fmt, rows, cols, n_exp, seed=62, layout=layout, stream=synth.S_WEIGHT3)
    idx = np.array([8, 0, 4, 4, 2, 9, 1, 7, 3, 6], dtype=np.int32)   # 9 is out of range
    n = len(idx)
    # per-slot activations at a 16-byte stride (the entry points' alignment rule)
    vec = cols // 32 * 34
    xs = (vec + 15) // 16 * 16
    xq = np.zeros((n, xs), dtype=np.uint8)
    xq[:, :vec] = oracle.quantize_q8_0(synth.activations(cols, seed=63, batch=n)).reshape(n, vec)
    xq = xq.reshape(-1)
    di, dx = dev(idx), dev(xq)
    st_gu = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = nan_out(n, rows)
    Z.expert_gather2(fmt, d_gu, d_gu, per_gu, rows, cols, di, n_exp, dx, xs, status=st_gu, layout=layout)
    Z.expert_gather(fmt, d_dn, per_dn, rows, cols, di, n_exp, dx, xs, y=y, status=st, layout=layout,
                    idx_ready=True)
    y_ref = Z.expert_gather(fmt, d_dn, per_dn, rows, cols, di, n_exp, dx, xs, y=nan_out(n, rows), status=st_ref,
                            layout=layout)
    torch.cuda.synchronize()
    assert st.item() == 1 and st_ref.item() == 1 and st_gu.item() == 1
    good = [k for k in range(n) if idx[k] < n_exp]
    assert torch.isnan(y[5]).all()
    assert torch.equal(y[good], y_ref[good])
    yo, eo, sto = oracle.expert_gather(fmt, s_dn, per_dn, rows, cols, idx, n_exp, xq, xs)
    assert sto == 1
    ok, worst = oracle.within_tolerance(y[good].double().cpu().numpy(), yo[good], eo[good])
    assert ok, worst


@pytest.mark.parametrize("graph", [False, True])
def test_ready_gather_sees_each_layers_list(graph):
    """One device index buffer rewritten by a kernel before every layer; per layer a
    gate/up SwiGLU call reads it after its dependency wait and a down gather reads
    it at once (ready). Each layer's down rows equal a separate zdmmv_expert_gather
    with that layer's list, bit for bit, eager and replayed as a CUDA graph."""
    hidden, ffn, n_exp, layers = 2048, 512, 33, 12
    n = 9
    _, d_g, per_gu = _stack(Q4_0, ffn, hidden, n_exp, seed=71, layout=Z.GGUF)
    _, d_u, _ = _stack(Q4_0, ffn, hidden, n_exp, seed=72, layout=Z.GGUF, stream=synth.S_WEIGHT2)
    _, d_d, per_dn = _stack(Q8_0, hidden, ffn, n_exp, seed=73, layout=Z.GGUF, stream=synth.S_WEIGHT3)
    lists = np.stack([synth.expert_indices(100 + l, n_routed=n_exp - 1, top_k=n - 1) for l in range(layers)])
    assert lists.shape == (layers, n) and len({tuple(r) for r in lists}) == layers
    src = dev(lists.astype(np.int32))
    idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    xq = dev(oracle.quantize_q8_0(synth.activations(hidden, seed=74)))
    xqd = dev(oracle.quantize_q8_0(synth.activations(ffn, seed=75, batch=n)))
    xs = ffn // 32 * 34
    h = torch.empty(n, ffn, device="cuda")
    ys = [nan_out(n, hidden) for _ in range(layers)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        for l in range(layers):
            torch.add(src[l], 0, out=idx)     # the "router": a kernel writes this layer's list
            Z.expert_swiglu(Q4_0, d_g, d_u, ffn, hidden, xq, idx=idx, expert_stride=per_gu, n_experts=n_exp,
                            h=h, status=st)
            Z.expert_gather(Q8_0, d_d, per_dn, hidden, ffn, idx, n_exp, xqd, xs, y=ys[l], status=st,
                            idx_ready=True)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()                               # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        for y in ys:
            y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    assert st.item() == 0
    for l in range(layers):
        ref = Z.expert_gather(Q8_0, d_d, per_dn, hidden, ffn, src[l].clone(), n_exp, xqd, xs,
                              y=nan_out(n, hidden))
        torch.cuda.synchronize()
        assert torch.equal(ys[l], ref), f"layer {l}: the ready gather did not use that layer's list"


@pytest.mark.parametrize("ready", [0, 1])
@pytest.mark.parametrize("layout", [Z.GGUF, Z.REPACKED])
@pytest.mark.parametrize("fmt,rows,cols,shared", [(Q8_0, 2048, 512, False), (Q4_0, 512, 2048, False),
                                                  (Q8_0, 300, 4096, True), (Q4_0, 1000, 256, False)])
def test_gather_f32_equals_quantize_then_gather(fmt, rows, cols, shared, layout, ready):
    """Slot k of the fp32-activation gather equals zdmmv_quantize_act_q8_0 of its
    activation followed by zdmmv_expert_gather, bit for bit (the same quantizer
    arithmetic in the kernel's prologue); per-slot activations at a padded stride
    or one shared activation; an out-of-range index gives NaN rows and status 1."""
    n_exp = 9
    _, d_gu, per_gu = _stack(fmt, rows, cols, n_exp, seed=81, layout=layout)
    s_dn, d_dn, per_dn = _stack(fmt, rows, cols, n_exp, seed=82, layout=layout, stream=synth.S_WEIGHT3)
    idx = np.array([3, 8, 0, 9, 5, 5, 1], dtype=np.int32)   # 9 is out of range
    n = len(idx)
    xs = 0 if shared else cols + 8                         # floats; a multiple of 4
    xv = synth.activations(cols, seed=83, batch=1 if shared else n).reshape(1 if shared else n, cols)
    xpad = np.zeros((xv.shape[0], cols if shared else xs), dtype=np.float32)
    xpad[:, :cols] = xv
    di, dx = dev(idx), dev(xpad.reshape(-1))
    st_gu = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    # an earlier expert call of the same list (the ready read's requirement)
    Z.expert_gather2(fmt, d_gu, d_gu, per_gu, rows, cols, di, n_exp, Z.quantize_act_q8_0(dev(xv[0])), 0,
                     status=st_gu, layout=layout)
    y = Z.expert_gather_f32(fmt, d_dn, per_dn, rows, cols, di, n_exp, dx, xs, y=nan_out(n, rows), status=st,
                            layout=layout, idx_ready=bool(ready))
    xq = Z.quantize_act_q8_0(dev(np.ascontiguousarray(xv)))
    y_ref = Z.expert_gather(fmt, d_dn, per_dn, rows, cols, di, n_exp, xq, 0 if shared else cols // 32 * 34,
                            y=nan_out(n, rows), status=st_ref, layout=layout)
    torch.cuda.synchronize()
    assert st.item() == 1 and st_ref.item() == 1
    good = [k for k in range(n) if idx[k] < n_exp]
    assert torch.isnan(y[3]).all()
    assert torch.equal(y[good], y_ref[good])
    xq_o = oracle.quantize_q8_0(xv.reshape(-1))
    assert np.array_equal(xq.cpu().numpy(), xq_o)
    yo, eo, _ = oracle.expert_gather(fmt, s_dn, per_dn, rows, cols, idx, n_exp, xq_o,
                                     0 if shared else cols // 32 * 34)
    ok, worst = oracle.within_tolerance(y[good].double().cpu().numpy(), yo[good], eo[good])
    assert ok, worst


@pytest.mark.parametrize("graph", [False, True])
def test_two_launch_ffn_equals_one_launch_ffn(graph):
    """The selected experts' FFN as two launches, zdmmv_expert_swiglu (h) then the
    ready fp32-activation down gather of h, in a 10-layer loop that rewrites one
    index buffer by a kernel before every layer: each layer's y equals the
    one-launch zdmmv_expert_ffn of that layer's list, and its h, bit for bit."""
    hidden, ffn, n_exp, layers, n = 2048, 512, 33, 10, 9
    _, d_g, per_gu = _stack(Q4_0, ffn, hidden, n_exp, seed=91, layout=Z.GGUF)
    _, d_u, _ = _stack(Q4_0, ffn, hidden, n_exp, seed=92, layout=Z.GGUF, stream=synth.S_WEIGHT2)
    _, d_d, per_dn = _stack(Q8_0, hidden, ffn, n_exp, seed=93, layout=Z.GGUF, stream=synth.S_WEIGHT3)
    lists = np.stack([synth.expert_indices(200 + l, n_routed=n_exp - 1, top_k=n - 1) for l in range(layers)])
    src = dev(lists.astype(np.int32))
    idx = torch.zeros(n, dtype=torch.int32, device="cuda")
    xq = dev(oracle.quantize_q8_0(synth.activations(hidden, seed=94)))
    hs = [torch.full((n, ffn), float("nan"), device="cuda") for _ in range(layers)]
    ys = [nan_out(n, hidden) for _ in range(layers)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        for l in range(layers):
            torch.add(src[l], 0, out=idx)     # the "router"
            Z.expert_swiglu(Q4_0, d_g, d_u, ffn, hidden, xq, idx=idx, expert_stride=per_gu, n_experts=n_exp,
                            h=hs[l], status=st)
            Z.expert_gather_f32(Q8_0, d_d, per_dn, hidden, ffn, idx, n_exp, hs[l], ffn, y=ys[l], status=st,
                                idx_ready=True)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.current_stream().wait_stream(s)
        for t in hs + ys:
            t.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    assert st.item() == 0
    ws = Z.expert_ffn_workspace(n, ffn)
    for l in range(layers):
        y1, h1 = Z.expert_ffn(Q4_0, d_g, d_u, per_gu, Q8_0, d_d, per_dn, hidden, ffn, src[l].clone(), n_exp, xq,
                              y=nan_out(n, hidden), workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(hs[l], h1), f"layer {l}: h differs"
        assert torch.equal(ys[l], y1), f"layer {l}: y differs from the one-launch FFN"


@pytest.mark.parametrize("graph", [False, True])
def test_ready_gather_after_a_device_router(graph):
    """The index list written by a kernel that lets its dependents start before it
    writes: the argmax DMMV (a 33-row router, top-1 pick) releases the next launch
    before its reduction stores the index. Per layer: the router's argmax writes
    one index into a shared buffer, a gate+up gather2 reads it after its wait, and
    the ready down gather reads it at once. If the gather2 let the down gather
    start before its own wait, the down gather could read the previous layer's
    pick; each layer's down rows must equal a separate gather with that layer's
    pick, bit for bit, eager and as a replayed CUDA graph."""
    hidden, ffn, n_exp, layers = 2048, 512, 33, 16
    r_np = synth.weight_blocks(Q8_0, n_exp, hidden, seed=101)
    router = dev(r_np)
    _, d_g, per_gu = _stack(Q4_0, ffn, hidden, n_exp, seed=102, layout=Z.GGUF)
    _, d_u, _ = _stack(Q4_0, ffn, hidden, n_exp, seed=103, layout=Z.GGUF, stream=synth.S_WEIGHT2)
    _, d_d, per_dn = _stack(Q8_0, hidden, ffn, n_exp, seed=104, layout=Z.GGUF, stream=synth.S_WEIGHT3)
    xqs = [dev(oracle.quantize_q8_0(synth.activations(hidden, seed=110 + l))) for l in range(layers)]
    xqd = dev(oracle.quantize_q8_0(synth.activations(ffn, seed=105)))
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(Z.ARGMAX_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    ya = torch.empty(1, ffn, device="cuda")
    yb = torch.empty(1, ffn, device="cuda")
    ys = [nan_out(1, hidden) for _ in range(layers)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        for l in range(layers):
            Z.dmmv_argmax(Q8_0, router, n_exp, hidden, xqs[l], workspace=ws, out=idx)
            Z.expert_gather2(Q4_0, d_g, d_u, per_gu, ffn, hidden, idx, n_exp, xqs[l], 0, y_a=ya, y_b=yb,
                             status=st)
            Z.expert_gather(Q8_0, d_d, per_dn, hidden, ffn, idx, n_exp, xqd, 0, y=ys[l], status=st,
                            idx_ready=True)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.current_stream().wait_stream(s)
        for y in ys:
            y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        g.replay()
    else:
        run()
    torch.cuda.synchronize()
    assert st.item() == 0
    picks = []
    for l in range(layers):
        logits = Z.dmmv(Q8_0, router, n_exp, hidden, xqs[l]).cpu().numpy()   # the argmax kernel's fp32 logits
        pick = int(np.argmax(logits))                                       # first index of the maximum
        picks.append(pick)
        ref = Z.expert_gather(Q8_0, d_d, per_dn, hidden, ffn, torch.tensor([pick], dtype=torch.int32,
                              device="cuda"), n_exp, xqd, 0, y=nan_out(1, hidden))
        torch.cuda.synchronize()
        assert torch.equal(ys[l], ref), f"layer {l}: the ready gather did not use that layer's pick {pick}"
    assert len(set(picks)) >= 4, picks   # the picks change from layer to layer
