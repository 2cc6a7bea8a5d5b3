"""zdmmv_expert_gather_ready: the expert gather that reads its index list as soon
as its kernel starts, for a list an earlier expert call on the stream has read
(the down projections after the gate/up launch of the same experts).

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
