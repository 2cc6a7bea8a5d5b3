"""Every environment knob that selects another kernel or launch shape
(include/zdmmv.h, "Launch-shape tuning"), each in a child process (the library
reads them once per process), over one fixed set of cases: single-vector DMMVs
in both layouts, the fused quantize + DMMV, batched calls of 2-8 vectors
(widths the vector split, the streaming batch kernel and the tensor-core kernel
take and do not take, and a 6-vector call the tensor-core kernel takes by
default), an expert gather, the one-launch expert FFN, the same FFN in two
launches (SwiGLU, then the fp32-activation gather reading its indices at once)
and a ready gather.

Knobs documented as leaving the bits unchanged must give the default run's
outputs bit for bit. The knobs that choose a batched kernel summing a row's
blocks in another order than the default's ("stream", "mma", one vector per
warp, which sends batches of more than 4 vectors to "stream", and "vsplit" and
"slots", which take the 6-vector call off the tensor cores) are checked against
the oracle within the DMMV tolerance, and must differ from the default somewhere
(so the other kernel ran). The default run itself is checked against the oracle."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from gguf_block_quant_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
Q4, Q8 = synth.Q4_0, synth.Q8_0
GGUF, REPACKED = 0, 1

# name: (fmt, rows, cols, batch, layout, fused); batch 1 is the single-vector call
DENSE_CASES = {
    "q4_4096": (Q4, 4096, 4096, 1, GGUF, False),
    "q8_2048_repacked": (Q8, 1000, 2048, 1, REPACKED, False),
    "q4_2048_fused": (Q4, 3001, 2048, 1, GGUF, True),
    "q8_4096_b2": (Q8, 1434, 4096, 2, GGUF, False),
    "q8_4096_b8": (Q8, 1434, 4096, 8, GGUF, False),
    "q4_2048_b5_repacked": (Q4, 777, 2048, 5, REPACKED, False),
    "q8_1280_b3": (Q8, 300, 1280, 3, GGUF, False),
    "q8_4096_b4_fused": (Q8, 1434, 4096, 4, GGUF, True),
    # a 32-row group for each of the GB300's 152 SMs: the tensor-core kernel by default
    "q8_4096_b6_tc": (Q8, 4900, 4096, 6, GGUF, False),
}
# the batched calls (and, under "mma", the fused batched one): the only results the
# batched-kernel knobs change
REORDERED = {"q8_4096_b2", "q8_4096_b8", "q4_2048_b5_repacked", "q8_1280_b3", "q8_4096_b6_tc", "q8_4096_b4_fused"}
MOE = dict(hidden=2048, ffn=512, slots=12, sel=[7, 0, 11, 3, 5, 9, 2, 10, 1])

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from gguf_block_quant_gb300 import zdmmv as Z
inp = np.load({inp!r})
cases = {cases!r}
moe = {moe!r}
out = {{}}
for name, (fmt, rows, cols, batch, layout, fused) in cases.items():
    w = torch.from_numpy(inp[name + ":w"]).cuda()
    if layout == 1:
        w = Z.repack(fmt, w, rows, cols)
    if fused:
        x = torch.from_numpy(inp[name + ":x"]).cuda()
        y = Z.dmmv_f32(fmt, w, rows, cols, x, batch=batch, layout=layout)
    else:
        xq = torch.from_numpy(inp[name + ":xq"]).cuda()
        y = Z.dmmv(fmt, w, rows, cols, xq, layout=layout) if batch == 1 else \
            Z.dmmv_batched(fmt, w, rows, cols, xq, batch, layout=layout)
    out[name] = y
gate = torch.from_numpy(inp["moe:gate"]).cuda()
up = torch.from_numpy(inp["moe:up"]).cuda()
down = torch.from_numpy(inp["moe:down"]).cuda()
idx = torch.tensor(moe["sel"], dtype=torch.int32, device="cuda")
xq = torch.from_numpy(inp["moe:xq"]).cuda()
h_, f_ = moe["hidden"], moe["ffn"]
gu, dn = f_ * (h_ // 32) * 18, h_ * (f_ // 32) * 34
out["gather"] = Z.expert_gather(Z.Q4_0, gate, gu, f_, h_, idx, moe["slots"], xq, 0)
y, h = Z.expert_ffn(Z.Q4_0, gate, up, gu, Z.Q8_0, down, dn, h_, f_, idx, moe["slots"], xq)
out["ffn_y"], out["ffn_h"] = y, h.clone()
# the same FFN in two launches (the down gather of the fp32 h, indices read at once),
# then a gate gather of the same selection reading its indices at once
h2 = Z.expert_swiglu(Z.Q4_0, gate, up, f_, h_, xq, idx=idx, expert_stride=gu, n_experts=moe["slots"])
out["ffn2_y"] = Z.expert_gather_f32(Z.Q8_0, down, dn, h_, f_, idx, moe["slots"], h2, f_, idx_ready=True)
out["gather_ready"] = Z.expert_gather(Z.Q4_0, gate, gu, f_, h_, idx, moe["slots"], xq, 0, idx_ready=True)
torch.cuda.synchronize()
assert Z.device_status() == 0
np.savez({dst!r}, **{{k: v.cpu().numpy() for k, v in out.items()}})
print("ok")
"""


@pytest.fixture(scope="module")
def inputs(tmp_path_factory):
    d = tmp_path_factory.mktemp("knobs")
    arrs = {}
    for i, (name, (fmt, rows, cols, batch, layout, fused)) in enumerate(DENSE_CASES.items()):
        arrs[name + ":w"] = synth.weight_blocks(fmt, rows, cols, seed=100 + i)
        x = np.ascontiguousarray(synth.activations(cols, seed=200 + i, batch=batch)).reshape(-1)
        if fused:
            arrs[name + ":x"] = x
        else:
            arrs[name + ":xq"] = oracle.quantize_q8_0(x)
    h, f, n = MOE["hidden"], MOE["ffn"], MOE["slots"]
    arrs["moe:gate"] = synth.weight_blocks(Q4, n * f, h, seed=300)
    arrs["moe:up"] = synth.weight_blocks(Q4, n * f, h, seed=301)
    arrs["moe:down"] = synth.weight_blocks(Q8, n * h, f, seed=302)
    arrs["moe:xq"] = oracle.quantize_q8_0(synth.activations(h, seed=303))
    path = str(d / "inputs.npz")
    np.savez(path, **arrs)
    return path, arrs


def _run(inputs_path, tmpdir, tag, env_extra):
    dst = os.path.join(tmpdir, f"out_{tag}.npz")
    code = _CHILD.format(root=ROOT, inp=inputs_path, cases=DENSE_CASES, moe=MOE, dst=dst)
    env = {k: v for k, v in os.environ.items() if not k.startswith("ZDMMV_")}
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr[-3000:]
    with np.load(dst) as z:
        return {k: z[k] for k in z.files}


@pytest.fixture(scope="module")
def default_run(inputs, tmp_path_factory):
    path, arrs = inputs
    out = _run(path, str(tmp_path_factory.mktemp("default")), "default", {})
    # the default run against the oracle
    for name, (fmt, rows, cols, batch, layout, fused) in DENSE_CASES.items():
        w = arrs[name + ":w"]
        xq = oracle.quantize_q8_0(arrs[name + ":x"]) if fused else arrs[name + ":xq"]
        y_ref, e_ref = oracle.dmmv_batched(fmt, w, rows, cols, xq, batch)
        ok, worst = oracle.within_tolerance(out[name].reshape(batch, rows), y_ref, e_ref)
        assert ok, (name, worst)
    h, f, n = MOE["hidden"], MOE["ffn"], MOE["slots"]
    sel = np.array(MOE["sel"], dtype=np.int32)
    gu, dn = f * (h // 32) * 18, h * (f // 32) * 34
    y_ref, e_ref, st = oracle.expert_gather(Q4, arrs["moe:gate"], gu, f, h, sel, n, arrs["moe:xq"], 0)
    assert st == 0
    ok, worst = oracle.within_tolerance(out["gather"], y_ref, e_ref)
    assert ok, ("gather", worst)
    # the FFN's down projection of its own h, quantized by the oracle
    hq = oracle.quantize_q8_0(out["ffn_h"].astype(np.float32))
    y_ref, e_ref, st = oracle.expert_gather(Q8, arrs["moe:down"], dn, h, f, sel, n, hq, (f // 32) * 34)
    assert st == 0
    ok, worst = oracle.within_tolerance(out["ffn_y"], y_ref, e_ref)
    assert ok, ("ffn", worst)
    # the two-launch FFN and the ready gather: the one-launch FFN's and the gather's bits
    assert np.array_equal(out["ffn2_y"], out["ffn_y"])
    assert np.array_equal(out["gather_ready"], out["gather"])
    return out


SAME_BITS = [
    {"ZDMMV_STAGE_KB": "8"},
    {"ZDMMV_STAGE_KB": "48"},
    {"ZDMMV_CTAS_PER_SM": "1"},
    {"ZDMMV_CTAS_PER_SM": "4"},
    {"ZDMMV_BATCH_CTAS_PER_SM": "1"},
    {"ZDMMV_BATCH_CTAS_PER_SM": "4"},
    {"ZDMMV_FFN_STAGES": "3"},
    {"ZDMMV_FFN_CTAS_PER_SM": "2"},
    {"ZDMMV_FFN_GU_PERCENT": "30"},
    {"ZDMMV_PDL": "0"},
]


@pytest.mark.parametrize("env", SAME_BITS, ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
def test_knob_keeps_the_bits(env, inputs, default_run, tmp_path):
    out = _run(inputs[0], str(tmp_path), "knob", env)
    for k, v in default_run.items():
        assert np.array_equal(out[k], v), k


REORDERING = [
    {"ZDMMV_BATCH_KERNEL": "stream"},
    {"ZDMMV_VSPLIT_V": "1"},          # more than 4 vectors off the tensor cores: the "stream" kernel
    {"ZDMMV_BATCH_KERNEL": "mma"},
    {"ZDMMV_BATCH_KERNEL": "vsplit"},  # the 6-vector call: the single-vector order
    {"ZDMMV_BATCH_KERNEL": "slots"},
    {"ZDMMV_BATCH_SLOTS": "1"},
]


@pytest.mark.parametrize("env", REORDERING, ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
def test_other_batched_kernel_within_tolerance(env, inputs, default_run, tmp_path):
    path, arrs = inputs
    out = _run(path, str(tmp_path), "knob", env)
    differs = False
    for name, (fmt, rows, cols, batch, layout, fused) in DENSE_CASES.items():
        if name not in REORDERED:
            assert np.array_equal(out[name], default_run[name]), name
            continue
        xq = oracle.quantize_q8_0(arrs[name + ":x"]) if fused else arrs[name + ":xq"]
        y_ref, e_ref = oracle.dmmv_batched(fmt, arrs[name + ":w"], rows, cols, xq, batch)
        ok, worst = oracle.within_tolerance(out[name].reshape(batch, rows), y_ref, e_ref)
        assert ok, (name, worst)
        differs |= not np.array_equal(out[name], default_run[name])
    assert differs, "the selected kernel gave the default kernel's bits everywhere"
    for k in ("gather", "gather_ready", "ffn_y", "ffn_h", "ffn2_y"):
        assert np.array_equal(out[k], default_run[k]), k
