"""CUDA-graph capture of whole stage sweeps (the NVIDIA Swin talk, section 2, and the
AIAK-Training talk, section 2: one graph launch for many kernels removes the launch gaps).

Each graph is captured once from the library's C entry points, then replayed twice: the
inputs are rewritten in place between the replays (new qkv, a new bias table for the
training step), and every replay's outputs are compared element by element, on every
image, with the fp64 oracle for the inputs of that replay. The outputs are filled with
NaN before each replay, so an element the replay did not write fails the comparison.
"""
import numpy as np
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, batch_chunks, oracle_bwd, plan

pytestmark = pytest.mark.gpu
DEV = "cuda"
L224 = ["swin_l224_s1", "swin_l224_s2", "swin_l224_s3", "swin_l224_s4"]
B224 = ["swin_b224_s1", "swin_b224_s2", "swin_b224_s3", "swin_b224_s4"]
L384 = ["swin_l384_s1", "swin_l384_s2", "swin_l384_s3", "swin_l384_s4"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from swin_window_attention_gb300 import build
    build.build()
    oracle.build()
    capi.load()


def _f64(t):
    return t.to(torch.float64).numpy()


def _capture(stream, fn):
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        fn()
    torch.cuda.synchronize()
    return g


def _replay(g, stream, outs):
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()


@pytest.mark.parametrize("names,kernel", [
    (L224, capi.KERNEL_MMA_SYNC),
    (L224, capi.KERNEL_TCGEN05),
    (L384, capi.KERNEL_AUTO),
], ids=["l224-mma_sync", "l224-tcgen05", "l384-auto"])
def test_sweep_graph_replays_match_the_oracle(names, kernel):
    """The headline step: the four Swin-L 224 stage forwards (B = 64) as one graph; and the
    four Swin-L 384 ones (12x12 windows, B = 16) with the kernels AUTO picks per stage."""
    stream = torch.cuda.Stream()
    wls = [inputs.BY_NAME[n] for n in names]
    tabs = [inputs.make_table(wl) for wl in wls]
    atts = [plan(wl, t.to(DEV)) for wl, t in zip(wls, tabs)]
    for a in atts:
        a.set_fwd_kernel(kernel)
    qs = [torch.empty(wl.B, wl.H, wl.W, 3 * wl.C, dtype=torch.bfloat16, device=DEV) for wl in wls]
    ys = [torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16, device=DEV) for wl in wls]
    g = _capture(stream, lambda: [a.fwd(q, out=y) for a, q, y in zip(atts, qs, ys)])
    for replay, offset in enumerate((0, 500)):
        host = [inputs.make_qkv(wl, seed_offset=offset) for wl in wls]
        for q, h in zip(qs, host):
            q.copy_(h)
        _replay(g, stream, ys)
        for wl, h, t, y in zip(wls, host, tabs, ys):
            acc, yc = Accum(), y.cpu()
            for bs in batch_chunks(wl.B):
                acc.add(yc[bs], oracle.fwd(inputs.act_f64(h[bs]), t.double().numpy(), wl.nH, wl.M, wl.s))
            acc.check(f"graph replay {replay} {wl.name} Y")
    for a in atts:
        a.device_status()
        a.close()


def test_attention_sub_block_graph_replays_match_the_oracle():
    """The 15-launch sub-block sweep of the bench (per Swin-L 224 stage: LayerNorm + qkv
    projection on weights prepared once, the attention, projection + bias + residual) as
    one graph; the block input x is rewritten between replays."""
    stream = torch.cuda.Stream()
    st = []
    for name in L224:
        wl = inputs.BY_NAME[name]
        x, g, be, w, b = inputs.make_producer(wl)
        _, wp, bp, _ = inputs.make_consumer(wl)
        table = inputs.make_table(wl)
        proj = capi.QkvProjection(g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV))
        proj.stats = torch.empty(max(capi.swin_wattn_qkv_stats_bytes(wl.tokens), 16), dtype=torch.uint8,
                                 device=DEV)
        xd = torch.empty(x.shape, dtype=torch.bfloat16, device=DEV)
        st.append(dict(wl=wl, host=(x, g, be, w, b, wp, bp, table), proj=proj, att=plan(wl, table.to(DEV)),
                       x=xd, wp=wp.to(DEV), bp=bp.to(DEV),
                       qkv=torch.empty(wl.B, wl.H, wl.W, 3 * wl.C, dtype=torch.bfloat16, device=DEV),
                       o=torch.empty_like(xd), y=torch.empty_like(xd)))
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step():
        for z in st:
            z["proj"](z["x"], qkv=z["qkv"], status=status)
            z["att"].fwd(z["qkv"], out=z["o"])
            capi.proj_residual(z["o"], z["wp"], z["bp"], z["x"], y=z["y"], status=status)

    for z in st:
        z["x"].copy_(z["host"][0])
    with torch.cuda.stream(stream):
        capi.swin_wattn_launch_count(reset=True)
        step()
        eager = capi.swin_wattn_launch_count(reset=True)
    graph = _capture(stream, step)
    assert eager == 15 and capi.swin_wattn_launch_count() == eager  # the kernels the graph holds
    for replay in range(2):
        xs = []
        for z in st:
            x = z["host"][0] if replay == 0 else (0.5 * inputs.normal(z["host"][0].shape, 77 + z["wl"].stage)
                                                  ).to(torch.bfloat16)
            z["x"].copy_(x)
            xs.append(x)
        _replay(graph, stream, [z["y"] for z in st] + [z["o"] for z in st])
        assert int(status.item()) == 0
        for z, x in zip(st, xs):
            wl = z["wl"]
            _, g, be, w, b, wp, bp, table = z["host"]
            acc, yc = Accum(rounded=True), z["y"].cpu()
            for bs in batch_chunks(wl.B):
                qkv_ref = oracle.qkv_proj(_f64(x[bs]), _f64(g), _f64(be), _f64(w), _f64(b))
                o_ref = oracle.fwd(qkv_ref, table.double().numpy(), wl.nH, wl.M, wl.s)
                acc.add(yc[bs], oracle.proj_residual(o_ref, _f64(wp), _f64(bp), _f64(x[bs])))
            acc.check(f"graph replay {replay} {wl.name} block y")
    for z in st:
        z["att"].close()


def test_training_step_graph_replays_match_the_oracle():
    """Per Swin-B 224 stage: set_bias from the table buffer, the forward (tcgen05 kernel,
    whose tables are rebuilt inside the graph after each set_bias) and the backward with
    the table gradient, as one graph; qkv, dO and the table are rewritten between replays."""
    stream = torch.cuda.Stream()
    st = []
    for name in B224:
        wl = inputs.BY_NAME[name].with_batch(32)
        t = torch.empty((2 * wl.M - 1) ** 2, wl.nH, device=DEV)
        t.copy_(inputs.make_table(wl))
        att = plan(wl, t)
        att.set_fwd_kernel(capi.KERNEL_TCGEN05)
        q = torch.empty(wl.B, wl.H, wl.W, 3 * wl.C, dtype=torch.bfloat16, device=DEV)
        d = torch.empty(wl.B, wl.H, wl.W, wl.C, dtype=torch.bfloat16, device=DEV)
        st.append(dict(wl=wl, att=att, t=t, q=q, d=d, y=torch.empty_like(d), dq=torch.empty_like(q),
                       dt=torch.empty_like(t)))
    torch.cuda.synchronize()

    def step():
        for z in st:
            z["att"].set_bias(z["t"])
            z["att"].fwd(z["q"], out=z["y"])
            z["att"].bwd(z["q"], z["d"], dqkv=z["dq"], dtable=z["dt"])

    graph = _capture(stream, step)
    host_t0 = {z["wl"].name: inputs.make_table(z["wl"]) for z in st}
    for replay, offset in enumerate((0, 300)):
        host = []
        for z in st:
            wl = z["wl"]
            q = inputs.make_qkv(wl, seed_offset=offset)
            d = inputs.normal((wl.B, wl.H, wl.W, wl.C), wl.seed + 2 + offset).to(torch.bfloat16)
            # replay 1: another draw at twice the spread (std 0.04); a stale bias would move
            # the outputs well past the tolerance (checked below on the first images)
            t = inputs.make_table(wl) if replay == 0 else inputs.trunc_normal(
                ((2 * wl.M - 1) ** 2, wl.nH), wl.seed + 91) * 2.0
            z["q"].copy_(q)
            z["d"].copy_(d)
            z["t"].copy_(t)
            host.append((q, d, t))
        _replay(graph, stream, [z[k] for z in st for k in ("y", "dq", "dt")])
        for z, (q, d, t) in zip(st, host):
            wl = z["wl"]
            z["att"].device_status()
            yc, dqc = z["y"].cpu(), z["dq"].cpu()
            acc_y, acc_dq = Accum(), Accum()
            ref_dt = np.zeros(tuple(t.shape))
            for bs in batch_chunks(wl.B):
                acc_y.add(yc[bs], oracle.fwd(inputs.act_f64(q[bs]), t.double().numpy(), wl.nH, wl.M, wl.s))
                rdq, rdt = oracle_bwd(q, d, t, wl, batches=bs)
                acc_dq.add(dqc[bs], rdq)
                ref_dt += rdt
            acc_y.check(f"graph replay {replay} {wl.name} Y")
            if replay == 1:
                stale = oracle.fwd(inputs.act_f64(q[:2]), host_t0[wl.name].double().numpy(), wl.nH, wl.M, wl.s)
                gap = float(abs(yc[:2].double().numpy() - stale).max())
                assert gap > 5e-2, f"the new table changes Y by only {gap:.3g}: the check could miss a stale bias"
            acc_dq.check(f"graph replay {replay} {wl.name} dqkv")
            assert_close(f"graph replay {replay} {wl.name} dtable", z["dt"], ref_dt)
    for z in st:
        z["att"].close()
