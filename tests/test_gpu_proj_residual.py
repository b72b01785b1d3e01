"""The consumer step (the output projection, then its bias and the residual added) on the
GPU against the fp64 oracle, through the C ABI: ragged token counts, every Swin channel
width, the full-size Swin-L 224 stages on every image, many tokens on sampled rows,
the result written over the residual, the attention sub-block chain (producer ->
attention -> consumer) against the oracle's chain, and the error paths."""
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close_rounded, batch_chunks, plan, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


def _run(o, wp, bp, r, y=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = capi.proj_residual(o, wp, bp, r, y=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y


def _dev(*ts):
    return [t.to(DEV) for t in ts]


@pytest.mark.parametrize("T,C", [(1, 32), (127, 96), (129, 128), (300, 192), (1000, 256), (77, 384),
                                 (555, 160), (260, 768), (130, 1536), (4096, 192), (3136, 1024)])
def test_proj_residual_against_oracle(T, C):
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=T + C)
    o, wp, bp, r = inputs.make_consumer(wl)
    y = _run(*_dev(o, wp, bp, r))
    assert y.shape == (1, 1, T, C) and y.dtype == torch.bfloat16
    assert_close_rounded("y", y, oracle.proj_residual(_f64(o), _f64(wp), _f64(bp), _f64(r)))


@pytest.mark.parametrize("name", ["swin_l224_s1", "swin_l224_s2", "swin_l224_s3", "swin_l224_s4"])
def test_proj_residual_full_size_workloads(name):
    wl = inputs.BY_NAME[name]
    o, wp, bp, r = inputs.make_consumer(wl)
    y = _run(*_dev(o, wp, bp, r)).cpu()
    acc = Accum(rounded=True)
    for bs in batch_chunks(wl.B):
        acc.add(y[bs], oracle.proj_residual(_f64(o[bs]), _f64(wp), _f64(bp), _f64(r[bs])))
    acc.check(f"{name} y")


def test_proj_residual_many_tokens_sampled_rows():
    """Over four 128-token tiles per SM (one work item per token tile) with a ragged last
    tile; compared on sampled rows (the operation is row-independent)."""
    T, C = 80001, 96
    wl = workload(1, 1, T, C, 3, 1, 0, seed=17)
    o, wp, bp, r = inputs.make_consumer(wl)
    y = _run(*_dev(o, wp, bp, r)).cpu().reshape(T, C)
    gen = torch.Generator().manual_seed(3)
    rows = torch.cat([torch.arange(0, 256), torch.randint(256, T - 256, (512,), generator=gen),
                      torch.arange(T - 256, T)])
    o2, r2 = o.reshape(T, C)[rows], r.reshape(T, C)[rows]
    assert_close_rounded("y (sampled rows)", y[rows], oracle.proj_residual(_f64(o2), _f64(wp), _f64(bp), _f64(r2)))


def test_proj_residual_in_place_over_the_residual_and_deterministic():
    wl = workload(2, 14, 14, 384, 12, 7, 3, seed=5)
    o, wp, bp, r = inputs.make_consumer(wl)
    od, wd, bd, rd = _dev(o, wp, bp, r)
    y1 = _run(od, wd, bd, rd)
    y2 = _run(od, wd, bd, rd)
    assert torch.equal(y1, y2)
    rd2 = rd.clone()
    y3 = _run(od, wd, bd, rd2, y=rd2)  # written over its own residual
    assert y3.data_ptr() == rd2.data_ptr() and torch.equal(y3, y1)


def test_attention_sub_block_matches_the_oracle_chain():
    """x -> LayerNorm + qkv projection -> shifted-window attention -> projection + bias +
    residual x, against the oracle's three steps on fp64 intermediates."""
    wl = workload(2, 14, 21, 96, 3, 7, 3, seed=13)
    x, g, be, w, b = inputs.make_producer(wl)
    _, wp, bp, _ = inputs.make_consumer(wl)
    table = inputs.make_table(wl)
    xd, gd, bed, wd, bd, wpd, bpd = _dev(x, g, be, w, b, wp, bp)
    qkv = capi.qkv_proj(xd, gd, bed, wd, bd)
    att = plan(wl, table.to(DEV))
    o = att.fwd(qkv)
    y = _run(o, wpd, bpd, xd)
    att.close()
    qkv_ref = oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b))
    o_ref = oracle.fwd(qkv_ref, table.double().numpy(), wl.nH, wl.M, wl.s)
    assert_close_rounded("block y", y, oracle.proj_residual(o_ref, _f64(wp), _f64(bp), _f64(x)))


def test_proj_residual_error_paths():
    o = torch.zeros(4, 96, dtype=torch.bfloat16, device=DEV)
    r = torch.zeros(4, 96, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(96, 96, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(96, dtype=torch.float32, device=DEV)
    y = torch.full((4, 96), 3.0, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    f = lambda op, yp, T, C: capi.swin_wattn_proj_residual(op, w.data_ptr(), b.data_ptr(), r.data_ptr(), yp, T, C,
                                                           None, s)
    assert f(o.data_ptr(), y.data_ptr(), 0, 96) == capi.OK
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)  # no tokens: nothing written
    assert f(o.data_ptr(), y.data_ptr(), 4, 80) == capi.ERR_UNSUPPORTED
    assert f(o.data_ptr(), y.data_ptr(), -1, 96) == capi.ERR_INVALID_ARG
    assert f(o.data_ptr(), o.data_ptr(), 4, 96) == capi.ERR_INVALID_ARG          # y is o
    assert f(o.data_ptr(), o.data_ptr() + 192, 4, 96) == capi.ERR_INVALID_ARG    # y overlaps o
    host = torch.zeros(4, 96, dtype=torch.bfloat16)
    assert f(host.data_ptr(), y.data_ptr(), 4, 96) == capi.ERR_INVALID_ARG
    assert f(o.data_ptr() + 2, y.data_ptr(), 4, 96) == capi.ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


def test_gemm_steps_count_their_launches():
    """The launch accounting covers the GEMM entry points: the one-call producer launches
    the fold and the product, the prepared producer the product after at most one
    statistics pass, and the consumer one kernel."""
    wl = workload(1, 1, 300, 96, 3, 1, 0, seed=21)
    x, g, be, w, b = _dev(*inputs.make_producer(wl))
    o, wp, bp, r = _dev(*inputs.make_consumer(wl))
    proj = capi.QkvProjection(g, be, w, b)
    torch.cuda.synchronize()
    capi.swin_wattn_launch_count(reset=True)
    capi.qkv_proj(x, g, be, w, b)
    assert capi.swin_wattn_launch_count(reset=True) == 2
    proj(x)
    assert capi.swin_wattn_launch_count(reset=True) in (1, 2)
    capi.proj_residual(o, wp, bp, r)
    assert capi.swin_wattn_launch_count(reset=True) == 1
    torch.cuda.synchronize()
