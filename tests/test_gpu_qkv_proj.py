"""The producer step (LayerNorm over C, then the qkv projection) on the GPU against the
fp64 oracle, through the C ABI: ragged token counts, every Swin channel width, the
full-size Swin-L 224 stages on every image, the chain producer -> attention against the
oracle's chain, and the error paths."""
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, assert_close_rounded, batch_chunks, plan, workload

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


# qkv values grow with sqrt(C) (|qkv| reaches ~3 at C = 1536 with W ~ 0.02): the bound
# is 1e-2 plus one bf16 ulp of the value (tests.gpu_util.assert_close_rounded).
assert_close_qkv = assert_close_rounded


def _run(x, g, be, w, b, eps=1e-5):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = capi.qkv_proj(x.to(DEV), g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV), eps=eps, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y


@pytest.mark.parametrize("T,C", [(1, 32), (127, 96), (129, 128), (300, 192), (1000, 256), (77, 384),
                                 (260, 768), (130, 1536), (4096, 192), (555, 160)])
def test_qkv_proj_against_oracle(T, C):
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=T + C)
    x, g, be, w, b = inputs.make_producer(wl)
    y = _run(x, g, be, w, b)
    assert y.shape == (1, 1, T, 3 * C) and y.dtype == torch.bfloat16
    assert_close_qkv("qkv", y, oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b)))


@pytest.mark.parametrize("name", ["swin_l224_s1", "swin_l224_s2", "swin_l224_s3", "swin_l224_s4"])
def test_qkv_proj_full_size_workloads(name):
    wl = inputs.BY_NAME[name]
    x, g, be, w, b = inputs.make_producer(wl)
    y = _run(x, g, be, w, b).cpu()
    acc = Accum(rounded=True)
    for bs in batch_chunks(wl.B):
        acc.add(y[bs], oracle.qkv_proj(_f64(x[bs]), _f64(g), _f64(be), _f64(w), _f64(b)))
    acc.check(f"{name} qkv")


@pytest.mark.parametrize("C", [160, 96])
def test_qkv_proj_many_tokens_statistics_on_chip(C):
    """Enough tokens (over four 128-token tiles per SM) that every token tile is one work
    item and the statistics are summed from the staged x tiles; C not a multiple of the
    64-channel chunk (zero-filled tail), a ragged last token tile and a large common offset
    per token. Compared on sampled rows (the operation is row-independent)."""
    T = 80001
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=C)
    x, g, be, w, b = inputs.make_producer(wl)
    x = (x.float() * 3.0 + 20.0).to(torch.bfloat16)
    y = _run(x, g, be, w, b).cpu().reshape(T, 3 * C)
    xs = x.reshape(T, C)
    gen = torch.Generator().manual_seed(C)
    rows = torch.cat([torch.arange(0, 256), torch.randint(256, T - 256, (512,), generator=gen),
                      torch.arange(T - 256, T)])
    ref = oracle.qkv_proj(_f64(xs[rows]), _f64(g), _f64(be), _f64(w), _f64(b))
    assert_close_qkv(f"qkv T={T} C={C} (sampled rows)", y[rows], ref)


def test_qkv_proj_is_deterministic_and_large_offsets_are_stable():
    """x with a large common offset per token (LayerNorm must remove it) and a wide spread."""
    wl = workload(2, 14, 14, 192, 6, 7, 3, seed=5)
    x, g, be, w, b = inputs.make_producer(wl)
    x = (x.float() * 4.0 + 30.0).to(torch.bfloat16)
    y1 = _run(x, g, be, w, b)
    y2 = _run(x, g, be, w, b)
    assert torch.equal(y1, y2)
    assert_close_qkv("qkv", y1, oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b)))


def test_producer_then_attention_matches_the_oracle_chain():
    """LayerNorm + qkv projection, then the shifted-window attention, against the oracle's
    two steps (the attention oracle applied to the oracle's fp64 qkv)."""
    wl = workload(2, 14, 21, 96, 3, 7, 3, seed=11)
    x, g, be, w, b = inputs.make_producer(wl)
    table = inputs.make_table(wl)
    qkv = _run(x, g, be, w, b)
    att = plan(wl, table.to(DEV))
    y = att.fwd(qkv)
    torch.cuda.synchronize()
    att.close()
    qkv_ref = oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b))
    assert_close("Y", y, oracle.fwd(qkv_ref, table.double().numpy(), wl.nH, wl.M, wl.s))


def test_qkv_proj_error_paths():
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device=DEV)
    v = torch.zeros(288, dtype=torch.float32, device=DEV)
    w = torch.zeros(288, 96, dtype=torch.bfloat16, device=DEV)
    out = torch.full((4, 288), 3.0, dtype=torch.bfloat16, device=DEV)
    nws = capi.swin_wattn_qkv_workspace_bytes(96, 4)
    assert nws >= 288 * 96 * 2 + 2 * 288 * 4 + 4 * 8
    assert capi.swin_wattn_qkv_workspace_bytes(80, 4) == 0
    ws = torch.empty(nws, dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    f = lambda xp, T, C, nb: capi.swin_wattn_qkv_proj(xp, v.data_ptr(), v.data_ptr(), w.data_ptr(), v.data_ptr(),
                                                      out.data_ptr(), T, C, 1e-5, ws.data_ptr(), nb, None, s)
    assert f(x.data_ptr(), 0, 96, nws) == capi.OK
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)  # no tokens: nothing written
    assert f(x.data_ptr(), 4, 80, nws) == capi.ERR_UNSUPPORTED
    assert f(x.data_ptr(), -1, 96, nws) == capi.ERR_INVALID_ARG
    assert f(x.data_ptr(), 4, 96, nws - 16) == capi.ERR_INVALID_ARG  # workspace too small
    host = torch.zeros(4, 96, dtype=torch.bfloat16)
    assert f(host.data_ptr(), 4, 96, nws) == capi.ERR_INVALID_ARG
    assert f(x.data_ptr() + 2, 4, 96, nws) == capi.ERR_MISALIGNED


@pytest.mark.parametrize("T,C", [(300, 192), (3136, 1536), (80001, 96)])
def test_prepared_weights_give_the_same_bits(T, C):
    """Weights prepared once, then two different inputs: bit-identical to the one-call form
    (statistics from the prep pass at 300 and 3136 tokens, on chip at 80001)."""
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=3 * T + C)
    x, g, be, w, b = inputs.make_producer(wl)
    gd, bed, wd, bd = g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV)
    proj = capi.QkvProjection(gd, bed, wd, bd)
    for xi in (x, (x.float() * 0.5 - 1.0).to(torch.bfloat16)):
        xd = xi.to(DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        y1 = proj(xd, status=status)
        y2 = capi.qkv_proj(xd, gd, bed, wd, bd, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(y1, y2)
    if T <= 4096:
        assert_close_qkv("qkv (prepared)", y1, oracle.qkv_proj(_f64(xi), _f64(g), _f64(be), _f64(w), _f64(b)))


def test_prepared_error_paths():
    C, T = 96, 4
    v = torch.zeros(3 * C, dtype=torch.float32, device=DEV)
    w = torch.zeros(3 * C, C, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros(T, C, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(T, 3 * C, dtype=torch.bfloat16, device=DEV)
    npb = capi.swin_wattn_qkv_prepared_bytes(C)
    nst = capi.swin_wattn_qkv_stats_bytes(T)
    assert npb >= 3 * C * C * 2 + 2 * 3 * C * 4 and nst >= T * 8
    assert capi.swin_wattn_qkv_prepared_bytes(80) == 0
    prep = torch.empty(npb, dtype=torch.uint8, device=DEV)
    st = torch.empty(nst, dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    pr = lambda C_, nb: capi.swin_wattn_qkv_prepare(v.data_ptr(), v.data_ptr(), w.data_ptr(), v.data_ptr(), C_,
                                                    prep.data_ptr(), nb, s)
    assert pr(80, npb) == capi.ERR_UNSUPPORTED
    assert pr(C, npb - 256) == capi.ERR_INVALID_ARG
    assert pr(C, npb) == capi.OK
    f = lambda T_, nb, sp: capi.swin_wattn_qkv_proj_prepared(x.data_ptr(), prep.data_ptr(), out.data_ptr(), T_, C,
                                                             1e-5, sp, nb, None, s)
    assert f(T, nst - 8, st.data_ptr()) == capi.ERR_INVALID_ARG
    assert f(-1, nst, st.data_ptr()) == capi.ERR_INVALID_ARG
    assert f(T, nst, st.data_ptr() + 8) == capi.ERR_MISALIGNED
    assert f(T, nst, st.data_ptr()) == capi.OK
    torch.cuda.synchronize()
    assert torch.all(out == 0)  # zero weights and biases
