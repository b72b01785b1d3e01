"""The producer step with OCP FP8 E4M3 output (swin_wattn_qkv_proj_prepared_fp8) on the GPU,
and the chain producer -> attention on 8-bit operands (swin_wattn_fwd_fp8).

The producer's 8-bit values are decoded on the host and compared with the fp64 oracle's
qkv: each element within one E4M3 ulp of the scaled exact value (the rounding itself, plus
the GEMM step's own error of at most a few thousandths) plus 1e-2; the per-tensor max |qkv|
it reports against the oracle's. The chain is checked under the FP8 reading of the
attention: the FP8 forward must give the attention of the decoded values it was handed,
within the bf16 forward's tolerance."""
import numpy as np
import pytest
import torch

import oracle
from swin_window_attention_gb300 import capi, inputs
from tests.gpu_util import Accum, assert_close, batch_chunks, plan, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_MAX = 448.0


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


def e4m3_ulp(x):
    """The E4M3 unit in the last place at |x|: 2^(e-3) for |x| in [2^e, 2^(e+1)), e >= -6;
    2^-9 below the smallest normal 2^-6."""
    a = np.maximum(np.abs(x), 2.0 ** -6)
    return np.exp2(np.floor(np.log2(a)) - 3.0)


def decoded(q8, scales, C):
    """float64 values scale_t * E4M3 byte for each tensor t of a [..., 3C] uint8 tensor."""
    return inputs.fp8_decoded_f64(q8.cpu().view(torch.float8_e4m3fn), scales, C)


def _producer(wl):
    x, g, be, w, b = inputs.make_producer(wl)
    ref = oracle.qkv_proj(_f64(x), _f64(g), _f64(be), _f64(w), _f64(b))
    C = wl.C
    scales = tuple(float(np.abs(ref[..., t * C:(t + 1) * C]).max()) / FP8_MAX for t in range(3))
    proj = capi.QkvProjection(g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV))
    return x, ref, scales, proj


def _check_producer(name, q8, ref, scales, C):
    dec = decoded(q8, scales, C)
    s = np.concatenate([np.full(C, scales[t]) for t in range(3)])
    bound = s * e4m3_ulp(ref / s) + 1e-2
    excess = float((np.abs(dec - ref) - bound).max())
    assert excess <= 0.0, f"{name}: an element is off its E4M3 bound by {excess:.3g}"
    # most elements are the nearest E4M3 value of the scaled exact value (the others lie
    # within the GEMM step's own error of a rounding boundary)
    nearest = torch.from_numpy(ref / s).to(torch.float8_e4m3fn).to(torch.float64).numpy() * s
    assert float(np.mean(dec != nearest)) < 0.1


@pytest.mark.parametrize("T,C", [(1, 32), (129, 96), (300, 192), (1000, 256), (260, 768), (130, 1536),
                                 (80001, 96)])
def test_fp8_producer_against_oracle(T, C):
    wl = workload(1, 1, T, C, C // 32, 1, 0, seed=T + 3 * C)
    x, ref, scales, proj = _producer(wl)
    amax = torch.zeros(3, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q8 = proj.fp8(x.to(DEV), scales, amax=amax, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert q8.dtype == torch.uint8 and q8.shape == (1, 1, T, 3 * C)
    _check_producer(f"qkv8 T={T} C={C}", q8, ref, scales, C)
    ref_amax = [float(np.abs(ref[..., t * C:(t + 1) * C]).max()) for t in range(3)]
    for t in range(3):
        assert abs(float(amax[t]) - ref_amax[t]) <= 1e-2 + 2.0 ** -8 * ref_amax[t]


def test_fp8_producer_is_deterministic_and_amax_accumulates():
    wl = workload(2, 14, 14, 192, 6, 7, 3, seed=21)
    x, ref, scales, proj = _producer(wl)
    xd = x.to(DEV)
    amax = torch.zeros(3, dtype=torch.float32, device=DEV)
    a = proj.fp8(xd, scales, amax=amax)
    first = amax.clone()
    b = proj.fp8(xd, [2 * v for v in scales], amax=amax)  # other scales, same values
    c = proj.fp8(xd, scales)
    torch.cuda.synchronize()
    assert torch.equal(a, c) and not torch.equal(a, b)
    assert torch.equal(first, amax)  # max-ed, not summed


@pytest.mark.parametrize("name", ["smoke", "swin_l224_s1"])
def test_fp8_producer_then_fp8_attention(name):
    """x -> LayerNorm + qkv projection to E4M3 -> the FP8 forward, against the oracle's
    attention of the decoded qkv the forward was handed (every image). The scales come from
    the producer's own max |qkv| of a first pass (delayed scaling)."""
    wl = workload(2, 14, 21, 96, 3, 7, 3, seed=23) if name == "smoke" else inputs.BY_NAME[name]
    x, g, be, w, b = inputs.make_producer(wl)
    proj = capi.QkvProjection(g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV))
    xd = x.to(DEV)
    amax = torch.zeros(3, dtype=torch.float32, device=DEV)
    proj.fp8(xd, (1.0, 1.0, 1.0), amax=amax)
    scales = tuple(float(a) / FP8_MAX for a in amax.cpu())
    ref = oracle.qkv_proj(_f64(x[:2]), _f64(g), _f64(be), _f64(w), _f64(b))
    table = inputs.make_table(wl)
    q8 = proj.fp8(xd, scales)
    att = plan(wl, table.to(DEV))
    y = att.fwd_fp8(q8, scales)
    att.device_status()
    att.close()
    q8c, yc = q8.cpu(), y.cpu()
    _check_producer(f"{name} qkv8", q8c[:2], ref[:2], scales, wl.C)
    acc = Accum()
    for bs in batch_chunks(wl.B):
        dec = decoded(q8c[bs[0]:bs[-1] + 1], scales, wl.C)
        acc.add(yc[bs], oracle.fwd(dec, table.double().numpy(), wl.nH, wl.M, wl.s))
    acc.check(f"{name} Y from the FP8 producer")


def test_fp8_producer_error_paths():
    C, T = 96, 4
    wl = workload(1, 1, T, C, 3, 1, 0, seed=5)
    x, g, be, w, b = inputs.make_producer(wl)
    proj = capi.QkvProjection(g.to(DEV), be.to(DEV), w.to(DEV), b.to(DEV))
    xd = x.to(DEV)
    q8 = torch.empty(1, 1, T, 3 * C, dtype=torch.uint8, device=DEV)
    st = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(max(capi.swin_wattn_qkv_stats_bytes(T), 16), dtype=torch.uint8, device=DEV)
    call = lambda sq, sk, sv, tokens=T, wsb=ws.numel(): capi.swin_wattn_qkv_proj_prepared_fp8(
        xd.data_ptr(), proj.prepared.data_ptr(), q8.data_ptr(), tokens, C, 1e-5, sq, sk, sv, None, ws.data_ptr(),
        wsb, None, st)
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-45):
        assert call(bad, 1.0, 1.0) == capi.ERR_INVALID_ARG
        assert call(1.0, 1.0, bad) == capi.ERR_INVALID_ARG
    assert call(1.0, 1.0, 1.0, tokens=0) == capi.OK
    assert call(1.0, 1.0, 1.0, tokens=-1) == capi.ERR_INVALID_ARG
    assert call(1.0, 1.0, 1.0, wsb=0) == capi.ERR_INVALID_ARG
    assert call(1.0, 1.0, 1.0) == capi.OK
    torch.cuda.synchronize()
