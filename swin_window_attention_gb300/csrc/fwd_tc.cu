// Fused (shifted-)window attention forward on the fifth-generation tensor cores
// (tcgen05 + tensor memory) for 7x7 windows and bf16 tensors.
//
// The same single fused pass as the mma.sync kernel (roll, partition, Q K^T, bias, mask,
// softmax, P V, reverse and un-roll in one kernel: NVIDIA Swin talk transcript, uticex.com
// article 1598, sections 2 and 3; Baidu AIAK-Training talk, jxzklqfsx.com article 743345,
// section 2), laid out for tcgen05:
//
// * A CTA (4 warps) owns one head and a range of windows, taken two at a time. The two
//   windows' 49 query rows, each padded to 64, stack into one M = 128 MMA: lane r of
//   tensor memory holds query row r, and thread r (warp r / 32 reaches lanes 32w..32w+31)
//   owns that row for the whole softmax: no shuffles, no fragment bookkeeping.
// * S = Q K^T: two M128 N64 K32 MMAs (one per window's keys) into tensor-memory columns
//   [0, 128); a boundary window adds its shift mask with one more K16 MMA (the rank-4
//   product of a one-hot region matrix U and a per-class matrix V, exact to 2e-4 of the
//   -100 logit offset).
// * Thread r loads its 49 logits, adds the relative-position bias (staged once per CTA
//   from the plan's dense bias), takes max and exp2, and writes the bf16 row of P to
//   tensor memory, where the P V MMA reads its A operand.
// * O = P V: eight M128 N48 K16 MMAs over both windows' keys (the other window's block of
//   P is zero). Columns 32..47 of the V operand are a ones column and zeros, so O column
//   32 is the row sum of the very bf16 P that weighted V.
// * q/k/v head slices are gathered with 16-byte cp.async straight from the rolled token
//   positions into core-matrix tiles, three window pairs deep; while thread r finishes pair
//   n, the tensor core already runs pair n + 1's Q K^T.
//
// One thread issues every MMA; completion reaches the others through two mbarriers. All
// waits are bounded (1 s): a wait that runs out sets the plan's error word and the CTA
// leaves after releasing its tensor memory.
#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kTM = 7, kTN = 49;
constexpr int kTHREADS = 128;
constexpr int kQK_TILE = 64 * 64;             // q or k: 8 row groups x 4 chunks x 128 B
constexpr int kV_GROUP = 6 * 128;             // v row group: 4 data chunks, ones, zeros
constexpr int kV_TILE = 8 * kV_GROUP;         // 6144 B
constexpr int kOFF_K = 2 * kQK_TILE;          // stage layout: q_a q_b | k_a k_b | v_a v_b
constexpr int kOFF_V = 4 * kQK_TILE;
constexpr int kSTAGE = 4 * kQK_TILE + 2 * kV_TILE;  // 28672 B
constexpr int kSTAGES = 3;
constexpr int kBIAS_STRIDE = 52;              // floats per bias row (13 x 16 B)
constexpr int kBIAS_BYTES = 64 * kBIAS_STRIDE * 4;
constexpr int kU_BYTES = 128 * 16 * 2;        // U: 128 rows x K16
constexpr int kVC_BYTES = 64 * 16 * 2;        // V of one boundary class: 64 keys x K16
constexpr int kOFF_BIAS = kSTAGES * kSTAGE;
constexpr int kOFF_U = kOFF_BIAS + kBIAS_BYTES;
constexpr int kOFF_VC = kOFF_U + kU_BYTES;
constexpr int kOFF_BAR = kOFF_VC + 3 * kVC_BYTES;
constexpr int kSMEM = kOFF_BAR + 64;
// Tensor memory: S [0, 128) (window a keys, window b keys), O [128, 176), P [192, 256).
constexpr int kTMEM_COLS = 256;
constexpr int kS_COL = 0, kO_COL = 128, kP_COL = 192;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

static_assert(kSMEM * 3 > 233472, "at most two CTAs per SM: each holds half the tensor memory");
static_assert(kP_COL + 64 <= kTMEM_COLS, "tensor memory layout");

// Byte offset of 16-byte chunk c of row r in a q/k tile, and in a v tile.
__device__ __forceinline__ uint32_t qk_off(int r, int c) { return (r >> 3) * 512 + c * 128 + (r & 7) * 16; }
__device__ __forceinline__ uint32_t v_off(int r, int c) { return (r >> 3) * kV_GROUP + c * 128 + (r & 7) * 16; }
// Byte offset of bf16 element (r, k) in a K16 tile (U, or a class V).
__device__ __forceinline__ uint32_t k16_off(int r, int k) {
  return (r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

struct TcParams {
  const __nv_bfloat16* qkv;
  __nv_bfloat16* out;
  const float* dense_bias;  // [nH, 49, 49]
  int* err;                 // plan error word (bit 0: a wait ran out)
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;
  int chunks;
  float qk_scale_log2;  // hd^-0.5 * log2(e)
};

__global__ void __launch_bounds__(kTHREADS, 1) fwd_tc_kernel(const TcParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* sbias = reinterpret_cast<float*>(smem + kOFF_BIAS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 16);
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar_s = smem_u32(&bars[0]), bar_o = smem_u32(&bars[1]);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int npair = (nwin + 1) >> 1;
  const int C3 = 3 * p.C, H = p.H, W = p.W, s = p.s;

  if (warp == 0) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::mbar_init_fence();
  }

  // ---- gather slots: 16-byte chunk c of window slot i, the same for q, k and v ------
  constexpr int TCH = kTN * 4, TI = (TCH + kTHREADS - 1) / kTHREADS;
  uint32_t qk_soff[TI], v_soff[TI];
  int ld_rc[TI], ld_chan[TI];
#pragma unroll
  for (int j = 0; j < TI; ++j) {
    const int id = tid + j * kTHREADS;
    const int c = id & 3, i = (id >> 2) < kTN ? (id >> 2) : 0;
    qk_soff[j] = qk_off(i, c);
    v_soff[j] = v_off(i, c);
    ld_rc[j] = ((i / kTM) << 8) | (i % kTM);
    ld_chan[j] = h * kHeadDim + c * 8;
  }
  int lb, lwy, lwx;  // cursor of the next window to load
  {
    lb = (int)(w_begin / p.nW);
    const int w = (int)(w_begin - (int64_t)lb * p.nW);
    lwy = w / p.nWx;
    lwx = w - lwy * p.nWx;
  }
  int cb = lb, cwy = lwy, cwx = lwx;  // cursor of the first window of the pair being computed
  const __nv_bfloat16* __restrict__ qkv = p.qkv;

  auto issue_window = [&](uint32_t qk_base, uint32_t v_base) {
    const int y0 = lwy * kTM + s, x0 = lwx * kTM + s;
    const int hy = H - y0, hx = W - x0;  // rows ly >= hy / columns lx >= hx wrap around
    const __nv_bfloat16* wbase = qkv + (((int64_t)lb * H + y0) * W + x0) * C3;
#pragma unroll
    for (int j = 0; j < TI; ++j) {
      if (j < TI - 1 || tid + j * kTHREADS < TCH) {
        const int ly = ld_rc[j] >> 8, lx = ld_rc[j] & 255;
        int64_t rel = (int64_t)ly * W + lx;
        if (ly >= hy) rel -= (int64_t)H * W;
        if (lx >= hx) rel -= W;
        const __nv_bfloat16* src = wbase + rel * C3 + ld_chan[j];
        cp_async_16(qk_base + qk_soff[j], src);
        cp_async_16(qk_base + kOFF_K + qk_soff[j], src + p.C);
        cp_async_16(v_base + v_soff[j], src + 2 * p.C);
      }
    }
    if (++lwx == p.nWx) {
      lwx = 0;
      if (++lwy == p.nWy) {
        lwy = 0;
        ++lb;
      }
    }
  };
  auto issue_pair = [&](int pair, int stage) {
    const uint32_t base = smem0 + stage * kSTAGE;
    issue_window(base, base + kOFF_V);
    if (2 * pair + 1 < nwin) issue_window(base + kQK_TILE, base + kOFF_V + kV_TILE);
  };

#pragma unroll
  for (int st = 0; st < kSTAGES; ++st) {
    if (st < npair) issue_pair(st, st);
    cp_async_commit();
  }

  // ---- constant shared data: padding rows, the ones column, bias, mask operands -----
  for (int e = tid; e < kSTAGES * 15 * 4 * 4; e += kTHREADS) {  // q/k rows 49..63
    const int c = e & 3, r = 49 + (e >> 2) % 15, tile = (e >> 2) / 15;
    *reinterpret_cast<uint4*>(smem + (tile >> 2) * kSTAGE + (tile & 3) * kQK_TILE + qk_off(r, c)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  for (int e = tid; e < kSTAGES * 2 * 64 * 6; e += kTHREADS) {  // v: padding, ones, zeros
    const int c = e % 6, r = (e / 6) & 63, tile = e / 384;
    if (c < 4 && r < kTN) continue;  // data chunks: written by the gather
    *reinterpret_cast<uint4*>(smem + (tile >> 1) * kSTAGE + kOFF_V + (tile & 1) * kV_TILE + v_off(r, c)) =
        make_uint4(c == 4 ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
  {
    const float* db = p.dense_bias + (int64_t)h * kTN * kTN;
    for (int e = tid; e < 64 * kBIAS_STRIDE; e += kTHREADS) {
      const int i = e / kBIAS_STRIDE, j = e % kBIAS_STRIDE;
      sbias[e] = (i < kTN && j < kTN) ? db[i * kTN + j] * kLog2e : 0.0f;
    }
  }
  if (s > 0) {
    for (int e = tid; e < 128 * 8; e += kTHREADS) {  // U: -100 where k & 3 is the row's region
      const int r = e >> 3, k = 2 * (e & 7), i = r & 63;
      const int c = (i / kTM >= kTM - s ? 2 : 0) | (i % kTM >= kTM - s ? 1 : 0);
      uint32_t w = 0u;
      if (i < kTN && k < 8) w = (((k & 3) == c) ? kMaskUBits : 0u) | (((k + 1) & 3) == c ? kMaskUBits << 16 : 0u);
      *reinterpret_cast<uint32_t*>(smem + kOFF_U + k16_off(r, k)) = w;
    }
    for (int e = tid; e < 3 * 64 * 8; e += kTHREADS) {  // V of classes 1..3
      const int cls = 1 + (e >> 9), j = (e >> 3) & 63, k = 2 * (e & 7);
      const uint32_t w = mask_v_bits(cls, j, k, H, W, kTM, s) | (mask_v_bits(cls, j, k + 1, H, W, kTM, s) << 16);
      *reinterpret_cast<uint32_t*>(smem + kOFF_VC + (cls - 1) * kVC_BYTES + k16_off(j, k)) = w;
    }
  }

  // ---- per-thread row ---------------------------------------------------------------
  const int win = tid >> 6, i = tid & 63;  // window of the pair (warp-uniform) and slot
  const int ly = i / kTM, lx = i % kTM;
  const float c_l2 = p.qk_scale_log2;
  const float* brow = sbias + i * kBIAS_STRIDE;

  cp_async_wait<kSTAGES - 1>();  // pair 0 landed (own copies)
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
  {
    // the other window's half of this row of P stays zero for the whole kernel
    uint32_t z[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) z[q] = 0u;
    tc::st_x32(trow + kP_COL + 32 * (1 - win), z);
    tc::wait_st();
  }

  const uint32_t idesc_qk = tc::idesc_bf16(128, 64, false);
  const uint32_t idesc_pv = tc::idesc_bf16(128, 48, true);
  // Window class of the two windows of a pair (0 = interior or no shift).
  auto wclass = [&](int wy, int wx) {
    return s > 0 ? ((wy == p.nWy - 1 ? 2 : 0) | (wx == p.nWx - 1 ? 1 : 0)) : 0;
  };
  auto issue_qk = [&](int stage, int cls_a, int cls_b, bool has_b) {
    const uint32_t base = smem0 + stage * kSTAGE;
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      if (w2 == 1 && !has_b) break;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        tc::mma_ss(tmem + kS_COL + 64 * w2, tc::sdesc(base + kk * 256, 128, 512),
                   tc::sdesc(base + kOFF_K + w2 * kQK_TILE + kk * 256, 128, 512), idesc_qk, kk > 0);
      const int cls = w2 ? cls_b : cls_a;
      if (cls)
        tc::mma_ss(tmem + kS_COL + 64 * w2, tc::sdesc(smem0 + kOFF_U, 128, 256),
                   tc::sdesc(smem0 + kOFF_VC + (cls - 1) * kVC_BYTES, 128, 256), idesc_qk, true);
    }
    tc::commit(bar_s);
  };
  auto issue_pv = [&](int stage, bool has_b) {
    const uint32_t vbase = smem0 + stage * kSTAGE + kOFF_V;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if (kk >= 4 && !has_b) break;
      tc::mma_ts(tmem + kO_COL, tmem + kP_COL + 8 * kk,
                 tc::sdesc(vbase + (kk >> 2) * kV_TILE + (kk & 3) * 2 * kV_GROUP, kV_GROUP, 128), idesc_pv, kk > 0);
    }
    tc::commit(bar_o);
  };
  // Window coordinates after the pair's first window.
  auto next_window = [&](int& b, int& wy, int& wx) {
    if (++wx == p.nWx) {
      wx = 0;
      if (++wy == p.nWy) {
        wy = 0;
        ++b;
      }
    }
  };

  if (tid == 0 && npair > 0) {
    tc::fence_after_sync();
    int b2 = cb, wy2 = cwy, wx2 = cwx;
    next_window(b2, wy2, wx2);
    issue_qk(0, wclass(cwy, cwx), wclass(wy2, wx2), nwin > 1);
  }

  int bad = 0;
  int stage = 0;
  for (int n = 0; n < npair; ++n) {
    // this thread's window and token
    int b = cb, wy = cwy, wx = cwx;
    if (win) next_window(b, wy, wx);
    const bool has_b = 2 * n + 1 < nwin;
    const bool active = i < kTN && (win == 0 || has_b);

    // ---- softmax of row i over its window's 49 keys ---------------------------------
    bool ok = tc::mbar_wait(bar_s, n & 1, kWaitLimitNs);
    tc::fence_after_sync();
    uint32_t sa[32], sb[16], sc;
    tc::ld49_wait(trow + kS_COL + 64 * win, sa, sb, sc);
    float y[kTN];
    {
      const float2 c2 = make_float2(c_l2, c_l2);
      const float4* b4 = reinterpret_cast<const float4*>(brow);
#pragma unroll
      for (int q = 0; q < 12; ++q) {
        const float4 bb = b4[q];
        const uint32_t* src = q < 8 ? &sa[4 * q] : &sb[4 * (q - 8)];
        const float2 e0 = __ffma2_rn(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])), c2,
                                     make_float2(bb.x, bb.y));
        const float2 e1 = __ffma2_rn(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])), c2,
                                     make_float2(bb.z, bb.w));
        y[4 * q] = e0.x;
        y[4 * q + 1] = e0.y;
        y[4 * q + 2] = e1.x;
        y[4 * q + 3] = e1.y;
      }
      y[48] = fmaf(__uint_as_float(sc), c_l2, brow[48]);
    }
    float ma = y[48], mb = y[47];
#pragma unroll
    for (int q = 0; q < 46; q += 4) {
      ma = fmax3(ma, y[q], y[q + 1]);
      mb = fmax3(mb, y[q + 2], y[q + 3]);
    }
    ma = fmax3(ma, mb, y[46]);
    uint32_t pw[32];
    {
      const float2 nm = make_float2(-ma, -ma);
#pragma unroll
      for (int q = 0; q < 24; ++q) {
        const float2 d = __fadd2_rn(make_float2(y[2 * q], y[2 * q + 1]), nm);
        pw[q] = pack_bf16(fast_exp2(d.x), fast_exp2(d.y));
      }
      pw[24] = pack_bf16(fast_exp2(y[48] - ma), 0.0f);
#pragma unroll
      for (int q = 25; q < 32; ++q) pw[q] = 0u;
    }
    tc::st_x32(trow + kP_COL + 32 * win, pw);
    tc::wait_st();
    if (n + 1 < npair) cp_async_wait<kSTAGES - 2>();  // pair n + 1 landed (own copies)
    tc::fence_proxy_async();
    tc::fence_before_sync();
    bad = __syncthreads_or(bad | (ok ? 0 : 1));
    if (bad) break;

    // ---- one thread: P V of this pair, then Q K^T of the next ------------------------
    const int next_stage = stage + 1 == kSTAGES ? 0 : stage + 1;
    if (tid == 0) {
      tc::fence_after_sync();
      issue_pv(stage, has_b);
      if (n + 1 < npair) {
        int b1 = cb, wy1 = cwy, wx1 = cwx;
        next_window(b1, wy1, wx1);
        next_window(b1, wy1, wx1);
        int b2 = b1, wy2 = wy1, wx2 = wx1;
        next_window(b2, wy2, wx2);
        issue_qk(next_stage, wclass(wy1, wx1), wclass(wy2, wx2), 2 * n + 3 < nwin);
      }
    }

    // ---- epilogue: O / rowsum to the token this row was read from --------------------
    ok = tc::mbar_wait(bar_o, n & 1, kWaitLimitNs);
    tc::fence_after_sync();
    uint32_t o[32], osum;
    tc::ld33_wait(trow + kO_COL, o, osum);
    bad |= ok ? 0 : 1;
    if (active && ok) {
      const float inv = 1.0f / __uint_as_float(osum);
      const float2 i2 = make_float2(inv, inv);
      int yy = wy * kTM + ly + s, xx = wx * kTM + lx + s;
      yy = yy >= H ? yy - H : yy;
      xx = xx >= W ? xx - W : xx;
      const int64_t tok = ((int64_t)b * H + yy) * W + xx;
      uint4* dst = reinterpret_cast<uint4*>(p.out + tok * p.C + h * kHeadDim);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[8 * q + 2 * u]), __uint_as_float(o[8 * q + 2 * u + 1])), i2);
          w4[u] = pack_bf16(v.x, v.y);
        }
        dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    // the pair's stage is free: both of its MMAs have completed
    if (n + kSTAGES < npair) issue_pair(n + kSTAGES, stage);
    cp_async_commit();
    next_window(cb, cwy, cwx);
    next_window(cb, cwy, cwx);
    stage = next_stage;
  }
  if (bad) atomicOr(p.err, 1);

  cp_async_wait<0>();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

}  // namespace

// ---- host side ---------------------------------------------------------------------

bool fwd_tc_applies(const Plan& pl) { return pl.M == kTM && pl.dtype == SWIN_WATTN_BF16; }

cudaError_t fwd_tc_config(const Plan& pl, FwdLaunch* L) {
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  // all of the unified L1 / shared storage as shared memory: two CTAs per SM
  e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fwd_tc_kernel, kTHREADS, kSMEM);
  if (e != cudaSuccess) return e;
  // Each CTA allocates half of the SM's 512 tensor-memory columns, and its shared memory
  // (more than a third of the SM's) keeps a third CTA from becoming resident, so no
  // allocation ever waits. The grid is sized for the two CTAs per SM that the shared
  // memory admits (the occupancy query reports one for kernels that allocate tensor
  // memory).
  if (occ < 1 || occ > 2) return cudaErrorInvalidConfiguration;
  int smem_sm = 0, smem_reserved = 0;
  e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, pl.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, pl.device);
  if (e != cudaSuccess) return e;
  occ = smem_sm / (kSMEM + smem_reserved);
  if (occ < 1) return cudaErrorInvalidConfiguration;
  if (occ > 2) occ = 2;
  const int64_t total = (int64_t)pl.B * pl.nW;
  int64_t chunks = ((int64_t)pl.num_sms * occ) / pl.nH;
  if (chunks < 1) chunks = 1;
  if (chunks > total) chunks = total;
  L->chunks = (int)chunks;
  L->grid = (int)(chunks * pl.nH);
  L->threads = kTHREADS;
  L->smem = kSMEM;
  L->ctas_per_sm = occ;
  return cudaSuccess;
}

cudaError_t fwd_tc_launch(const Plan& pl, const FwdLaunch& L0, const void* qkv, void* out, int batch,
                          cudaStream_t st) {
  FwdLaunch L = L0;
  const int64_t total = (int64_t)batch * pl.nW;
  if (batch != pl.B) {
    int64_t chunks = ((int64_t)pl.num_sms * L0.ctas_per_sm) / pl.nH;
    if (chunks < 1) chunks = 1;
    if (chunks > total) chunks = total;
    L.chunks = (int)chunks;
    L.grid = (int)(chunks * pl.nH);
  }
  TcParams p;
  p.qkv = reinterpret_cast<const __nv_bfloat16*>(qkv);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.dense_bias = pl.dense_bias;
  p.err = pl.err;
  p.H = pl.H;
  p.W = pl.W;
  p.C = pl.C;
  p.nH = pl.nH;
  p.s = pl.s;
  p.nWy = pl.nWy;
  p.nWx = pl.nWx;
  p.nW = pl.nW;
  p.total_windows = total;
  p.chunks = L.chunks;
  p.qk_scale_log2 = kLog2e / kInvScale;
  fwd_tc_kernel<<<L.grid, L.threads, L.smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace swin
