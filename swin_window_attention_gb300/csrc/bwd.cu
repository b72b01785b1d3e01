// Fused (shifted-)window attention backward for sm_103a, with the bias-table gradient.
//
// The backward recomputes the forward's logits and probabilities from q and k instead
// of reloading stored ones (Baidu AIAK-Training talk, jxzklqfsx.com article 743345,
// section 2, fused WindowAttention case): a whole window row fits one tile, so nothing
// but q, k, v and the upstream gradient is read. The shift, partition, reverse and
// un-roll are again pure addressing (NVIDIA Swin talk transcript, uticex.com article
// 1598, section 2), so dq, dk and dv land at exactly the channels q, k and v came from.
//
// Per window and head (P row-stochastic, dO upstream gradient of O):
//   dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
//   dtable[idx(i,j), h] += dS_ij   (fp32 dS, never bf16-rounded).
// Warp w owns query rows [16w, 16w+16) for S, P, dP, dS and dQ, then key rows
// [16w, 16w+16) for dK and dV, reading every warp's P and dS from shared memory. P and
// dS enter the dV, dQ and dK products as bf16 hi/lo pairs: a single bf16 operand costs
// up to 2^-9 relative per term, which over a 49-term sum reaches the size of the bf16
// rounding of the result itself and breaks a 1e-2 absolute bound on its own. The
// per-(i,j) dS sums stay in registers across the CTA's windows; at the end one thread
// per table row folds them in a fixed order into a per-CTA partial, and a second
// kernel sums the partials in a fixed order: the result is deterministic.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace swin {

template <int M>
struct BGeo {
  using G = Geo<M>;
  // Tiles hold the N rows of a window plus one zero row (row N): every padded row an MMA
  // operand needs (query or key index >= N) is read from that zero row.
  static constexpr int ROWS = G::N + 1;
  static constexpr int TILE = (ROWS * 64 + 127) / 128 * 128;  // one of q, k, v, dO
  static constexpr int PS_STRIDE = G::NPAD * 2 + 16;  // bytes per row of the P / dS tiles
  static constexpr int PS_BYTES = ROWS * PS_STRIDE;
  static constexpr int STAGE_BYTES = 4 * TILE;
  static constexpr int TCH = G::N * 4;                            // 16-byte chunks per tensor
  static constexpr int TI = (TCH + G::THREADS - 1) / G::THREADS;  // per-thread chunks per tensor
  static constexpr int STG_BYTES = G::WARPS * 16 * 64;  // per-warp bf16 output staging
  static constexpr int R = (2 * M - 1) * (2 * M - 1);
};

struct BwdParams {
  const void* qkv;
  const void* dout;
  void* dqkv;
  const float4* bias_frag;
  const uint32_t* mask_frag;
  float* partial;  // [grid, R]
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;
  int chunks;
  float qk_scale_log2;
  float scale;
};

template <int M, int STAGES>
constexpr int bwd_smem_bytes() {
  return Geo<M>::BIAS_BYTES + Geo<M>::MASK_BYTES + 4 * BGeo<M>::PS_BYTES + BGeo<M>::STG_BYTES +
         STAGES * BGeo<M>::STAGE_BYTES;
}

// Store a warp's 16 rows x 32 channels (fp32 fragments of m16n8 tiles nd = 0..3) scaled
// by `mul` to slice `slice` (0: q, 1: k, 2: v) of the gradient tensor at the tokens of
// window rows 16*warp + r.
template <int M, typename TIO>
__device__ __forceinline__ void store_rows(float (&acc)[4][4], float mul, unsigned char* stg,
                                           TIO* dqkv, int slice, int warp, int lane, int b,
                                           int wy, int wx, int s, int H, int W, int C, int h) {
  constexpr int N = M * M;
  const int g = lane >> 2, t = lane & 3;
  if constexpr (sizeof(TIO) == 2) {
    // two stmatrix: matrix (row half mi & 1, column chunk 2 * call + (mi >> 1))
    const int mi = lane >> 3, rr = (lane & 7) + ((mi & 1) << 3);
    const uint32_t sb = smem_u32(stg);
    const float2 m2 = make_float2(mul, mul);
    uint32_t w[4][2];
#pragma unroll
    for (int nd = 0; nd < 4; ++nd) {
      const float2 a = __fmul2_rn(make_float2(acc[nd][0], acc[nd][1]), m2);
      const float2 c = __fmul2_rn(make_float2(acc[nd][2], acc[nd][3]), m2);
      w[nd][0] = pack_bf16(a.x, a.y);
      w[nd][1] = pack_bf16(c.x, c.y);
    }
    stsm_x4(sb + tile_off(rr, mi >> 1), w[0][0], w[0][1], w[1][0], w[1][1]);
    stsm_x4(sb + tile_off(rr, 2 + (mi >> 1)), w[2][0], w[2][1], w[3][0], w[3][1]);
    __syncwarp();
#pragma unroll
    for (int e = lane; e < 64; e += 32) {
      const int r = e >> 2, c = e & 3, i = warp * 16 + r;
      if (i < N) {
        const int64_t tok = gather_token(b, wy, wx, i, M, s, H, W);
        *reinterpret_cast<uint4*>(dqkv + tok * 3 * C + slice * C + h * kHeadDim + c * 8) =
            *reinterpret_cast<const uint4*>(stg + tile_off(r, c));
      }
    }
    __syncwarp();
  } else {
    const int i0 = warp * 16 + g, i1 = i0 + 8;
    if (i0 < N) {
      float* dst = dqkv + gather_token(b, wy, wx, i0, M, s, H, W) * 3 * C + slice * C + h * kHeadDim + 2 * t;
#pragma unroll
      for (int nd = 0; nd < 4; ++nd)
        *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(acc[nd][0] * mul, acc[nd][1] * mul);
    }
    if (i1 < N) {
      float* dst = dqkv + gather_token(b, wy, wx, i1, M, s, H, W) * 3 * C + slice * C + h * kHeadDim + 2 * t;
#pragma unroll
      for (int nd = 0; nd < 4; ++nd)
        *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(acc[nd][2] * mul, acc[nd][3] * mul);
    }
  }
}

// Resident CTAs per SM the register budget is sized for (shared memory allows three).
template <int M> struct BwdMinBlocks { static constexpr int value = 3; };

template <int M, typename TIO, int STAGES>
__global__ void __launch_bounds__(Geo<M>::THREADS, BwdMinBlocks<M>::value) bwd_kernel(const BwdParams p) {
  using G = Geo<M>;
  using BG = BGeo<M>;
  constexpr int N = G::N, NT = G::NT, KT = G::KT, THREADS = G::THREADS;
  constexpr int PS = BG::PS_STRIDE;
  auto zr = [](int r) { return r < N ? r : N; };  // row, or the zero row for padding
  extern __shared__ __align__(128) unsigned char smem[];
  float4* sbias = reinterpret_cast<float4*>(smem);
  uint32_t* smask = reinterpret_cast<uint32_t*>(smem + G::BIAS_BYTES);
  unsigned char* sP = smem + G::BIAS_BYTES + G::MASK_BYTES;
  // The next kernel may be scheduled now; everything this one reads (activations, and the
  // plan's fragments, which the previous kernel may just have rebuilt) waits for the
  // previous kernel to complete.
  pdl_launch_dependents();
  pdl_wait();
  unsigned char* sPlo = sP + BG::PS_BYTES;
  unsigned char* sdS = sPlo + BG::PS_BYTES;
  unsigned char* sdSlo = sdS + BG::PS_BYTES;
  unsigned char* sstg = sdSlo + BG::PS_BYTES;
  unsigned char* stiles = sstg + BG::STG_BYTES;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int C = p.C, H = p.H, W = p.W, s = p.s;
  unsigned char* stg = sstg + warp * 16 * 64;

  // Per-thread gather slots, the same for all four tensors (q, k, v from qkv; dO from
  // dout): chunk j of this thread is 16-byte chunk c of window slot i = (ly, lx).
  uint32_t ld_soff[BG::TI];  // tile-relative shared offset
  int ld_rc[BG::TI];         // (ly << 8) | lx
  int ld_chan[BG::TI];       // h * 32 + c * 8
#pragma unroll
  for (int j = 0; j < BG::TI; ++j) {
    const int id = tid + j * THREADS;
    const int c = id & 3, i = (id >> 2) < N ? (id >> 2) : 0;
    ld_soff[j] = tile_off(i, c);
    ld_rc[j] = ((i / M) << 8) | (i % M);
    ld_chan[j] = h * kHeadDim + c * 8;
  }
  int lb, lwy, lwx;
  {
    lb = (int)(w_begin / p.nW);
    const int w = (int)(w_begin - (int64_t)lb * p.nW);
    lwy = w / p.nWx;
    lwx = w - lwy * p.nWx;
  }
  int cb = lb, cwy = lwy, cwx = lwx;

  auto issue = [&](int stage) {
    const uint32_t base = smem_u32(stiles + stage * BG::STAGE_BYTES);
    const int y0 = lwy * M + s, x0 = lwx * M + s;
    const int hy = H - y0, hx = W - x0;  // window rows ly >= hy / columns lx >= hx wrap
    const int64_t tok0 = ((int64_t)lb * H + y0) * W + x0;
    const TIO* qbase = reinterpret_cast<const TIO*>(p.qkv) + tok0 * 3 * C;
    const TIO* obase = reinterpret_cast<const TIO*>(p.dout) + tok0 * C;
#pragma unroll
    for (int j = 0; j < BG::TI; ++j) {
      if (j < BG::TI - 1 || tid + j * THREADS < BG::TCH) {
        const int ly = ld_rc[j] >> 8, lx = ld_rc[j] & 255;
        int64_t rel = (int64_t)ly * W + lx;  // token offset from the window's first token
        if (ly >= hy) rel -= (int64_t)H * W;
        if (lx >= hx) rel -= W;
#pragma unroll
        for (int tt = 0; tt < 3; ++tt)
          load_chunk<TIO>(base + tt * BG::TILE + ld_soff[j], qbase + rel * 3 * C + tt * C + ld_chan[j]);
        load_chunk<TIO>(base + 3 * BG::TILE + ld_soff[j], obase + rel * C + ld_chan[j]);
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

  // This head's bias fragments and the class mask fragments (built by the plan in this
  // kernel's fragment order) travel in the first copy group, with window 0.
  {
    const unsigned char* bsrc = reinterpret_cast<const unsigned char*>(p.bias_frag) + (size_t)h * G::BIAS_BYTES;
    for (int e = tid; e < G::BIAS_BYTES / 16; e += THREADS) cp_async_16(smem_u32(smem + e * 16), bsrc + e * 16);
    if (p.mask_frag != nullptr) {
      const unsigned char* msrc = reinterpret_cast<const unsigned char*>(p.mask_frag);
      for (int e = tid; e < G::MASK_BYTES / 16; e += THREADS)
        cp_async_16(smem_u32(smem + G::BIAS_BYTES + e * 16), msrc + e * 16);
    }
  }
#pragma unroll
  for (int st = 0; st < STAGES - 1; ++st) {
    if (st < nwin) issue(st);
    cp_async_commit();
  }

  // The zero row (row N) of every q/k/v/dO tile; loads never touch it.
  for (int e = tid; e < STAGES * 4 * 4; e += THREADS) {
    const int c = e & 3, tile = e >> 2;
    *reinterpret_cast<uint4*>(stiles + tile * BG::TILE + tile_off(N, c)) = make_uint4(0u, 0u, 0u, 0u);
  }
  // P and dS tiles (hi and lo) start zeroed: columns NT*8..NPAD-1 are never written.
  for (int e = tid; e < 4 * BG::PS_BYTES / 16; e += THREADS)
    reinterpret_cast<uint4*>(sP)[e] = make_uint4(0u, 0u, 0u, 0u);
  const float4* bfrag = sbias + warp * NT * 32 + lane;
  const int r0 = warp * 16 + g, r1 = r0 + 8;
  // U operand of the shift-mask MMA for rows r0, r1 (k-slots 8..15 are zero).
  const uint32_t mu0 = mask_u_frag(r0, t, M, s), mu1 = mask_u_frag(r1, t, M, s);
  float dtacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) dtacc[nt][0] = dtacc[nt][1] = dtacc[nt][2] = dtacc[nt][3] = 0.0f;

  for (int it = 0; it < nwin; ++it) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nx = it + STAGES - 1;
      if (nx < nwin) issue(nx % STAGES);
      cp_async_commit();
    }
    const int b = cb, wy = cwy, wx = cwx;
    if (++cwx == p.nWx) {
      cwx = 0;
      if (++cwy == p.nWy) {
        cwy = 0;
        ++cb;
      }
    }
    const uint32_t qb = smem_u32(stiles + (it % STAGES) * BG::STAGE_BYTES);
    const uint32_t kb = qb + BG::TILE, vb = kb + BG::TILE, ob = vb + BG::TILE;

    // ---- recompute S and P ---------------------------------------------------------
    float pr[NT][4];
    {
      uint32_t qa[2][4];
      const int mi = lane >> 3, row = zr(warp * 16 + (lane & 7) + ((mi & 1) << 3));
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        ldsm_x4(qb + tile_off(row, 2 * kk + (mi >> 1)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 bb = bfrag[nt * 32];  // z = q.k + bias/scale starts from the bias
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + tile_off(zr(nt * 8 + (lane & 7)), lane >> 3), b0, b1, b2, b3);
        mma_bf16_c(pr[nt], qa[0][0], qa[0][1], qa[0][2], qa[0][3], b0, b1, bb.x, bb.y, bb.z, bb.w);
        mma_bf16(pr[nt], qa[1][0], qa[1][1], qa[1][2], qa[1][3], b2, b3);
      }
    }
    // shift mask (boundary windows only): z += U V^T, one k16 MMA per key tile
    if (p.mask_frag != nullptr && (wy == p.nWy - 1 || wx == p.nWx - 1)) {
      const int cls = (wy == p.nWy - 1 ? 2 : 0) | (wx == p.nWx - 1 ? 1 : 0);
      const uint4* mv = reinterpret_cast<const uint4*>(smask) + (cls - 1) * (G::NTP / 4) * 32 + lane;
#pragma unroll
      for (int q4 = 0; q4 < G::NTP / 4; ++q4) {
        const uint4 v = mv[q4 * 32];
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q4 * 4 + u < NT) mma_bf16(pr[q4 * 4 + u], mu0, mu1, 0u, 0u, vw[u], 0u);
      }
    }
    float m0a = -INFINITY, m0b = -INFINITY, m1a = -INFINITY, m1b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      m0a = fmax3(m0a, pr[nt][0], pr[nt][1]);
      m1a = fmax3(m1a, pr[nt][2], pr[nt][3]);
      if (nt + 1 < NT) {
        m0b = fmax3(m0b, pr[nt + 1][0], pr[nt + 1][1]);
        m1b = fmax3(m1b, pr[nt + 1][2], pr[nt + 1][3]);
      }
    }
    float mx0 = fmaxf(m0a, m0b), mx1 = fmaxf(m1a, m1b);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float2 c2 = make_float2(p.qk_scale_log2, p.qk_scale_log2);
    const float2 nm0 = make_float2(-mx0 * p.qk_scale_log2, -mx0 * p.qk_scale_log2);
    const float2 nm1 = make_float2(-mx1 * p.qk_scale_log2, -mx1 * p.qk_scale_log2);
    float2 l0v = make_float2(0.0f, 0.0f), l1v = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 e0 = __ffma2_rn(make_float2(pr[nt][0], pr[nt][1]), c2, nm0);
      const float2 e1 = __ffma2_rn(make_float2(pr[nt][2], pr[nt][3]), c2, nm1);
      pr[nt][0] = fast_exp2(e0.x);
      pr[nt][1] = fast_exp2(e0.y);
      pr[nt][2] = fast_exp2(e1.x);
      pr[nt][3] = fast_exp2(e1.y);
      l0v = __fadd2_rn(l0v, make_float2(pr[nt][0], pr[nt][1]));
      l1v = __fadd2_rn(l1v, make_float2(pr[nt][2], pr[nt][3]));
    }
    float l0 = l0v.x + l0v.y, l1 = l1v.x + l1v.y;
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // Normalised probabilities; padded query rows are zeroed so they add nothing below.
    const float inv0 = r0 < N ? 1.0f / l0 : 0.0f, inv1 = r1 < N ? 1.0f / l1 : 0.0f;
    {
      const float2 i0 = make_float2(inv0, inv0), i1 = make_float2(inv1, inv1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 a = __fmul2_rn(make_float2(pr[nt][0], pr[nt][1]), i0);
        const float2 c = __fmul2_rn(make_float2(pr[nt][2], pr[nt][3]), i1);
        pr[nt][0] = a.x;
        pr[nt][1] = a.y;
        pr[nt][2] = c.x;
        pr[nt][3] = c.y;
      }
    }

    // ---- dP = dO V^T ---------------------------------------------------------------
    float ds[NT][4];
    {
      uint32_t da[2][4];
      const int mi = lane >> 3, row = zr(warp * 16 + (lane & 7) + ((mi & 1) << 3));
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        ldsm_x4(ob + tile_off(row, 2 * kk + (mi >> 1)), da[kk][0], da[kk][1], da[kk][2], da[kk][3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        ds[nt][0] = ds[nt][1] = ds[nt][2] = ds[nt][3] = 0.0f;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(vb + tile_off(zr(nt * 8 + (lane & 7)), lane >> 3), b0, b1, b2, b3);
        mma_bf16(ds[nt], da[0][0], da[0][1], da[0][2], da[0][3], b0, b1);
        mma_bf16(ds[nt], da[1][0], da[1][1], da[1][2], da[1][3], b2, b3);
      }
    }
    // ---- D = rowsum(P o dP), dS = P o (dP - D) ---------------------------------------
    float2 D0v = make_float2(0.0f, 0.0f), D1v = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      D0v = __ffma2_rn(make_float2(pr[nt][0], pr[nt][1]), make_float2(ds[nt][0], ds[nt][1]), D0v);
      D1v = __ffma2_rn(make_float2(pr[nt][2], pr[nt][3]), make_float2(ds[nt][2], ds[nt][3]), D1v);
    }
    float D0 = D0v.x + D0v.y, D1 = D1v.x + D1v.y;
    D0 += __shfl_xor_sync(0xffffffffu, D0, 1);
    D0 += __shfl_xor_sync(0xffffffffu, D0, 2);
    D1 += __shfl_xor_sync(0xffffffffu, D1, 1);
    D1 += __shfl_xor_sync(0xffffffffu, D1, 2);
    // P and dS go to shared memory (and dS also stays in registers for dQ) as bf16
    // hi/lo pairs: the lo term is the rounding residual of the hi term, so the MMAs that
    // read them keep ~16 bits of each.
    uint32_t dsh[NT][2], dsl[NT][2];
    {
      uint32_t ph[NT][2], pl[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // dS = P o (dP - D): one packed subtract and one packed multiply per pair
        const float2 s0 = __fmul2_rn(make_float2(pr[nt][0], pr[nt][1]),
                                     __fadd2_rn(make_float2(ds[nt][0], ds[nt][1]), make_float2(-D0, -D0)));
        const float2 s1 = __fmul2_rn(make_float2(pr[nt][2], pr[nt][3]),
                                     __fadd2_rn(make_float2(ds[nt][2], ds[nt][3]), make_float2(-D1, -D1)));
        ds[nt][0] = s0.x;
        ds[nt][1] = s0.y;
        ds[nt][2] = s1.x;
        ds[nt][3] = s1.y;
        const float2 t0 = __fadd2_rn(make_float2(dtacc[nt][0], dtacc[nt][1]), s0);
        const float2 t1 = __fadd2_rn(make_float2(dtacc[nt][2], dtacc[nt][3]), s1);
        dtacc[nt][0] = t0.x;
        dtacc[nt][1] = t0.y;
        dtacc[nt][2] = t1.x;
        dtacc[nt][3] = t1.y;
        split_bf16(pr[nt][0], pr[nt][1], ph[nt][0], pl[nt][0]);
        split_bf16(pr[nt][2], pr[nt][3], ph[nt][1], pl[nt][1]);
        split_bf16(ds[nt][0], ds[nt][1], dsh[nt][0], dsl[nt][0]);
        split_bf16(ds[nt][2], ds[nt][3], dsh[nt][1], dsl[nt][1]);
      }
      // stmatrix: matrix (n-tile nt + (mi >> 1), row half mi & 1) per 8-lane group
      const int mi = lane >> 3;
      // padded rows (all zero) land on the zero row
      const uint32_t rowoff = (uint32_t)(zr(warp * 16 + 8 * (mi & 1) + (lane & 7)) * PS + (mi >> 1) * 16);
      const uint32_t aP = smem_u32(sP) + rowoff, aPl = smem_u32(sPlo) + rowoff;
      const uint32_t aS = smem_u32(sdS) + rowoff, aSl = smem_u32(sdSlo) + rowoff;
#pragma unroll
      for (int nt = 0; nt + 1 < NT; nt += 2) {
        stsm_x4(aP + nt * 16, ph[nt][0], ph[nt][1], ph[nt + 1][0], ph[nt + 1][1]);
        stsm_x4(aPl + nt * 16, pl[nt][0], pl[nt][1], pl[nt + 1][0], pl[nt + 1][1]);
        stsm_x4(aS + nt * 16, dsh[nt][0], dsh[nt][1], dsh[nt + 1][0], dsh[nt + 1][1]);
        stsm_x4(aSl + nt * 16, dsl[nt][0], dsl[nt][1], dsl[nt + 1][0], dsl[nt + 1][1]);
      }
      if constexpr (NT % 2 == 1) {
        constexpr int nt = NT - 1;
        stsm_x2(aP + nt * 16, ph[nt][0], ph[nt][1]);
        stsm_x2(aPl + nt * 16, pl[nt][0], pl[nt][1]);
        stsm_x2(aS + nt * 16, dsh[nt][0], dsh[nt][1]);
        stsm_x2(aSl + nt * 16, dsl[nt][0], dsl[nt][1]);
      }
    }

    // ---- dQ = scale dS K --------------------------------------------------------------
    {
      float dq[4][4];
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) dq[nd][0] = dq[nd][1] = dq[nd][2] = dq[nd][3] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const uint32_t a0 = dsh[2 * kk][0], a1 = dsh[2 * kk][1], l0 = dsl[2 * kk][0], l1 = dsl[2 * kk][1];
        uint32_t a2 = 0u, a3 = 0u, l2 = 0u, l3 = 0u;
        if (2 * kk + 1 < NT) {
          a2 = dsh[2 * kk + 1][0];
          a3 = dsh[2 * kk + 1][1];
          l2 = dsl[2 * kk + 1][0];
          l3 = dsl[2 * kk + 1][1];
        }
        const int mi = lane >> 3, row = zr(kk * 16 + (lane & 7) + ((mi & 1) << 3));
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(kb + tile_off(row, 2 * pp + (mi >> 1)), v0, v1, v2, v3);
          mma_bf16(dq[2 * pp], a0, a1, a2, a3, v0, v1);
          mma_bf16(dq[2 * pp + 1], a0, a1, a2, a3, v2, v3);
          mma_bf16(dq[2 * pp], l0, l1, l2, l3, v0, v1);
          mma_bf16(dq[2 * pp + 1], l0, l1, l2, l3, v2, v3);
        }
      }
      store_rows<M, TIO>(dq, p.scale, stg, reinterpret_cast<TIO*>(p.dqkv), 0, warp, lane, b, wy, wx,
                         s, H, W, C, h);
    }
    __syncthreads();  // every warp's P and dS rows are in shared memory

    // ---- dK = scale dS^T Q and dV = P^T dO for key rows [16w, 16w+16) -----------------
    {
      float dk[4][4], dv[4][4];
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        dk[nd][0] = dk[nd][1] = dk[nd][2] = dk[nd][3] = 0.0f;
        dv[nd][0] = dv[nd][1] = dv[nd][2] = dv[nd][3] = 0.0f;
      }
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
        const int rowA = zr(kk * 16 + (lane & 7) + 8 * (mi >> 1)), chA = 2 * warp + (mi & 1);
        uint32_t a0, a1, a2, a3, f0, f1, f2, f3, p0, p1, p2, p3, e0, e1, e2, e3;
        ldsm_x4_t(smem_u32(sdS + rowA * PS + chA * 16), a0, a1, a2, a3);
        ldsm_x4_t(smem_u32(sdSlo + rowA * PS + chA * 16), f0, f1, f2, f3);
        ldsm_x4_t(smem_u32(sP + rowA * PS + chA * 16), p0, p1, p2, p3);
        ldsm_x4_t(smem_u32(sPlo + rowA * PS + chA * 16), e0, e1, e2, e3);
        const int rowB = zr(kk * 16 + (lane & 7) + ((mi & 1) << 3));
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          uint32_t q0, q1, q2, q3, d0, d1, d2, d3;
          ldsm_x4_t(qb + tile_off(rowB, 2 * pp + (mi >> 1)), q0, q1, q2, q3);
          mma_bf16(dk[2 * pp], a0, a1, a2, a3, q0, q1);
          mma_bf16(dk[2 * pp + 1], a0, a1, a2, a3, q2, q3);
          mma_bf16(dk[2 * pp], f0, f1, f2, f3, q0, q1);
          mma_bf16(dk[2 * pp + 1], f0, f1, f2, f3, q2, q3);
          ldsm_x4_t(ob + tile_off(rowB, 2 * pp + (mi >> 1)), d0, d1, d2, d3);
          mma_bf16(dv[2 * pp], p0, p1, p2, p3, d0, d1);
          mma_bf16(dv[2 * pp + 1], p0, p1, p2, p3, d2, d3);
          mma_bf16(dv[2 * pp], e0, e1, e2, e3, d0, d1);
          mma_bf16(dv[2 * pp + 1], e0, e1, e2, e3, d2, d3);
        }
      }
      store_rows<M, TIO>(dk, p.scale, stg, reinterpret_cast<TIO*>(p.dqkv), 1, warp, lane, b, wy, wx,
                         s, H, W, C, h);
      store_rows<M, TIO>(dv, 1.0f, stg, reinterpret_cast<TIO*>(p.dqkv), 2, warp, lane, b, wy, wx,
                         s, H, W, C, h);
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- fold the per-(i,j) dS sums into this CTA's table-gradient partial -------------
  float* sdt = reinterpret_cast<float*>(stiles);  // N*N floats fit the tile buffers
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + 8 * (q >> 1), c = nt * 8 + 2 * t + (q & 1);
      if (r < N && c < N) sdt[r * N + c] = dtacc[nt][q];
    }
  __syncthreads();
  for (int rr = tid; rr < BG::R; rr += THREADS) {
    const int dy = rr / (2 * M - 1) - (M - 1), dx = rr % (2 * M - 1) - (M - 1);
    float acc = 0.0f;
    for (int yi = 0; yi < M; ++yi) {
      const int yj = yi - dy;
      if (yj < 0 || yj >= M) continue;
      for (int xi = 0; xi < M; ++xi) {
        const int xj = xi - dx;
        if (xj < 0 || xj >= M) continue;
        acc += sdt[(yi * M + xi) * N + (yj * M + xj)];
      }
    }
    p.partial[(int64_t)blockIdx.x * BG::R + rr] = acc;
  }
}

// dtable[r, h] = sum over chunks c (in order) of partial[c*nH + h, r].
__global__ void dtable_reduce_kernel(const float* __restrict__ partial, int R, int nH, int chunks,
                                     float* __restrict__ dtable) {
  pdl_wait();  // launched early; the partials are complete once the backward grid is
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= R * nH) return;
  const int r = e / nH, h = e % nH;
  float acc = 0.0f;
  for (int c = 0; c < chunks; ++c) acc += partial[(int64_t)(c * nH + h) * R + r];
  dtable[e] = acc;
}

// ---- host side ---------------------------------------------------------------------

cudaError_t launch_dtable_reduce(const float* partial, int R, int nH, int chunks, float* dtable, cudaStream_t st) {
  return launch_pdl(dtable_reduce_kernel, dim3((R * nH + 255) / 256), dim3(256), 0, st, partial, R, nH, chunks,
                    dtable);
}

bool bwd_tc_applies(const Plan& pl);
cudaError_t bwd_tc_config(const Plan& pl, BwdLaunch* L);
cudaError_t bwd_tc_launch(const Plan& pl, const BwdLaunch& L, const void* qkv, const void* dout, void* dqkv,
                          float* dtable, cudaStream_t st);

template <int M> struct BwdStages { static constexpr int value = 2; };

template <int M, typename TIO, int STAGES>
static cudaError_t bconfig_t(const Plan& pl, BwdLaunch* L) {
  using G = Geo<M>;
  constexpr int smem = bwd_smem_bytes<M, STAGES>();
  static_assert(G::N * G::N * 4 <= STAGES * BGeo<M>::STAGE_BYTES, "dS sums must fit the tiles");
  auto kern = bwd_kernel<M, TIO, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, G::THREADS, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t total = (int64_t)pl.B * pl.nW;
  int64_t chunks = ((int64_t)pl.num_sms * occ) / pl.nH;
  if (chunks < 1) chunks = 1;
  if (total > 0 && chunks > total) chunks = total;
  L->chunks = (int)chunks;
  L->grid = (int)(chunks * pl.nH);
  L->threads = G::THREADS;
  L->smem = smem;
  L->partial_rows = L->grid;
  return cudaSuccess;
}

template <int M, typename TIO, int STAGES>
static cudaError_t blaunch_t(const Plan& pl, const BwdLaunch& L, const void* qkv, const void* dout,
                             void* dqkv, float* dtable, cudaStream_t st) {
  BwdParams p;
  p.qkv = qkv;
  p.dout = dout;
  p.dqkv = dqkv;
  p.bias_frag = pl.bias_frag;
  p.mask_frag = pl.s > 0 ? pl.mask_frag : nullptr;
  p.partial = pl.dt_partial;
  p.H = pl.H;
  p.W = pl.W;
  p.C = pl.C;
  p.nH = pl.nH;
  p.s = pl.s;
  p.nWy = pl.nWy;
  p.nWx = pl.nWx;
  p.nW = pl.nW;
  p.total_windows = (int64_t)pl.B * pl.nW;
  p.chunks = L.chunks;
  p.scale = 1.0f / kInvScale;
  p.qk_scale_log2 = kLog2e / kInvScale;
  cudaError_t e = launch_pdl(bwd_kernel<M, TIO, STAGES>, dim3(L.grid), dim3(L.threads), L.smem, st, p);
  if (e != cudaSuccess) return e;
  const int R = BGeo<M>::R;
  return launch_dtable_reduce(pl.dt_partial, R, pl.nH, L.chunks, dtable, st);
}

// Kernel choice: the tcgen05 kernel when the plan asks for it (7x7 windows, bf16), or
// by default where it applies and was measured faster (all but shifted layers at most two
// windows wide, where its right-edge gathers dominate); else the mma.sync kernel.
cudaError_t bwd_config(const Plan& pl, BwdLaunch* L) {
  *L = BwdLaunch();
  if (pl.bwd_kernel == SWIN_WATTN_KERNEL_TCGEN05) return bwd_tc_applies(pl) ? bwd_tc_config(pl, L) : cudaErrorNotSupported;
  if (pl.bwd_kernel == SWIN_WATTN_KERNEL_AUTO && bwd_tc_applies(pl) && !(pl.s > 0 && pl.nWx <= 2))
    return bwd_tc_config(pl, L);
  const bool f32 = pl.dtype == SWIN_WATTN_FP32;
  switch (pl.M) {
    case 4:
      return f32 ? bconfig_t<4, float, BwdStages<4>::value>(pl, L)
                 : bconfig_t<4, __nv_bfloat16, BwdStages<4>::value>(pl, L);
    case 7:
      return f32 ? bconfig_t<7, float, BwdStages<7>::value>(pl, L)
                 : bconfig_t<7, __nv_bfloat16, BwdStages<7>::value>(pl, L);
    default:  // no backward for this window size: the plan still serves the forward
      *L = BwdLaunch();
      return cudaSuccess;
  }
}

cudaError_t bwd_launch(const Plan& pl, const BwdLaunch& L, const void* qkv, const void* dout,
                       void* dqkv, float* dtable, cudaStream_t st) {
  if (L.tc) return bwd_tc_launch(pl, L, qkv, dout, dqkv, dtable, st);
  const bool f32 = pl.dtype == SWIN_WATTN_FP32;
  switch (pl.M) {
    case 4:
      return f32 ? blaunch_t<4, float, BwdStages<4>::value>(pl, L, qkv, dout, dqkv, dtable, st)
                 : blaunch_t<4, __nv_bfloat16, BwdStages<4>::value>(pl, L, qkv, dout, dqkv, dtable, st);
    case 7:
      return f32 ? blaunch_t<7, float, BwdStages<7>::value>(pl, L, qkv, dout, dqkv, dtable, st)
                 : blaunch_t<7, __nv_bfloat16, BwdStages<7>::value>(pl, L, qkv, dout, dqkv, dtable, st);
    default:
      return cudaErrorNotSupported;
  }
}

// ---- backward without device allocation --------------------------------------------
//
// Some callers cannot allocate device memory at the point where they run the backward:
// runtimes that fix their device memory plan at start-up and forbid any later
// cudaMalloc (real-time or certified inference/training stacks), and frameworks whose own
// allocator must account for every device byte. A plan allocates (its dense bias, mask
// and reduction buffers), so such a caller cannot create one. swin_wattn_bwd_noalloc
// runs the same backward with all of its working memory in one fixed array below.

// Working memory of swin_wattn_bwd_noalloc: bias fragments, class mask fragments and the
// per-CTA table-gradient partials, packed at 256-byte boundaries.
constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t launch_bias_frags(int M, const float* table, int nH, int H, int W, int s, float4* bias_frag,
                              uint32_t* mask_frag, float* dense, cudaStream_t st);
void count_launches(int n);

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_ptr[kMaxDevices] = {};

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t noalloc_scratch(int device, unsigned char** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[device] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[device] = static_cast<unsigned char*>(ptr);
  }
  *out = g_noalloc_ptr[device];
  return cudaSuccess;
}

template <int M, typename TIO>
cudaError_t noalloc_bwd_t(Plan& pl, const float* table, const void* qkv, const void* dout,
                          void* dqkv, float* dtable, cudaStream_t st, size_t* need) {
  constexpr int STAGES = BwdStages<M>::value;
  BwdLaunch L;
  cudaError_t e = bconfig_t<M, TIO, STAGES>(pl, &L);
  if (e != cudaSuccess) return e;
  const size_t bias_bytes = round256((size_t)pl.nH * Geo<M>::BIAS_BYTES);
  const size_t mask_bytes = round256(Geo<M>::MASK_BYTES);
  const size_t part_bytes = round256((size_t)L.partial_rows * BGeo<M>::R * sizeof(float));
  *need = bias_bytes + mask_bytes + part_bytes;
  if (*need > kNoAllocScratchBytes) return cudaErrorMemoryAllocation;
  unsigned char* base = nullptr;
  e = noalloc_scratch(pl.device, &base);
  if (e != cudaSuccess) return e;
  pl.bias_frag = reinterpret_cast<float4*>(base);
  pl.mask_frag = pl.s > 0 ? reinterpret_cast<uint32_t*>(base + bias_bytes) : nullptr;
  pl.dt_partial = reinterpret_cast<float*>(base + bias_bytes + mask_bytes);
  // the plan's own fragment kernel, without the dense bias (the kernels never read it)
  e = launch_bias_frags(M, table, pl.nH, pl.H, pl.W, pl.s, pl.bias_frag, pl.mask_frag, nullptr, st);
  if (e != cudaSuccess) return e;
  e = blaunch_t<M, TIO, STAGES>(pl, L, qkv, dout, dqkv, dtable, st);
  if (e == cudaSuccess) count_launches(3);  // fragments, backward, table-gradient reduction
  return e;
}

}  // namespace

}  // namespace swin

namespace swin {
void set_last_error(const char* msg);
int check_device_ptr_abi(const void* ptr, size_t align);
}

extern "C" int swin_wattn_bwd_noalloc(const void* qkv, const void* dout, void* dqkv, float* dtable,
                                      const float* bias_table, int B, int H, int W, int C,
                                      int num_heads, int window, int shift, int dtype,
                                      struct CUstream_st* stream) {
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || num_heads <= 0) return SWIN_WATTN_ERR_INVALID_ARG;
  if (dtype != SWIN_WATTN_BF16 && dtype != SWIN_WATTN_FP32) return SWIN_WATTN_ERR_INVALID_ARG;
  if (window != 4 && window != 7) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (shift < 0 || shift >= window) return SWIN_WATTN_ERR_INVALID_ARG;
  if (H % window != 0 || W % window != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (C % num_heads != 0 || C / num_heads != swin::kHeadDim) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * H * W * 3 * C >= ((int64_t)1 << 40)) return SWIN_WATTN_ERR_UNSUPPORTED;
  int rc = swin::check_device_ptr_abi(dtable, 4);
  if (rc == SWIN_WATTN_OK) rc = swin::check_device_ptr_abi(bias_table, 4);
  if (rc != SWIN_WATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) {
    const size_t tbytes = sizeof(float) * (size_t)(2 * window - 1) * (2 * window - 1) * num_heads;
    const cudaError_t e = cudaMemsetAsync(dtable, 0, tbytes, st);
    if (e != cudaSuccess) {
      swin::set_last_error(cudaGetErrorString(e));
      return SWIN_WATTN_ERR_CUDA;
    }
    return SWIN_WATTN_OK;
  }
  if ((rc = swin::check_device_ptr_abi(qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = swin::check_device_ptr_abi(dout, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = swin::check_device_ptr_abi(dqkv, 16)) != SWIN_WATTN_OK) return rc;

  swin::Plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.B = B;
  pl.H = H;
  pl.W = W;
  pl.C = C;
  pl.nH = num_heads;
  pl.M = window;
  pl.s = shift;
  pl.dtype = dtype;
  pl.N = window * window;
  pl.nWy = H / window;
  pl.nWx = W / window;
  pl.nW = pl.nWy * pl.nWx;
  cudaError_t e = cudaGetDevice(&pl.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&pl.num_sms, cudaDevAttrMultiProcessorCount, pl.device);
  size_t need = 0;
  if (e == cudaSuccess) {
    const bool f32 = dtype == SWIN_WATTN_FP32;
    if (window == 4)
      e = f32 ? swin::noalloc_bwd_t<4, float>(pl, bias_table, qkv, dout, dqkv, dtable, st, &need)
              : swin::noalloc_bwd_t<4, __nv_bfloat16>(pl, bias_table, qkv, dout, dqkv, dtable, st, &need);
    else
      e = f32 ? swin::noalloc_bwd_t<7, float>(pl, bias_table, qkv, dout, dqkv, dtable, st, &need)
              : swin::noalloc_bwd_t<7, __nv_bfloat16>(pl, bias_table, qkv, dout, dqkv, dtable, st, &need);
  }
  if (e == cudaErrorMemoryAllocation) {
    char msg[160];
    std::snprintf(msg, sizeof(msg),
                  "swin_wattn_bwd_noalloc: this shape needs %zu bytes of working memory, above "
                  "the fixed %zu bytes",
                  need, swin::kNoAllocScratchBytes);
    swin::set_last_error(msg);
    return SWIN_WATTN_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) {
    swin::set_last_error(cudaGetErrorString(e));
    return SWIN_WATTN_ERR_CUDA;
  }
  return SWIN_WATTN_OK;
}
