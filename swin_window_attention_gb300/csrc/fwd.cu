// Fused (shifted-)window attention forward for sm_103a.
//
// One kernel replaces the roll, window partition, batch GEMM, bias add, mask add,
// softmax, batch GEMM, window reverse and un-roll chain (NVIDIA Swin talk transcript,
// uticex.com article 1598, section 2 "training optimisation" for the window ops and
// the fused attention, section 3 for the transposes folded into the fused kernel's
// loads and stores; Baidu AIAK-Training talk, jxzklqfsx.com article 743345, section 2,
// for the single fused WindowAttention kernel staging HBM -> shared -> registers).
//
// Work decomposition. A CTA owns one head h and a contiguous range of windows (across
// the batch). Its dense bias (divided by the softmax scale, in mma-fragment order) and
// the shift-mask V fragments of the three boundary window classes (last column, last
// row, corner: with the interior, the only patterns the region labels can form; the
// mask enters as one extra k16 MMA per key tile) are staged in shared memory once. Each window's q/k/v head slices (64 bytes per token each) are gathered with
// 16-byte cp.async straight from the rolled positions into a swizzled shared tile,
// STAGES deep, so several windows are in flight per CTA. Warp w owns query rows
// [16w, 16w+16): S = Q K^T on bf16 tensor cores (m16n8k16, fp32 accumulate), fused
// scale + bias + mask, a register softmax with quad shuffles, P (bf16) V, and the
// normalised rows go back to the token positions they were read from.
#include <cstring>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

struct FwdParams {
  const void* qkv;
  void* out;
  const float4* bias_frag;    // plan fragments [nH][WARPS][NT][32]
  const uint32_t* mask_frag;  // plan boundary-class mask V fragments, or null
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;  // B * nW
  int chunks;             // window ranges per head
  float qk_scale_log2;    // hd^-0.5 * log2(e)
  int* err;               // plan error word (bit 0: a bounded wait ran out)
  uint64_t wait_ns;       // bound of each wait on a stage barrier
  int fault;              // armed fault site (fault-injection build only)
};

// With TMA loads the tiles sit on 1024-byte boundaries (the copy engine's 64-byte swizzle
// is a function of the address; the tile layout is that swizzle), followed by one
// mbarrier per stage.
template <int M, typename TIO, int STAGES, bool TMA>
constexpr int fwd_smem_bytes() {
  return Geo<M>::BIAS_BYTES + Geo<M>::MASK_BYTES + STAGES * Geo<M>::STAGE_BYTES + (TMA ? 1024 + 8 * STAGES : 0);
}

// Resident CTAs per SM the register budget is sized for.
template <int M> struct FwdMinBlocks { static constexpr int value = 4; };
template <> struct FwdMinBlocks<12> { static constexpr int value = 1; };

// Tiles come either from 16-byte cp.async gathers by every thread, or (TMA, 7x7 windows,
// bf16) from the copy engine: one 7 x 7-token box per tensor for a window that does not
// wrap around the image border, two row bands for one that wraps at the bottom only, and
// the cp.async gather for the last window column of a shifted layer; a stage's mbarrier
// then counts every thread's cp.async arrival plus the copy engine's bytes.
template <int M, typename TIO, int STAGES, bool TMA>
__global__ void __launch_bounds__(Geo<M>::THREADS, FwdMinBlocks<M>::value)
    fwd_kernel(const __grid_constant__ CUtensorMap box_map, const __grid_constant__ CUtensorMap top_map,
               const __grid_constant__ CUtensorMap bot_map, const FwdParams p) {
  using G = Geo<M>;
  constexpr int N = G::N, NT = G::NT, KT = G::KT, THREADS = G::THREADS;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = TMA ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
  // The next kernel may be scheduled now; everything this one reads (activations, and the
  // plan's fragments, which the previous kernel may just have rebuilt) waits for the
  // previous kernel to complete.
  pdl_launch_dependents();
  const uint32_t bar0 = smem_u32(smem) + G::BIAS_BYTES + G::MASK_BYTES + STAGES * G::STAGE_BYTES;
  float4* sbias = reinterpret_cast<float4*>(smem);
  uint32_t* smask = reinterpret_cast<uint32_t*>(smem + G::BIAS_BYTES);
  unsigned char* stiles = smem + G::BIAS_BYTES + G::MASK_BYTES;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int C3 = 3 * p.C, H = p.H, W = p.W, s = p.s;
  const TIO* __restrict__ qkv = reinterpret_cast<const TIO*>(p.qkv);

  // Per-thread gather slots, the same for q, k and v: chunk j of this thread is 16-byte
  // chunk c of window slot i = (ly, lx) of each of the three tensors.
  constexpr int TCH = N * 4, TI = (TCH + THREADS - 1) / THREADS;
  uint32_t ld_soff[TI];  // tile-relative shared offset
  int ld_rc[TI];         // (ly << 8) | lx
  int ld_chan[TI];       // h * 32 + c * 8
#pragma unroll
  for (int j = 0; j < TI; ++j) {
    const int id = tid + j * THREADS;
    const int c = id & 3, i = (id >> 2) < N ? (id >> 2) : 0;
    ld_soff[j] = tile_off(i, c);
    ld_rc[j] = ((i / M) << 8) | (i % M);
    ld_chan[j] = h * kHeadDim + c * 8;
  }
  // Window cursor of the next window to load: (b, wy, wx) advanced one window at a time.
  int lb, lwy, lwx;
  {
    const int64_t w0 = w_begin;
    lb = (int)(w0 / p.nW);
    const int w = (int)(w0 - (int64_t)lb * p.nW);
    lwy = w / p.nWx;
    lwx = w - lwy * p.nWx;
  }
  int cb = lb, cwy = lwy, cwx = lwx;  // cursor of the window being computed
  const uint32_t tiles_u32 = smem_u32(stiles);
#ifdef SWIN_WATTN_FAULT_INJECTION
  bool first_gather = true;  // the CTA's first cp.async-gathered window is being issued
#endif

  auto issue = [&](uint32_t stage_off, int stage) {
    const uint32_t base = tiles_u32 + stage_off;
    const int y0 = lwy * M + s, x0 = lwx * M + s;
    const int hy = H - y0, hx = W - x0;  // window rows ly >= hy / columns lx >= hx wrap
    if constexpr (TMA) {
      const uint32_t full = bar0 + 8 * stage;
      // 0: one box per tensor; 1: two row bands (wraps at the bottom only, and the second
      // band starts on a 128-byte boundary); 2: cp.async gather (wraps at the right)
      const int kind = hx >= M ? (hy >= M ? 0 : (((M - s) & 1) == 0 ? 1 : 2)) : 2;
      if (kind < 2) {
        if (tid == 0) {
          tc::fence_proxy_async();  // the stage's previous reads before the copy engine's writes
          tc::mbar_expect_tx(full, 3 * N * 64);
          const int cq = h * kHeadDim, ck = p.C + cq, cv = 2 * p.C + cq;
          if (kind == 0) {
            tc::box_load(base, &box_map, cq, x0, y0, lb, full);
            tc::box_load(base + G::TILE_BYTES, &box_map, ck, x0, y0, lb, full);
            tc::box_load(base + 2 * G::TILE_BYTES, &box_map, cv, x0, y0, lb, full);
          } else {
            const uint32_t bot = base + (M - s) * M * 64;
            tc::box_load(base, &top_map, cq, x0, y0, lb, full);
            tc::box_load(base + G::TILE_BYTES, &top_map, ck, x0, y0, lb, full);
            tc::box_load(base + 2 * G::TILE_BYTES, &top_map, cv, x0, y0, lb, full);
            tc::box_load(bot, &bot_map, cq, x0, 0, lb, full);
            tc::box_load(bot + G::TILE_BYTES, &bot_map, ck, x0, 0, lb, full);
            tc::box_load(bot + 2 * G::TILE_BYTES, &bot_map, cv, x0, 0, lb, full);
          }
        }
        tc::cp_async_arrive(full);
        if (++lwx == p.nWx) {
          lwx = 0;
          if (++lwy == p.nWy) {
            lwy = 0;
            ++lb;
          }
        }
        return;
      }
      if (tid == 0) tc::mbar_expect_tx(full, 0);
    }
    const TIO* wbase = qkv + (((int64_t)lb * H + y0) * W + x0) * C3;
#pragma unroll
    for (int j = 0; j < TI; ++j) {
      if (j < TI - 1 || tid + j * THREADS < TCH) {
        const int ly = ld_rc[j] >> 8, lx = ld_rc[j] & 255;
        int64_t rel = (int64_t)ly * W + lx;  // token offset from the window's first token
        if (ly >= hy) rel -= (int64_t)H * W;
        if (lx >= hx) rel -= W;
        const TIO* src = wbase + rel * C3 + ld_chan[j];
#pragma unroll
        for (int tt = 0; tt < 3; ++tt)
          load_chunk<TIO>(base + tt * G::TILE_BYTES + ld_soff[j], src + tt * p.C);
      }
    }
    if constexpr (TMA) {
#ifdef SWIN_WATTN_FAULT_INJECTION
      // armed: thread 0 withholds its arrival on the CTA's first cp.async-gathered window
      // (no copy-engine bytes land after it), so that window's bounded wait runs out
      if (!(p.fault == kFaultFwdMmaSync && tid == 0 && first_gather))
#endif
        tc::cp_async_arrive(bar0 + 8 * stage);
    }
#ifdef SWIN_WATTN_FAULT_INJECTION
    first_gather = false;
#endif
    if (++lwx == p.nWx) {
      lwx = 0;
      if (++lwy == p.nWy) {
        lwy = 0;
        ++lb;
      }
    }
  };

  if constexpr (TMA) {
    if (tid == 0) {
      for (int st = 0; st < STAGES; ++st) tc::mbar_init(bar0 + 8 * st, THREADS + 1);
      tc::mbar_init_fence();
    }
    __syncthreads();
  }
  // Padded rows N..NPAD-1 of every q/k/v tile are zero (loads never touch them).
  if constexpr (G::NPAD > N) {
    constexpr int PADROWS = G::NPAD - N;
    for (int e = tid; e < STAGES * 3 * PADROWS * 4; e += THREADS) {
      const int c = e & 3, r = (e >> 2) % PADROWS, tile = (e >> 2) / PADROWS;
      *reinterpret_cast<uint4*>(stiles + tile * G::TILE_BYTES + tile_off(N + r, c)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  pdl_wait();
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
    if (st < nwin) issue(st * G::STAGE_BYTES, st);
    if constexpr (!TMA) cp_async_commit();
  }

  const float4* bfrag = sbias + warp * NT * 32 + lane;
  const float c_l2 = p.qk_scale_log2;            // scale * log2(e)
  // Output slots of this lane: rows warp*16 + g + {0, 8}, 16-byte chunk t.
  const int os0 = warp * 16 + g, os1 = os0 + 8;
  const int oly0 = os0 / M, olx0 = os0 % M, oly1 = os1 / M, olx1 = os1 % M;
  // U operand of the shift-mask MMA for these two rows (k-slots 8..15 are zero).
  const uint32_t mu0 = mask_u_frag(os0, t, M, s), mu1 = mask_u_frag(os1, t, M, s);
  // B operand of all ones: one extra m16n8 tile of P V yields the row sums of the very
  // bf16 P values that weight V.
  const uint32_t ones = 0x3F803F80u;
  // Lane parts of the ldmatrix addresses (tile-relative; key tile nt adds nt*512 bytes,
  // value k-step kk adds kk*1024 bytes).
  const int mi = lane >> 3, r8 = lane & 7, r16 = r8 + ((mi & 1) << 3);
  const uint32_t q_off0 = tile_off(warp * 16 + r16, mi >> 1);
  const uint32_t q_off1 = tile_off(warp * 16 + r16, 2 + (mi >> 1));
  const uint32_t k_off = G::TILE_BYTES + tile_off(r8, mi);
  const uint32_t v_off0 = 2 * G::TILE_BYTES + tile_off(r16, mi >> 1);
  const uint32_t v_off1 = 2 * G::TILE_BYTES + tile_off(r16, 2 + (mi >> 1));
  // stmatrix row addresses: matrix mi = (row half mi & 1, column chunk 2*call + (mi >> 1))
  const uint32_t st_off0 = tile_off(warp * 16 + r8 + ((mi & 1) << 3), mi >> 1);
  const uint32_t st_off1 = tile_off(warp * 16 + r8 + ((mi & 1) << 3), 2 + (mi >> 1));

  uint32_t cur_off = 0, nxt_off = (STAGES - 1) * G::STAGE_BYTES;
  int cur_st = 0, nxt_st = STAGES - 1, bad = 0, bad_it = 0;
  for (int it = 0; it < nwin; ++it) {
    if constexpr (TMA) {
      // the window's tiles: every thread's cp.async and the copy engine's bytes (bounded)
      const bool ok = tc::mbar_wait(bar0 + 8 * cur_st, (it / STAGES) & 1, p.wait_ns);
      if (__syncthreads_or(ok ? 0 : 1)) {
        bad = 1;
        bad_it = it;
        break;
      }
      if (it + STAGES - 1 < nwin) issue(nxt_off, nxt_st);
    } else {
      cp_async_wait<STAGES - 2>();
      __syncthreads();
      if (it + STAGES - 1 < nwin) issue(nxt_off, nxt_st);
      cp_async_commit();
    }
    cur_st = cur_st + 1 == STAGES ? 0 : cur_st + 1;
    nxt_st = nxt_st + 1 == STAGES ? 0 : nxt_st + 1;
    nxt_off = nxt_off + G::STAGE_BYTES == STAGES * G::STAGE_BYTES ? 0 : nxt_off + G::STAGE_BYTES;
    const int b = cb, wy = cwy, wx = cwx;
    if (++cwx == p.nWx) {
      cwx = 0;
      if (++cwy == p.nWy) {
        cwy = 0;
        ++cb;
      }
    }
    unsigned char* tq = stiles + cur_off;
    const uint32_t tb = tiles_u32 + cur_off;
    cur_off = cur_off + G::STAGE_BYTES == STAGES * G::STAGE_BYTES ? 0 : cur_off + G::STAGE_BYTES;

    // ---- z = Q K^T + bias/scale: the accumulators start from the bias fragment ------
    uint32_t qa[2][4];
    ldsm_x4(tb + q_off0, qa[0][0], qa[0][1], qa[0][2], qa[0][3]);
    ldsm_x4(tb + q_off1, qa[1][0], qa[1][1], qa[1][2], qa[1][3]);
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float4 bb = bfrag[nt * 32];
      uint32_t b0, b1, b2, b3;
      ldsm_x4(tb + k_off + nt * 512, b0, b1, b2, b3);
      mma_bf16_c(sacc[nt], qa[0][0], qa[0][1], qa[0][2], qa[0][3], b0, b1, bb.x, bb.y, bb.z, bb.w);
      mma_bf16(sacc[nt], qa[1][0], qa[1][1], qa[1][2], qa[1][3], b2, b3);
    }

    // ---- shift mask (boundary windows only): z += U V^T, one k16 MMA per key tile ----
    if (p.mask_frag != nullptr && (wy == p.nWy - 1 || wx == p.nWx - 1)) {
      const int cls = (wy == p.nWy - 1 ? 2 : 0) | (wx == p.nWx - 1 ? 1 : 0);
      const uint4* mv = reinterpret_cast<const uint4*>(smask) + (cls - 1) * (G::NTP / 4) * 32 + lane;
#pragma unroll
      for (int q4 = 0; q4 < G::NTP / 4; ++q4) {
        const uint4 v = mv[q4 * 32];
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q4 * 4 + u < NT) mma_bf16(sacc[q4 * 4 + u], mu0, mu1, 0u, 0u, vw[u], 0u);
      }
    }
    // two interleaved three-input max chains per row
    float m0a = -INFINITY, m0b = -INFINITY, m1a = -INFINITY, m1b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; nt += 2) {
      m0a = fmax3(m0a, sacc[nt][0], sacc[nt][1]);
      m1a = fmax3(m1a, sacc[nt][2], sacc[nt][3]);
      if (nt + 1 < NT) {
        m0b = fmax3(m0b, sacc[nt + 1][0], sacc[nt + 1][1]);
        m1b = fmax3(m1b, sacc[nt + 1][2], sacc[nt + 1][3]);
      }
    }
    float mx0 = fmaxf(m0a, m0b), mx1 = fmaxf(m1a, m1b);
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));

    // ---- softmax numerators: exp2((z - max) * scale * log2e) ------------------------
    // (pairs of one row share the shift: one packed FFMA2 per pair)
    const float2 c2 = make_float2(c_l2, c_l2);
    const float2 nm0 = make_float2(-mx0 * c_l2, -mx0 * c_l2), nm1 = make_float2(-mx1 * c_l2, -mx1 * c_l2);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 e0 = __ffma2_rn(make_float2(sacc[nt][0], sacc[nt][1]), c2, nm0);
      const float2 e1 = __ffma2_rn(make_float2(sacc[nt][2], sacc[nt][3]), c2, nm1);
      sacc[nt][0] = fast_exp2(e0.x);
      sacc[nt][1] = fast_exp2(e0.y);
      sacc[nt][2] = fast_exp2(e1.x);
      sacc[nt][3] = fast_exp2(e1.y);
    }

    // ---- O = P V, row sums from the ones tile ---------------------------------------
    float o[4][4], lsum[4];
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const uint32_t a0 = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      const uint32_t a1 = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      uint32_t a2 = 0u, a3 = 0u;
      if (2 * kk + 1 < NT) {
        a2 = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        a3 = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
      }
      uint32_t v0, v1, v2, v3, w0, w1, w2, w3;
      ldsm_x4_t(tb + v_off0 + kk * 1024, v0, v1, v2, v3);
      ldsm_x4_t(tb + v_off1 + kk * 1024, w0, w1, w2, w3);
      if (kk == 0) {
        mma_bf16_c(o[0], a0, a1, a2, a3, v0, v1, 0.f, 0.f, 0.f, 0.f);
        mma_bf16_c(o[1], a0, a1, a2, a3, v2, v3, 0.f, 0.f, 0.f, 0.f);
        mma_bf16_c(o[2], a0, a1, a2, a3, w0, w1, 0.f, 0.f, 0.f, 0.f);
        mma_bf16_c(o[3], a0, a1, a2, a3, w2, w3, 0.f, 0.f, 0.f, 0.f);
        mma_bf16_c(lsum, a0, a1, a2, a3, ones, ones, 0.f, 0.f, 0.f, 0.f);
      } else {
        mma_bf16(o[0], a0, a1, a2, a3, v0, v1);
        mma_bf16(o[1], a0, a1, a2, a3, v2, v3);
        mma_bf16(o[2], a0, a1, a2, a3, w0, w1);
        mma_bf16(o[3], a0, a1, a2, a3, w2, w3);
        mma_bf16(lsum, a0, a1, a2, a3, ones, ones);
      }
    }

    // ---- normalise and store at the gathered token positions ----------------------
    const float inv0 = 1.0f / lsum[0], inv1 = 1.0f / lsum[2];
    const int y0 = wy * M + s, x0 = wx * M + s;
    int ya = y0 + oly0, xa = x0 + olx0, yb = y0 + oly1, xb = x0 + olx1;
    ya = ya >= H ? ya - H : ya;
    xa = xa >= W ? xa - W : xa;
    yb = yb >= H ? yb - H : yb;
    xb = xb >= W ? xb - W : xb;
    const int64_t img = (int64_t)b * H * W;
    const int64_t tok0 = img + ya * W + xa, tok1 = img + yb * W + xb;
    if constexpr (sizeof(TIO) == 2) {
      // Stage the warp's 16 x 32 bf16 rows in its own Q rows (only this warp reads
      // them, and they are consumed) with two stmatrix, then write 64 contiguous bytes
      // per token. Padded rows receive finite values that are never stored.
      const float2 i0 = make_float2(inv0, inv0), i1 = make_float2(inv1, inv1);
      uint32_t ow[4][2];
#pragma unroll
      for (int nd = 0; nd < 4; ++nd) {
        const float2 a = __fmul2_rn(make_float2(o[nd][0], o[nd][1]), i0);
        const float2 c = __fmul2_rn(make_float2(o[nd][2], o[nd][3]), i1);
        ow[nd][0] = pack_bf16(a.x, a.y);
        ow[nd][1] = pack_bf16(c.x, c.y);
      }
      stsm_x4(tb + st_off0, ow[0][0], ow[0][1], ow[1][0], ow[1][1]);
      stsm_x4(tb + st_off1, ow[2][0], ow[2][1], ow[3][0], ow[3][1]);
      __syncwarp();
      __nv_bfloat16* outp = reinterpret_cast<__nv_bfloat16*>(p.out) + h * kHeadDim + t * 8;
      if (os0 < N)
        *reinterpret_cast<uint4*>(outp + tok0 * p.C) = *reinterpret_cast<const uint4*>(tq + tile_off(os0, t));
      if (os1 < N)
        *reinterpret_cast<uint4*>(outp + tok1 * p.C) = *reinterpret_cast<const uint4*>(tq + tile_off(os1, t));
    } else {
      // fp32 output: each lane writes its own fragment pairs (rows g and g+8).
      float* outp = reinterpret_cast<float*>(p.out) + h * kHeadDim + 2 * t;
      // rows g / g+8 of this warp are slots os0 / os1 (same as the staging slots)
      if (os0 < N) {
        float* dst = outp + tok0 * p.C;
#pragma unroll
        for (int nd = 0; nd < 4; ++nd)
          *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][0] * inv0, o[nd][1] * inv0);
      }
      if (os1 < N) {
        float* dst = outp + tok1 * p.C;
#pragma unroll
        for (int nd = 0; nd < 4; ++nd)
          *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][2] * inv1, o[nd][3] * inv1);
      }
    }
  }
  if constexpr (TMA) {
    if (bad) {
      // after a timeout: the windows already issued behind the one whose wait ran out
      // land before the CTA leaves (their barriers complete with their last bytes)
      for (int k = bad_it + 1; k < nwin && k < bad_it + STAGES - 1; ++k)
        tc::mbar_wait(bar0 + 8 * (k % STAGES), (k / STAGES) & 1, p.wait_ns);
    }
  }
  cp_async_wait_all();
  if (bad && tid == 0) atomicOr(p.err, 1);
}

// ---- host side ---------------------------------------------------------------------

template <int M, typename TIO, int STAGES, bool TMA>
static cudaError_t config_t(const Plan& pl, FwdLaunch* L) {
  using G = Geo<M>;
  constexpr int smem = fwd_smem_bytes<M, TIO, STAGES, TMA>();
  auto kern = fwd_kernel<M, TIO, STAGES, TMA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, G::THREADS, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t total = (int64_t)pl.B * pl.nW;
  int64_t target = (int64_t)pl.num_sms * occ;
  int64_t chunks = target / pl.nH;
  if (chunks < 1) chunks = 1;
  if (chunks > total) chunks = total;
  L->chunks = (int)chunks;
  L->grid = (int)(chunks * pl.nH);
  L->threads = G::THREADS;
  L->smem = smem;
  L->ctas_per_sm = occ;
  L->tma = TMA;
  return cudaSuccess;
}

// Forward over `batch` images starting at the given pointers (batch <= the plan's B): one
// wave of CTAs sized as in config_t for that many windows.
template <int M, typename TIO, int STAGES, bool TMA>
static cudaError_t launch_t(const Plan& pl, const FwdLaunch& L0, const void* qkv, void* out,
                            int batch, cudaStream_t st) {
  FwdLaunch L = L0;
  if (batch != pl.B) {
    const int64_t total = (int64_t)batch * pl.nW;
    int64_t chunks = ((int64_t)pl.num_sms * L0.ctas_per_sm) / pl.nH;
    if (chunks < 1) chunks = 1;
    if (chunks > total) chunks = total;
    L.chunks = (int)chunks;
    L.grid = (int)(chunks * pl.nH);
  }
  CUtensorMap gather_map, box_map, top_map, bot_map;
  if constexpr (TMA) {
    cudaError_t e = make_qkv_maps(pl, qkv, batch, &gather_map, &box_map, &top_map, &bot_map);
    if (e != cudaSuccess) return e;
  } else {
    memset(&box_map, 0, sizeof(box_map));
    top_map = bot_map = box_map;
  }
  FwdParams p;
  p.qkv = qkv;
  p.out = out;
  p.bias_frag = pl.bias_frag;
  p.mask_frag = pl.s > 0 ? pl.mask_frag : nullptr;
  p.H = pl.H;
  p.W = pl.W;
  p.C = pl.C;
  p.nH = pl.nH;
  p.s = pl.s;
  p.nWy = pl.nWy;
  p.nWx = pl.nWx;
  p.nW = pl.nW;
  p.total_windows = (int64_t)batch * pl.nW;
  p.chunks = L.chunks;
  p.qk_scale_log2 = kLog2e / kInvScale;
  p.err = pl.err;
  p.wait_ns = wait_limit_ns();
  p.fault = fault_site();
  return launch_pdl(fwd_kernel<M, TIO, STAGES, TMA>, dim3(L.grid), dim3(L.threads), L.smem, st, box_map, top_map,
                    bot_map, p);
}

// Pipeline depth per window size: enough windows in flight per SM while keeping the
// shared-memory footprint within the residency target.
template <int M> struct FwdStages { static constexpr int value = 3; };
template <> struct FwdStages<12> { static constexpr int value = 2; };

// The copy engine feeds 7x7 bf16 windows (its boxes are 7 x 7 tokens; tokens are
// addressed by 32-bit coordinates).
static bool fwd_tma_applies(const Plan& pl) {
  return pl.M == 7 && pl.dtype == SWIN_WATTN_BF16 && (int64_t)pl.B * pl.H * pl.W < ((int64_t)1 << 31);
}

#define SWIN_FWD_DISPATCH(FN, ...)                                                       \
  do {                                                                                  \
    const bool f32 = pl.dtype == SWIN_WATTN_FP32;                                       \
    switch (pl.M) {                                                                     \
      case 4:                                                                           \
        return f32 ? FN<4, float, FwdStages<4>::value, false>(__VA_ARGS__)               \
                   : FN<4, __nv_bfloat16, FwdStages<4>::value, false>(__VA_ARGS__);      \
      case 7:                                                                           \
        if (f32) return FN<7, float, FwdStages<7>::value, false>(__VA_ARGS__);           \
        return tma ? FN<7, __nv_bfloat16, FwdStages<7>::value, true>(__VA_ARGS__)        \
                   : FN<7, __nv_bfloat16, FwdStages<7>::value, false>(__VA_ARGS__);      \
      case 12:                                                                          \
        return f32 ? FN<12, float, FwdStages<12>::value, false>(__VA_ARGS__)             \
                   : FN<12, __nv_bfloat16, FwdStages<12>::value, false>(__VA_ARGS__);    \
      default:                                                                          \
        return cudaErrorInvalidValue;                                                   \
    }                                                                                   \
  } while (0)

static cudaError_t mma_config(const Plan& pl, FwdLaunch* L) {
  const bool tma = fwd_tma_applies(pl);
  SWIN_FWD_DISPATCH(config_t, pl, L);
}

static cudaError_t mma_launch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out, int batch,
                              cudaStream_t st) {
  const bool tma = L.tma;
  SWIN_FWD_DISPATCH(launch_t, pl, L, qkv, out, batch, st);
}

bool fwd_tc_applies(const Plan& pl);
cudaError_t fwd_tc_config(const Plan& pl, FwdLaunch* L);
bool fwd12_tc_applies(const Plan& pl);
cudaError_t fwd12_tc_config(const Plan& pl, FwdLaunch* L);
cudaError_t fwd12_tc_launch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out, int batch,
                            cudaStream_t st);
cudaError_t fwd_tc_launch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out, int batch,
                          cudaStream_t st);

// Kernel choice: the tcgen05 kernel when the plan asks for it (7x7 or 12x12 windows,
// bf16); with AUTO, the tcgen05 kernel for 12x12 windows when there are at least 16
// window-heads per SM (its per-CTA start-up then amortises: measured faster on the Swin-L
// 384 96x96 and 48x48 stages, slower on the 24x24 one), else the mma.sync kernel.
static bool fwd12_auto(const Plan& pl) {
  return pl.fwd_kernel == SWIN_WATTN_KERNEL_AUTO && fwd12_tc_applies(pl) &&
         (int64_t)pl.B * pl.nW * pl.nH >= 16 * (int64_t)pl.num_sms;
}

cudaError_t fwd_config(const Plan& pl, FwdLaunch* L) {
  *L = FwdLaunch();
  if (pl.fwd_kernel == SWIN_WATTN_KERNEL_TCGEN05 || fwd12_auto(pl)) {
    L->tc = true;
    if (fwd_tc_applies(pl)) return fwd_tc_config(pl, L);
    if (fwd12_tc_applies(pl)) return fwd12_tc_config(pl, L);
    *L = FwdLaunch();
    return cudaErrorNotSupported;
  }
  return mma_config(pl, L);
}

cudaError_t fwd_launch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out,
                       cudaStream_t st) {
  if (L.tc) return pl.M == 12 ? fwd12_tc_launch(pl, L, qkv, out, pl.B, st) : fwd_tc_launch(pl, L, qkv, out, pl.B, st);
  return mma_launch(pl, L, qkv, out, pl.B, st);
}

cudaError_t fwd_launch_batch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out,
                             int batch, cudaStream_t st) {
  if (L.tc) return pl.M == 12 ? fwd12_tc_launch(pl, L, qkv, out, batch, st) : fwd_tc_launch(pl, L, qkv, out, batch, st);
  return mma_launch(pl, L, qkv, out, batch, st);
}

}  // namespace swin
