// Fused (shifted-)window attention forward on the fifth-generation tensor cores for 12 x 12
// windows (tcgen05, tensor memory, TMA), bf16 activations.
//
// The same function as fwd.cu (NVIDIA Swin talk transcript, uticex.com article 1598,
// section 2: the shift and the partition are index mappings folded into the loads, the
// reverse and un-roll into the stores; section 3: the bias lookup done once per plan):
//   Y[token(i)] = sum_j P_ij V[token(j)],  P = softmax_j(scale q_i.k_j + bias_h(i, j) + mask(i, j))
// for each window and head, i, j over the window's 144 slots.
//
// A CTA owns one head and a range of windows and holds all of the SM's tensor memory. A
// window's 144 query rows are two M = 128 row tiles: tile A rows 0-127 and tile B rows
// 32-159 (its lanes 96-111 are rows 128-143; the rest repeat tile A's rows or run past
// the window into the next tile of shared memory and are not read). Per window:
// * the producer warp loads q, k and v (144 rows x 64 bytes, 64-byte swizzled, four
//   stages) with one 12 x 12-token box per tensor, two row bands where the window wraps
//   at the bottom only; a window that wraps at the right comes in by tile::gather4 loads
//   (four tokens of any position each, 36 per tensor), so every tile is in slot order;
// * one MMA warp issues S = Q K^T (M128 N144 K16) into tensor memory for both row tiles,
//   a second one O = P V (M128 N32 K16, P from tensor memory) once P is written;
// * four softmax warps for tile A: thread r loads its row of S, scales it, adds the bias
//   row (the plan's dense bias, in shared memory) and the shift mask
//   (boundary windows of a shifted layer, from the slots' regions), takes the row maximum,
//   exp2, writes P as bf16 to tensor memory and keeps the row sum; one window later it
//   reads its row of O, divides by that sum and stores the row at the token it came from;
// * a fifth softmax warp does the same for rows 128-143 with the sixteen-lane access
//   shapes, four lanes to a row, so that the SM sub-partition that also runs tile A's
//   rows 96-127 does half a warp's row work more, not a whole warp's.
// Hand-offs are mbarriers; every wait is bounded and a wait that runs out ends in the
// plan's error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kTM = 12, kTN = 144;
constexpr int kROW = 64;                   // one token's 32 bf16 head channels
constexpr int kTILE = kTN * kROW;          // 9216 bytes: the window's 144 slot rows
// stage: q | k | v
constexpr int kSTAGE = 3 * kTILE;          // 27648 bytes (27 KB)
constexpr int kSTAGES = 4;
constexpr int kGROUPS = kTN / 4;           // gather4 row groups of a tile
constexpr int kOFF_BIAS = kSTAGES * kSTAGE;
// the head's dense bias, fp32, rows padded to 148 floats: the 16-byte reads of eight
// consecutive rows at one column then fall in distinct banks
constexpr int kBST = 148;
constexpr int kBIAS_ROW_BYTES = kTN * 4;
constexpr int kBIAS_BYTES = kTN * kBIAS_ROW_BYTES;
constexpr int kBIAS_SPACE = (kTN * kBST * 4 + 1023) / 1024 * 1024;
constexpr int kSTG_WARP = 32 * kROW;        // per softmax warp: its rows of Y, staged
constexpr int kOFF_STG = kOFF_BIAS + kBIAS_SPACE;
constexpr int kOFF_BAR = kOFF_STG + 5 * kSTG_WARP;
constexpr int kNBAR = 2 * kSTAGES + 7;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + the tensor-memory slot, alignment slack
static_assert(kSTAGE % 1024 == 0 && kOFF_BIAS % 1024 == 0 && kOFF_STG % 1024 == 0, "1024-byte aligned tiles");
static_assert(kSMEM <= 232448, "shared memory of one CTA");
// Tensor memory: S of tile A [0,144) and B [160,304), P (bf16 pairs) of A [304,376) and B
// [376,448), O of A [448,480) and B [480,512); S and O start on 32-column boundaries.
constexpr int kTMEM_COLS = 512;
constexpr int kSA = 0, kSB = 160, kPA = 304, kPB = 376, kOA = 448, kOB = 480;
// warps 0-3: softmax, tile A rows 32w..; 4: producer; 5: S products; 6: O products;
// 7: softmax, rows 128-143 (tile B lanes 96-111)
constexpr int kPROD_WARP = 4, kS_WARP = 5, kO_WARP = 6, kTAIL_WARP = 7;
constexpr int kTHREADS = 8 * 32;
constexpr uint32_t kSW64 = 4;

struct Fwd12Params {
  __nv_bfloat16* out;
  const float* bias;  // the plan's dense bias [nH][144][144]
  int* err;
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;
  int chunks;
  int fault;    // armed fault site (fault-injection build only)
  float scale;  // hd^-0.5
  // key j lies in the wrapped row band when j / 12 >= 12 - s (bit j % 32 of ky[j / 32]), in
  // the wrapped column band when j % 12 >= 12 - s (kx)
  uint32_t ky[5], kx[5];
  uint64_t wait_ns;
};

struct Cursor12 {
  int b, wy, wx;
  __device__ __forceinline__ void next(int nWy, int nWx) {
    if (++wx == nWx) {
      wx = 0;
      if (++wy == nWy) {
        wy = 0;
        ++b;
      }
    }
  }
};

__device__ __forceinline__ bool warp_wait12(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, limit_ns)) != 0;
}

// Byte offset of 16-byte chunk c of 64-byte row r in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz12(int r, int c) {
  return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

}  // namespace

__global__ void __launch_bounds__(kTHREADS, 1)
    fwd12_tc_kernel(const __grid_constant__ CUtensorMap q_box, const __grid_constant__ CUtensorMap q_top,
                    const __grid_constant__ CUtensorMap q_bot, const __grid_constant__ CUtensorMap q_rows,
                    const Fwd12Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 8 * kNBAR);
  pdl_launch_dependents();
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem0 + kOFF_BAR;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto empty_bar = [&](int st) { return bar0 + 8 * (kSTAGES + st); };
  const uint32_t s_full = bar0 + 8 * (2 * kSTAGES), s_free = s_full + 8, p_full = s_full + 16;
  const uint32_t o_full = s_full + 24, o_free = s_full + 32, const_bar = s_full + 40, drain_bar = s_full + 48;
  auto wwait = [&](uint32_t mbar, uint32_t parity) { return warp_wait12(mbar, parity, p.wait_ns); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int H = p.H, W = p.W, s = p.s;
  Cursor12 first;
  first.b = (int)(w_begin / p.nW);
  {
    const int w = (int)(w_begin - (int64_t)first.b * p.nW);
    first.wy = w / p.nWx;
    first.wx = w - first.wy * p.nWx;
  }
  // a window of a shifted layer wraps at the bottom in the last window row, at the right
  // in the last window column
  auto wraps_y = [&](const Cursor12& c) { return s > 0 && c.wy == p.nWy - 1; };
  auto wraps_x = [&](const Cursor12& c) { return s > 0 && c.wx == p.nWx - 1; };

  // ---- set-up: tensor memory, barriers ----------------------------------------------
  if (warp == 0) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < kSTAGES; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 1);  // the O products' commit
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_free, 5);  // the five softmax warps
    tc::mbar_init(p_full, 5);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(o_free, 5);
    tc::mbar_init(const_bar, 1);
    tc::mbar_init(drain_bar, 2);  // the two MMA warps' commits
    tc::mbar_init_fence();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int bad = 0;
  pdl_wait();  // activations and the plan's bias from here on

  if (warp == kPROD_WARP) {
    // ==== producer: q, k, v of window n into stage n % kSTAGES (one thread issues) ========
    int issued = 0;
    if (lane == 0) tc::mbar_expect_tx(const_bar, kBIAS_BYTES);
    __syncwarp();
    for (int r = lane; r < kTN; r += 32)
      tc::bulk_copy(smem0 + kOFF_BIAS + r * kBST * 4, p.bias + ((size_t)h * kTN + r) * kTN, kBIAS_ROW_BYTES, const_bar);
    Cursor12 cur = first;
    for (int n = 0, st = 0; n < nwin; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
      if (n >= kSTAGES && !wwait(empty_bar(st), ((n / kSTAGES) - 1) & 1)) {
        bad = 1;
        break;
      }
      issued = n + 1;
      const bool wy = wraps_y(cur), wx = wraps_x(cur);
      const uint32_t stage = smem0 + st * kSTAGE;
      if (lane == 0) tc::mbar_expect_tx(full_bar(st), 3 * kTILE);
      __syncwarp();
      if (!wx) {
        if (lane == 0) {
          const int x0 = cur.wx * kTM + s, y0 = cur.wy * kTM + s;
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const int col = t * p.C + h * kHeadDim;
            const uint32_t dst = stage + t * kTILE;
            if (!wy) {
              tc::box_load(dst, &q_box, col, x0, y0, cur.b, full_bar(st));
            } else {
              tc::box_load(dst, &q_top, col, x0, y0, cur.b, full_bar(st));
              tc::box_load(dst + (kTM - s) * kTM * kROW, &q_bot, col, x0, 0, cur.b, full_bar(st));
            }
          }
        }
      } else {
        // the window wraps at the right: four slots a load, slot i from token
        // ((wy 12 + i / 12 + s) mod H, (wx 12 + i % 12 + s) mod W)
        for (int g = lane; g < kGROUPS; g += 32) {
          int row[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = 4 * g + q;
            int y = cur.wy * kTM + i / kTM + s, x = cur.wx * kTM + i % kTM + s;
            y = y >= H ? y - H : y;
            x = x >= W ? x - W : x;
            row[q] = (cur.b * H + y) * W + x;
          }
#pragma unroll
          for (int t = 0; t < 3; ++t)
            tc::gather4(stage + t * kTILE + g * 4 * kROW, &q_rows, t * p.C + h * kHeadDim, row[0], row[1], row[2],
                        row[3], full_bar(st));
        }
      }
      __syncwarp();
      cur.next(p.nWy, p.nWx);
    }
    // every load issued has landed before the CTA leaves
    for (int m = issued > kSTAGES ? issued - kSTAGES : 0; m < issued; ++m)
      tc::mbar_wait(full_bar(m % kSTAGES), (m / kSTAGES) & 1, p.wait_ns);
    tc::mbar_wait(const_bar, 0, p.wait_ns);
  } else if (warp == kS_WARP || warp == kO_WARP) {
    // ==== MMA issue: one thread per warp ==================================================
    const uint32_t id_s = tc::idesc_bf16(128, kTN, false);  // Q, K: K-major
    const uint32_t id_o = tc::idesc_bf16(128, 32, true);    // V: MN-major; P in tensor memory
    for (int n = 0, st = 0; n < nwin && !bad; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
      const uint32_t stage = smem0 + st * kSTAGE;
      if (warp == kS_WARP) {
        // S = Q K^T for both row tiles, once the tiles have landed and the softmax warps
        // have read the last window's S
        if (!wwait(full_bar(st), (n / kSTAGES) & 1) || (n > 0 && !wwait(s_free, (n - 1) & 1))) {
          bad = 1;
          break;
        }
        if (lane == 0) {
          tc::fence_after_sync();
          const uint64_t dq = tc::sdesc(stage, 16, 512, kSW64);  // q; k at +kTILE
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const uint32_t qrow = tile ? 32 * kROW : 0;  // tile B starts at query row 32
            const uint32_t d = tmem + (tile ? kSB : kSA);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              tc::mma_ss(d, tc::desc_add(dq, qrow + kk * 32), tc::desc_add(dq, kTILE + kk * 32), id_s, kk > 0);
            }
          }
          tc::commit(s_full);
        }
        __syncwarp();
      } else {
        // O = P V for both row tiles, once P is written and the last window's O has been
        // read; then the stage is free
        if (!wwait(p_full, n & 1) || (n > 0 && !wwait(o_free, (n - 1) & 1))) {
          bad = 1;
          break;
        }
        if (lane == 0) {
          tc::fence_after_sync();
          const uint64_t dv = tc::sdesc(stage + 2 * kTILE, kTILE, 512, kSW64);
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const uint32_t d = tmem + (tile ? kOB : kOA), a = tmem + (tile ? kPB : kPA);
#pragma unroll
            for (int kk = 0; kk < kTN / 16; ++kk) {  // 16 keys a step
              tc::mma_ts(d, a + kk * 8, tc::desc_add(dv, kk * 1024), id_o, kk > 0);
            }
          }
          tc::commit(o_full);
          tc::commit(empty_bar(st));
        }
        __syncwarp();
      }
    }
    // every MMA this thread issued has completed before the tensor memory is released
    if (lane == 0) tc::commit(drain_bar);
    __syncwarp();
    if (!wwait(drain_bar, 0)) bad = 1;
  } else if (warp < 4) {
    // ==== softmax warps 0-3: tile A, thread r of warp w owns query row i = 32 w + r =========
    const int i = 32 * warp + lane;
    const int ly = i / kTM, lx = i % kTM;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    const float* brow = reinterpret_cast<const float*>(smem + kOFF_BIAS) + i * kBST;
    unsigned char* stg = smem + kOFF_STG + warp * kSTG_WARP;
    const float2 sc2 = make_float2(p.scale, p.scale), l2e2 = make_float2(kLog2e, kLog2e);
    const int th = kTM - s;  // local index from which a slot lies in the wrapped region
    if (!wwait(const_bar, 0)) bad = 1;
    const float4* brow4 = reinterpret_cast<const float4*>(brow);
    Cursor12 cur = first, prev = first;
    float inv_prev = 0.0f;
    for (int n = 0; n <= nwin && !bad; ++n) {
      uint32_t pw[9][8];  // window n's P row as bf16 pairs (keys 2c, 2c + 1 in word c = 8q + u)
      float inv = 0.0f;
      if (n < nwin) {
        // ---- S row, bias, mask, max, exp2, P -----------------------------------------
        if (!wwait(s_full, n & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t a0[32], a1[32], a2[32], a3[32], a4[16];
        tc::ld32_nowait(trow + kSA, a0);
        tc::ld32_nowait(trow + kSA + 32, a1);
        tc::ld32_nowait(trow + kSA + 64, a2);
        tc::ld32_nowait(trow + kSA + 96, a3);
        tc::ld16_nowait(trow + kSA + 128, a4);
        tc::wait_ld_then();
        tc::dep32(a0);
        tc::dep32(a1);
        tc::dep32(a2);
        tc::dep32(a3);
        tc::dep16(a4);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free);
        float2 t[kTN / 2];  // keys 2q, 2q + 1
#pragma unroll
        for (int q = 0; q < kTN / 4; ++q) {
          const float4 b4 = brow4[q];
          uint32_t sj[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * q + u;
            sj[u] = j < 32 ? a0[j] : j < 64 ? a1[j - 32] : j < 96 ? a2[j - 64] : j < 128 ? a3[j - 96] : a4[j - 128];
          }
          t[2 * q] = __ffma2_rn(make_float2(__uint_as_float(sj[0]), __uint_as_float(sj[1])), sc2, make_float2(b4.x, b4.y));
          t[2 * q + 1] =
              __ffma2_rn(make_float2(__uint_as_float(sj[2]), __uint_as_float(sj[3])), sc2, make_float2(b4.z, b4.w));
        }
        const bool lastrow = wraps_y(cur), lastcol = wraps_x(cur);
        if (lastrow || lastcol) {
          // the shift mask: slots of different regions of a boundary window never meet;
          // key j is cut when its row band differs from the query's (last window row) or
          // its column band does (last window column)
          const uint32_t fy = lastrow ? ~0u : 0u, fx = lastcol ? ~0u : 0u;
          const uint32_t ry = ly >= th ? ~0u : 0u, rx = lx >= th ? ~0u : 0u;
          uint32_t cw[5];
#pragma unroll
          for (int w = 0; w < 5; ++w) cw[w] = (fy & (p.ky[w] ^ ry)) | (fx & (p.kx[w] ^ rx));
#pragma unroll
          for (int j = 0; j < kTN; ++j) {
            const bool cut = (cw[j >> 5] >> (j & 31)) & 1u;
            if (j & 1)
              t[j >> 1].y = cut ? t[j >> 1].y + kMaskValue : t[j >> 1].y;
            else
              t[j >> 1].x = cut ? t[j >> 1].x + kMaskValue : t[j >> 1].x;
          }
        }
        float m0 = fmaxf(t[0].x, t[0].y), m1 = fmaxf(t[1].x, t[1].y);
#pragma unroll
        for (int q = 2; q < kTN / 2; q += 2) {
          m0 = fmax3(m0, t[q].x, t[q].y);
          m1 = fmax3(m1, t[q + 1].x, t[q + 1].y);
        }
        const float mx = fmaxf(m0, m1);
        const float2 nmx = make_float2(-mx * kLog2e, -mx * kLog2e);
        float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < kTN / 2; ++q) {
          const float2 d = __ffma2_rn(t[q], l2e2, nmx);  // (t - max) log2 e
          const float2 e = make_float2(fast_exp2(d.x), fast_exp2(d.y));
          pw[q >> 3][q & 7] = pack_bf16(e.x, e.y);
          sum2 = __fadd2_rn(sum2, e);
        }
        inv = 1.0f / (sum2.x + sum2.y);
      }
      if (n > 0) {
        // ---- window n - 1: O row / sum, stored at the token its query came from ------------
        if (!wwait(o_full, (n - 1) & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t o[32];
        tc::ld32_nowait(trow + kOA, o);
        tc::wait_ld_then();
        tc::dep32(o);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
        const float2 i2 = make_float2(inv_prev, inv_prev);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[8 * q + 2 * u]), __uint_as_float(o[8 * q + 2 * u + 1])), i2);
            w4[u] = pack_bf16(v.x, v.y);
          }
          *reinterpret_cast<uint4*>(stg + swz12(lane, q)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        int yy = prev.wy * kTM + ly + s, xx = prev.wx * kTM + lx + s;
        yy = yy >= H ? yy - H : yy;
        xx = xx >= W ? xx - W : xx;
        const long long tok = ((long long)prev.b * H + yy) * W + xx;
        __syncwarp();
        // the warp's rows, four lanes to a 64-byte row (eight rows per store instruction)
        const int rl = lane >> 2, ch = lane & 3;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int src = rl + 8 * k;
          const long long tk = __shfl_sync(0xffffffffu, tok, src);
          reinterpret_cast<uint4*>(p.out + tk * p.C + h * kHeadDim)[ch] = *reinterpret_cast<const uint4*>(stg + swz12(src, ch));
        }
        __syncwarp();  // the staging rows are read before the next window's
      }
      if (n < nwin) {
        // ---- P to tensor memory (the last window's P V products are done) ---------------
#pragma unroll
        for (int q = 0; q < 9; ++q) tc::st_x8(trow + kPA + 8 * q, pw[q]);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
#ifdef SWIN_WATTN_FAULT_INJECTION
        // armed: softmax warp 0 withholds its arrival for the first window, so the O
        // issuer's bounded wait for P runs out
        if (!(p.fault == kFaultFwdTcgen05 && warp == 0 && n == 0))
#endif
          if (lane == 0) tc::mbar_arrive(p_full);
        inv_prev = inv;
        prev = cur;
        cur.next(p.nWy, p.nWx);
      }
    }
  } else if (warp == kTAIL_WARP) {
    // ==== softmax warp 7: query rows 128 + a and 136 + a (a = lane / 4), tile B lanes 96-111,
    // read and written sixteen lanes at a time; the thread holds keys 8k + 2m and 8k + 2m + 1
    // (m = lane % 4) of both rows, and the quad of four lanes shares the row maximum and sum
    const int a = lane >> 2, m = lane & 3;
    const int ra = 128 + a, rb = 136 + a;
    const uint32_t trow = tmem + (96u << 16);
    const float* bra = reinterpret_cast<float*>(smem + kOFF_BIAS) + ra * kBST + 2 * m;
    const float* brb = reinterpret_cast<float*>(smem + kOFF_BIAS) + rb * kBST + 2 * m;
    unsigned char* stg = smem + kOFF_STG + 4 * kSTG_WARP;
    const float2 sc2 = make_float2(p.scale, p.scale), l2e2 = make_float2(kLog2e, kLog2e);
    const int th = kTM - s;
    // regions of the thread's keys (bit 2k + e: key 8k + 2m + e) and of its two rows
    uint64_t kyb = 0, kxb = 0;
#pragma unroll
    for (int k = 0; k < kTN / 8; ++k)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 8 * k + 2 * m + e;
        kyb |= (uint64_t)(j / kTM >= th) << (2 * k + e);
        kxb |= (uint64_t)(j % kTM >= th) << (2 * k + e);
      }
    const bool rya = ra / kTM >= th, rxa = ra % kTM >= th, ryb = rb / kTM >= th, rxb = rb % kTM >= th;
    if (!wwait(const_bar, 0)) bad = 1;
    // the staged output rows r = lane / 4 and r + 8 (query rows 128 + r, 136 + r), chunk lane % 4
    const int sr = lane >> 2, ch = lane & 3;
    const int ly0 = (128 + sr) / kTM, lx0 = (128 + sr) % kTM, ly1 = (136 + sr) / kTM, lx1 = (136 + sr) % kTM;
    Cursor12 cur = first, prev = first;
    float inva_prev = 0.0f, invb_prev = 0.0f;
    for (int n = 0; n <= nwin && !bad; ++n) {
      uint32_t pw[36];  // P words: pw[2k] row a, pw[2k + 1] row b, column 4k + m (keys 8k + 2m, + 1)
      float inva = 0.0f, invb = 0.0f;
      if (n < nwin) {
        if (!wwait(s_full, n & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t s0[32], s1[32], s2[8];
        tc::ld16x256b_x8_nowait(trow + kSB, s0);
        tc::ld16x256b_x8_nowait(trow + kSB + 64, s1);
        tc::ld16x256b_x2_nowait(trow + kSB + 128, s2);
        tc::wait_ld_then();
        tc::dep32(s0);
        tc::dep32(s1);
        tc::dep8(s2);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free);
        float2 ta[kTN / 8], tb[kTN / 8];
#pragma unroll
        for (int k = 0; k < kTN / 8; ++k) {
          const uint32_t* sk = k < 8 ? s0 + 4 * k : k < 16 ? s1 + 4 * (k - 8) : s2 + 4 * (k - 16);
          ta[k] = __ffma2_rn(make_float2(__uint_as_float(sk[0]), __uint_as_float(sk[1])), sc2,
                             *reinterpret_cast<const float2*>(bra + 8 * k));
          tb[k] = __ffma2_rn(make_float2(__uint_as_float(sk[2]), __uint_as_float(sk[3])), sc2,
                             *reinterpret_cast<const float2*>(brb + 8 * k));
        }
        const bool lastrow = wraps_y(cur), lastcol = wraps_x(cur);
        if (lastrow || lastcol) {
          const uint64_t ca = (lastrow ? (rya ? ~kyb : kyb) : 0) | (lastcol ? (rxa ? ~kxb : kxb) : 0);
          const uint64_t cb = (lastrow ? (ryb ? ~kyb : kyb) : 0) | (lastcol ? (rxb ? ~kxb : kxb) : 0);
#pragma unroll
          for (int k = 0; k < kTN / 8; ++k) {
            ta[k].x += (ca >> (2 * k)) & 1 ? kMaskValue : 0.0f;
            ta[k].y += (ca >> (2 * k + 1)) & 1 ? kMaskValue : 0.0f;
            tb[k].x += (cb >> (2 * k)) & 1 ? kMaskValue : 0.0f;
            tb[k].y += (cb >> (2 * k + 1)) & 1 ? kMaskValue : 0.0f;
          }
        }
        float ma = fmaxf(ta[0].x, ta[0].y), mb = fmaxf(tb[0].x, tb[0].y);
#pragma unroll
        for (int k = 1; k < kTN / 8; ++k) {
          ma = fmax3(ma, ta[k].x, ta[k].y);
          mb = fmax3(mb, tb[k].x, tb[k].y);
        }
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        const float2 nma = make_float2(-ma * kLog2e, -ma * kLog2e), nmb = make_float2(-mb * kLog2e, -mb * kLog2e);
        float2 suma = make_float2(0.0f, 0.0f), sumb = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < kTN / 8; ++k) {
          const float2 da = __ffma2_rn(ta[k], l2e2, nma), db = __ffma2_rn(tb[k], l2e2, nmb);
          const float2 ea = make_float2(fast_exp2(da.x), fast_exp2(da.y));
          const float2 eb = make_float2(fast_exp2(db.x), fast_exp2(db.y));
          pw[2 * k] = pack_bf16(ea.x, ea.y);
          pw[2 * k + 1] = pack_bf16(eb.x, eb.y);
          suma = __fadd2_rn(suma, ea);
          sumb = __fadd2_rn(sumb, eb);
        }
        float sa = suma.x + suma.y, sb = sumb.x + sumb.y;
        sa += __shfl_xor_sync(0xffffffffu, sa, 1);
        sb += __shfl_xor_sync(0xffffffffu, sb, 1);
        sa += __shfl_xor_sync(0xffffffffu, sa, 2);
        sb += __shfl_xor_sync(0xffffffffu, sb, 2);
        inva = 1.0f / sa;
        invb = 1.0f / sb;
      }
      if (n > 0) {
        // ---- window n - 1: rows 128-143 of O / sum -------------------------------------
        if (!wwait(o_full, (n - 1) & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t o[16];  // o[4k], o[4k + 1]: row a, channels 8k + 2m, + 1; o[4k + 2], o[4k + 3]: row b
        tc::ld16x256b_x4_nowait(trow + kOB, o);
        tc::wait_ld_then();
        tc::dep16(o);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
        const float2 ia = make_float2(inva_prev, inva_prev), ib = make_float2(invb_prev, invb_prev);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 va = __fmul2_rn(make_float2(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1])), ia);
          const float2 vb = __fmul2_rn(make_float2(__uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])), ib);
          *reinterpret_cast<uint32_t*>(stg + swz12(a, k) + 4 * m) = pack_bf16(va.x, va.y);
          *reinterpret_cast<uint32_t*>(stg + swz12(a + 8, k) + 4 * m) = pack_bf16(vb.x, vb.y);
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          int yy = prev.wy * kTM + (r ? ly1 : ly0) + s, xx = prev.wx * kTM + (r ? lx1 : lx0) + s;
          yy = yy >= H ? yy - H : yy;
          xx = xx >= W ? xx - W : xx;
          const long long tok = ((long long)prev.b * H + yy) * W + xx;
          reinterpret_cast<uint4*>(p.out + tok * p.C + h * kHeadDim)[ch] =
              *reinterpret_cast<const uint4*>(stg + swz12(sr + 8 * r, ch));
        }
        __syncwarp();
      }
      if (n < nwin) {
        uint32_t p0[32], p1[4];
#pragma unroll
        for (int u = 0; u < 32; ++u) p0[u] = pw[u];
#pragma unroll
        for (int u = 0; u < 4; ++u) p1[u] = pw[32 + u];
        tc::st16x128b_x16(trow + kPB, p0);
        tc::st16x128b_x2(trow + kPB + 64, p1);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full);
        inva_prev = inva;
        invb_prev = invb;
        prev = cur;
        cur.next(p.nWy, p.nWx);
      }
    }
  }
  if (bad) atomicOr(p.err, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

// ---- host side ---------------------------------------------------------------------

// 12 x 12 windows with bf16 activations, tokens addressed by 32-bit tensor-map rows.
bool fwd12_tc_applies(const Plan& pl) {
  return pl.M == kTM && pl.dtype == SWIN_WATTN_BF16 && (int64_t)pl.B * pl.H * pl.W < ((int64_t)1 << 31);
}

// The qkv maps of `batch` images: one 12 x 12-token box, the two row bands of a window
// that wraps at the bottom (12 - s rows, then s rows), and one-token rows for gather4.
static cudaError_t make_qkv12_maps(const Plan& pl, const void* qkv, int batch, CUtensorMap* box, CUtensorMap* top,
                                   CUtensorMap* bot, CUtensorMap* rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t row = (cuuint64_t)3 * pl.C * 2;
  {
    const cuuint64_t rdims[2] = {(cuuint64_t)3 * pl.C, (cuuint64_t)batch * pl.H * pl.W};
    const cuuint64_t rstrides[1] = {row};
    const cuuint32_t rbox[2] = {kHeadDim, 1};
    const cuuint32_t restride[2] = {1, 1};
    if (encode(rows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), rdims, rstrides, rbox, restride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const cuuint64_t dims[4] = {(cuuint64_t)3 * pl.C, (cuuint64_t)pl.W, (cuuint64_t)pl.H, (cuuint64_t)batch};
  const cuuint64_t strides[3] = {row, row * pl.W, row * pl.W * pl.H};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const cuuint32_t heights[3] = {kTM, (cuuint32_t)(pl.s > 0 ? kTM - pl.s : kTM), (cuuint32_t)(pl.s > 0 ? pl.s : kTM)};
  CUtensorMap* maps[3] = {box, top, bot};
  for (int m = 0; m < 3; ++m) {
    const cuuint32_t bbox[4] = {kHeadDim, kTM, heights[m], 1};
    if (encode(maps[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(qkv), dims, strides, bbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// One CTA of eight warps per SM (it holds all of the tensor memory), one wave.
cudaError_t fwd12_tc_config(const Plan& pl, FwdLaunch* L) {
  cudaError_t e = cudaFuncSetAttribute(fwd12_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fwd12_tc_kernel, kTHREADS, kSMEM);
  if (e != cudaSuccess) return e;
  if (occ != 1) return cudaErrorInvalidConfiguration;
  const int64_t total = (int64_t)pl.B * pl.nW;
  int64_t chunks = (int64_t)pl.num_sms / pl.nH;
  if (chunks < 1) chunks = 1;
  if (total > 0 && chunks > total) chunks = total;
  L->chunks = (int)chunks;
  L->grid = (int)(chunks * pl.nH);
  L->threads = kTHREADS;
  L->smem = kSMEM;
  L->ctas_per_sm = 1;
  L->tc = true;
  return cudaSuccess;
}

cudaError_t fwd12_tc_launch(const Plan& pl, const FwdLaunch& L0, const void* qkv, void* out, int batch,
                            cudaStream_t st) {
  FwdLaunch L = L0;
  const int64_t total = (int64_t)batch * pl.nW;
  if (batch != pl.B) {
    int64_t chunks = (int64_t)pl.num_sms / pl.nH;
    if (chunks < 1) chunks = 1;
    if (chunks > total) chunks = total;
    L.chunks = (int)chunks;
    L.grid = (int)(chunks * pl.nH);
  }
  CUtensorMap box, top, bot, rows;
  cudaError_t e = make_qkv12_maps(pl, qkv, batch, &box, &top, &bot, &rows);
  if (e != cudaSuccess) return e;
  Fwd12Params p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.bias = pl.dense_bias;
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
  p.scale = 1.0f / kInvScale;
  p.fault = fault_site();
  for (int w = 0; w < 5; ++w) {
    p.ky[w] = p.kx[w] = 0;
    for (int b = 0; b < 32; ++b) {
      const int j = 32 * w + b;
      if (j < kTN && j / kTM >= kTM - pl.s) p.ky[w] |= 1u << b;
      if (j < kTN && j % kTM >= kTM - pl.s) p.kx[w] |= 1u << b;
    }
  }
  p.wait_ns = wait_limit_ns();
  return launch_pdl(fwd12_tc_kernel, dim3(L.grid), dim3(L.threads), L.smem, st, box, top, bot, rows, p);
}

}  // namespace swin
