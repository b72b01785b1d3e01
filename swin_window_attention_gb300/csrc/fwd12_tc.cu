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
// 16-143 (its lanes 112-127 are rows 128-143; the rest repeat tile A's rows and are not
// read). Per window:
// * the producer warp loads q, k and v (144 rows x 64 bytes, 64-byte swizzled) with one
//   12 x 12-token box per tensor, two row bands where the window wraps at the bottom; a
//   window that wraps at the right comes in as two boxes per tensor, at x0 and at x0 - W,
//   whose out-of-range tokens the copy engine fills with zeros, so the window's tile is
//   their sum and every product below runs on both halves (Q K^T as four products);
// * one MMA warp issues S = Q K^T (M128 N144 K16) into tensor memory for both row tiles,
//   a second one O = P V (M128 N32 K16, P from tensor memory) once P is written;
// * five softmax warps (tile A's 128 rows, and the 16 rows of tile B in lanes 112-127):
//   thread r loads its row of S, adds the bias row (the plan's dense bias, in shared
//   memory) and the shift mask (boundary windows of a shifted layer, from the slots'
//   regions), takes the row maximum, exp2, writes P as bf16 to tensor memory and keeps the
//   sum of the bf16 P it wrote; one window later it reads its row of O, divides by that
//   sum and stores the row at the token it came from.
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
// stage: q_A k_A v_A | q_B k_B v_B (B: the wrapped part of a window that wraps at the right)
constexpr int kSTAGE = 6 * kTILE;          // 55296 bytes (54 KB)
constexpr int kSTAGES = 2;
constexpr int kOFF_BIAS = kSTAGES * kSTAGE;
constexpr int kBIAS_BYTES = kTN * kTN * 4;  // the head's dense bias, fp32
constexpr int kSTG_WARP = 32 * kROW;        // per softmax warp: its rows of Y, staged
constexpr int kOFF_STG = kOFF_BIAS + kBIAS_BYTES;
constexpr int kOFF_BAR = kOFF_STG + 5 * kSTG_WARP;
constexpr int kNBAR = 2 * kSTAGES + 7;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + alignment slack
static_assert(kSTAGE % 1024 == 0 && kOFF_BIAS % 1024 == 0 && kOFF_STG % 1024 == 0, "1024-byte aligned tiles");
static_assert(kSMEM <= 232448, "shared memory of one CTA");
// Tensor memory: S of tile A [0,144) and B [160,304), P (bf16 pairs) of A [304,376) and B
// [376,448), O of A [448,480) and B [480,512); S and O start on 32-column boundaries.
constexpr int kTMEM_COLS = 512;
constexpr int kSA = 0, kSB = 160, kPA = 304, kPB = 376, kOA = 448, kOB = 480;
// warps 0-3: softmax, tile A rows 32w..; 4: producer; 5: S products; 6: O products;
// 7: softmax, tile B rows 128-143 (lanes 16-31)
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
  float c_l2;  // hd^-0.5 * log2(e)
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
                    const __grid_constant__ CUtensorMap q_bot, const Fwd12Params p) {
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
    if (lane == 0) {
      tc::mbar_expect_tx(const_bar, kBIAS_BYTES);
      tc::bulk_copy(smem0 + kOFF_BIAS, p.bias + (size_t)h * kTN * kTN, kBIAS_BYTES, const_bar);
    }
    Cursor12 cur = first;
    for (int n = 0, st = 0; n < nwin; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
      if (n >= kSTAGES && !wwait(empty_bar(st), ((n / kSTAGES) - 1) & 1)) {
        bad = 1;
        break;
      }
      issued = n + 1;
      if (lane == 0) {
        const bool wy = wraps_y(cur), wx = wraps_x(cur);
        tc::mbar_expect_tx(full_bar(st), (wx ? 2 : 1) * 3 * kTILE);
        const int x0 = cur.wx * kTM + s, y0 = cur.wy * kTM + s;
        const uint32_t stage = smem0 + st * kSTAGE;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
          const int col = t * p.C + h * kHeadDim;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (half == 1 && !wx) continue;
            const uint32_t dst = stage + (3 * half + t) * kTILE;
            const int x = half ? x0 - W : x0;  // the wrapped half: the columns past the edge
            if (!wy) {
              tc::box_load(dst, &q_box, col, x, y0, cur.b, full_bar(st));
            } else {
              tc::box_load(dst, &q_top, col, x, y0, cur.b, full_bar(st));
              tc::box_load(dst + (kTM - s) * kTM * kROW, &q_bot, col, x, 0, cur.b, full_bar(st));
            }
          }
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
    Cursor12 cur = first;
    for (int n = 0, st = 0; n < nwin && !bad; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
      const bool wx = wraps_x(cur);
      cur.next(p.nWy, p.nWx);
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
          const uint64_t dq = tc::sdesc(stage, 16, 512, kSW64);  // q_A; k_A at +kTILE, the B halves at +3 tiles
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const uint32_t qrow = tile ? 16 * kROW : 0;  // tile B starts at query row 16
            const uint32_t d = tmem + (tile ? kSB : kSA);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              tc::mma_ss(d, tc::desc_add(dq, qrow + kk * 32), tc::desc_add(dq, kTILE + kk * 32), id_s, kk > 0);
              if (wx) {
                tc::mma_ss(d, tc::desc_add(dq, qrow + kk * 32), tc::desc_add(dq, 4 * kTILE + kk * 32), id_s, true);
                tc::mma_ss(d, tc::desc_add(dq, 3 * kTILE + qrow + kk * 32), tc::desc_add(dq, kTILE + kk * 32), id_s,
                           true);
                tc::mma_ss(d, tc::desc_add(dq, 3 * kTILE + qrow + kk * 32), tc::desc_add(dq, 4 * kTILE + kk * 32),
                           id_s, true);
              }
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
          const uint64_t dv = tc::sdesc(stage + 2 * kTILE, kTILE, 512, kSW64);  // v_A; v_B at +3 tiles
#pragma unroll
          for (int tile = 0; tile < 2; ++tile) {
            const uint32_t d = tmem + (tile ? kOB : kOA), a = tmem + (tile ? kPB : kPA);
#pragma unroll
            for (int kk = 0; kk < kTN / 16; ++kk) {  // 16 keys a step
              tc::mma_ts(d, a + kk * 8, tc::desc_add(dv, kk * 1024), id_o, kk > 0);
              if (wx) tc::mma_ts(d, a + kk * 8, tc::desc_add(dv, 3 * kTILE + kk * 1024), id_o, true);
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
  } else {
    // ==== softmax warps: 0-3 tile A rows 32w + lane; 7 tile B rows 128-143 (lanes 16-31) ====
    const bool tail = warp == kTAIL_WARP;
    const bool own = !tail || lane >= 16;  // the lane owns a query row of the window
    const int i = own ? (tail ? 128 + lane - 16 : 32 * warp + lane) : 0;
    const int ly = i / kTM, lx = i % kTM;
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t scol = tail ? kSB : kSA, pcol = tail ? kPB : kPA, ocol = tail ? kOB : kOA;
    const float4* brow = reinterpret_cast<const float4*>(smem + kOFF_BIAS + (size_t)i * kTN * 4);
    unsigned char* stg = smem + kOFF_STG + (tail ? 4 : warp) * kSTG_WARP;
    const float c_l2 = p.c_l2, mask_l2 = kMaskValue * kLog2e;
    const int th = kTM - s;  // local index from which a slot lies in the wrapped region
    if (!wwait(const_bar, 0)) bad = 1;
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
        tc::ld32_nowait(trow + scol, a0);
        tc::ld32_nowait(trow + scol + 32, a1);
        tc::ld32_nowait(trow + scol + 64, a2);
        tc::ld32_nowait(trow + scol + 96, a3);
        tc::ld16_nowait(trow + scol + 128, a4);
        tc::wait_ld_then();
        tc::dep32(a0);
        tc::dep32(a1);
        tc::dep32(a2);
        tc::dep32(a3);
        tc::dep16(a4);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free);
        float t[kTN];
#pragma unroll
        for (int q = 0; q < kTN / 4; ++q) {
          const float4 b4 = brow[q];
          const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * q + u;
            const uint32_t sj = j < 32 ? a0[j] : j < 64 ? a1[j - 32] : j < 96 ? a2[j - 64] : j < 128 ? a3[j - 96] : a4[j - 128];
            t[j] = fmaf(__uint_as_float(sj), c_l2, bb[u] * kLog2e);
          }
        }
        const bool lastrow = wraps_y(cur), lastcol = wraps_x(cur);
        if (lastrow || lastcol) {
          // the shift mask: slots of different regions of a boundary window never meet
          const bool ry = ly >= th, rx = lx >= th;
#pragma unroll
          for (int j = 0; j < kTN; ++j) {
            const bool cut = (lastrow && ((j / kTM >= th) != ry)) || (lastcol && ((j % kTM >= th) != rx));
            t[j] += cut ? mask_l2 : 0.0f;
          }
        }
        float m0 = t[0], m1 = t[1];
#pragma unroll
        for (int j = 2; j < kTN; j += 4) {
          m0 = fmax3(m0, t[j], t[j + 1]);
          m1 = fmax3(m1, t[j + 2], t[j + 3]);
        }
        const float mx = fmaxf(m0, m1);
        float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < kTN / 2; ++q) {
          const uint32_t w2 = pack_bf16(fast_exp2(t[2 * q] - mx), fast_exp2(t[2 * q + 1] - mx));
          pw[q >> 3][q & 7] = w2;
          sum2 = __fadd2_rn(sum2, make_float2(__uint_as_float(w2 << 16), __uint_as_float(w2 & 0xffff0000u)));
        }
        inv = 1.0f / (sum2.x + sum2.y);  // the rows' sums of the very bf16 P that weights V
      }
      if (n > 0) {
        // ---- window n - 1: O row / sum, stored at the token its query came from ------------
        if (!wwait(o_full, (n - 1) & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t o[32];
        tc::ld32_nowait(trow + ocol, o);
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
          if (!tail || src >= 16)
            reinterpret_cast<uint4*>(p.out + tk * p.C + h * kHeadDim)[ch] =
                *reinterpret_cast<const uint4*>(stg + swz12(src, ch));
        }
        __syncwarp();  // the staging rows are read before the next window's
      }
      if (n < nwin) {
        // ---- P to tensor memory (the last window's P V products are done) ---------------
#pragma unroll
        for (int q = 0; q < 9; ++q) tc::st_x8(trow + pcol + 8 * q, pw[q]);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full);
        inv_prev = inv;
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

// The qkv maps of `batch` images: one 12 x 12-token box, and the two row bands of a window
// that wraps at the bottom (12 - s rows, then s rows).
static cudaError_t make_qkv12_maps(const Plan& pl, const void* qkv, int batch, CUtensorMap* box, CUtensorMap* top,
                                   CUtensorMap* bot) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t row = (cuuint64_t)3 * pl.C * 2;
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
  CUtensorMap box, top, bot;
  cudaError_t e = make_qkv12_maps(pl, qkv, batch, &box, &top, &bot);
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
  p.c_l2 = kLog2e / kInvScale;
  p.wait_ns = wait_limit_ns();
  return launch_pdl(fwd12_tc_kernel, dim3(L.grid), dim3(L.threads), L.smem, st, box, top, bot, p);
}

}  // namespace swin
