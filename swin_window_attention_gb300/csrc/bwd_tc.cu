// Fused (shifted-)window attention backward on the fifth-generation tensor cores
// (tcgen05, tensor memory), 7 x 7 windows, bf16, with the bias-table gradient.
//
// The same computation as bwd.cu: the forward's logits and probabilities are recomputed
// from q and k (Baidu AIAK-Training talk, jxzklqfsx.com article 743345, section 2, fused
// WindowAttention: recompute instead of reload), and the shift, partition, reverse and
// un-roll are the addressing of the loads and stores (NVIDIA Swin talk transcript,
// uticex.com article 1598, section 2). Per window and head:
//   dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
//   dtable[idx(i,j), h] += dS_ij   (fp32 dS).
//
// A CTA owns one head and a range of windows, taken two at a time: the two windows' rows
// (49 each, padded to 64) stack into the M = 128 rows of the tensor core for S and dP, so
// tensor-memory lane r is row r of the pair. Twelve warps in three warpgroups:
// * softmax (warps 0-3, 232 registers): thread r loads row r of S and dP from tensor
//   memory, recomputes its probabilities (bias from shared memory), forms D, dS and the
//   running per-(i, j) sums of dS in registers, and writes P and dS as bf16 hi/lo pairs
//   (the lo half is the rounding residual of the hi half, so the products keep ~16 bits
//   of each);
// * epilogue (warps 4-7): thread r reads its lane of dQ, dK and dV, adds the partner
//   lane's partial sums (below) and stores its row at the token it was loaded from;
// * control (warps 8-11): S = Q K^T (+ the shift mask as a rank-4 product) and
//   dP = dO V^T as M128 N128 products; the TMA producer (7 x 7-token boxes, two row bands
//   at a bottom wrap, tile::gather4 at a right wrap), three stages deep; one thread that
//   issues the gradient products, dV, dK, dQ in that order with a commit after each kind,
//   so that the softmax warps write the next pair's P and dS as soon as each is free.
// The gradient products run per window with the hi and lo halves stacked in M: for
// dV = P^T dO the A operand is [P_hi^T ; P_lo^T] (64 keys twice, K = the window's 64
// queries), so D rows m and m + 64 are two partial sums of key m's gradient row and one
// M128 N32 K16 product does the work of both halves; the same for dK = dS^T Q and for
// dQ = dS K (A = [dS_hi ; dS_lo] in tensor memory). Window a keeps its hi halves in rows
// 0-63, window b in rows 64-127, so lane r always holds its own row's hi partial and the
// lo partial of the other window's row of the same slot; the epilogue trades the lo
// partials (~2^-8 of the row, sent as bf16) through shared memory and rounds once. In
// shared memory P and dS are, per window, four 4 KB blocks of 64 query rows x 32 keys
// (64-byte rows, 64-byte swizzled) read transposed, hi then lo for window a and lo then hi
// for window b. Hand-offs are mbarriers; every wait is bounded and a wait that runs out
// ends in the plan's error word (warps that share a named barrier leave together).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kTM = 7, kTN = 49;
constexpr int kR = (2 * kTM - 1) * (2 * kTM - 1);  // 169 table rows
constexpr int kGROUPS = (kTN + 3) / 4;              // gather4 row groups per window tile
// warps 0-3: softmax (one warpgroup), 4-7: epilogue, 8: MMA (S, dP), 9: producer,
// 10: MMA (dV, dK, dQ), 11: idle
constexpr int kA_WARP = 8, kPROD_WARP = 9, kGRAD_WARP = 10;
constexpr int kTHREADS = 12 * 32;
constexpr int kROW = 64;                     // one token's 32 bf16 head channels
constexpr int kWIN = 64 * kROW;              // 64 slot rows of one window (4 KB)
// stage: q_a q_b | k_a k_b | v_a v_b | o_a o_b (64-byte swizzled rows)
constexpr int kOFF_K = 2 * kWIN, kOFF_V = 4 * kWIN, kOFF_O = 6 * kWIN;
constexpr int kSTAGE = 8 * kWIN;             // 32 KB
constexpr int kSTAGES = 3;
// P and dS: per window four 4 KB blocks of 64 query rows x 32 keys (see the file comment)
constexpr int kBLK = 64 * kROW;
constexpr int kOP = 8 * kBLK;                // 32 KB
constexpr int kOFF_OPS = kSTAGES * kSTAGE;
// the tcgen05 forward's tables: mask U | V of classes 1..3 | the head's bias image
constexpr int kBIAS_STRIDE = 52;
constexpr int kBIAS_BYTES = 64 * kBIAS_STRIDE * 4;
constexpr int kU_BYTES = 128 * 16 * 2;
constexpr int kVC_BYTES = 64 * 16 * 2;
constexpr int kMASK_BYTES = kU_BYTES + 3 * kVC_BYTES;
constexpr int kOFF_U = kOFF_OPS + 2 * kOP;
constexpr int kOFF_VC = kOFF_U + kU_BYTES;
constexpr int kOFF_BIAS = kOFF_U + kMASK_BYTES;
// epilogue exchange and staging: dQ, dK, dV, 128 rows of 64 bytes each
constexpr int kXCH = 128 * kROW;
constexpr int kOFF_XCH = kOFF_BIAS + kBIAS_BYTES;
constexpr int kOFF_BAR = kOFF_XCH + 3 * kXCH;
constexpr int kNBAR = 2 * kSTAGES + 9;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + alignment slack
constexpr uint32_t kG4_TX = 4 * kGROUPS * 4 * kROW;     // one window's gather4 bytes, 4 tensors
constexpr uint32_t kBOX_TX = 4 * kTN * kROW;            // one window's box bytes, 4 tensors
// Tensor memory: S [0,128) (row r: keys of window a | keys of window b), dP [128,256),
// dS as the A operand of dQ [256,320) (32 columns of bf16 pairs over a window's 64 keys
// per window), then per window 32 columns each of dV [320,384), dK [384,448) and dQ
// [448,512).
constexpr int kTMEM_COLS = 512;
constexpr int kS_COL = 0, kDP_COL = 128, kDSA_COL = 256, kDV_COL = 320, kDK_COL = 384, kDQ_COL = 448;
constexpr uint32_t kSW64 = 4;

static_assert(kOFF_OPS % 1024 == 0 && kOFF_U % 1024 == 0, "swizzled tiles on 512-byte boundaries");
static_assert(kSMEM <= 232448, "shared memory of one CTA");
static_assert(kSMEM * 2 > 233472, "one CTA per SM: it holds all of the tensor memory");

struct BwdTcParams {
  __nv_bfloat16* dqkv;
  const unsigned char* tables;  // plan: U | V of classes 1..3 | bias image per head
  float* partial;               // [grid, 169] table-gradient partials
  int* err;
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;
  int chunks;
  float qk_scale_log2;  // hd^-0.5 * log2(e)
  float scale;          // hd^-0.5
  uint64_t wait_ns;
};

// Window cursor: (b, wy, wx) advanced one window at a time.
struct Cursor {
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

__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, limit_ns)) != 0;
}

// Byte offset of 16-byte chunk c of 64-byte row r in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4)); }

// Named barrier `id` over `count` threads that also returns whether any of them passed
// `pred` true.
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// hi = bf16x2(a, b), lo = bf16x2 of the residuals (a - hi_a, b - hi_b).
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  lo = pack_bf16(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}

}  // namespace

__global__ void __launch_bounds__(kTHREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap q_g4, const __grid_constant__ CUtensorMap q_box,
                  const __grid_constant__ CUtensorMap q_top, const __grid_constant__ CUtensorMap q_bot,
                  const __grid_constant__ CUtensorMap o_g4, const __grid_constant__ CUtensorMap o_box,
                  const __grid_constant__ CUtensorMap o_top, const __grid_constant__ CUtensorMap o_bot,
                  const BwdTcParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const float* sbias = reinterpret_cast<const float*>(smem + kOFF_BIAS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 8 * kNBAR);
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem0 + kOFF_BAR;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto empty_bar = [&](int st) { return bar0 + 8 * (kSTAGES + st); };
  const uint32_t sdp_full = bar0 + 8 * (2 * kSTAGES), sdp_free = sdp_full + 8, pds_full = sdp_full + 16;
  const uint32_t b_done = sdp_full + 24, acc_free = sdp_full + 32, const_bar = sdp_full + 40;
  const uint32_t drain_bar = sdp_full + 48, p_free = sdp_full + 56, ds_free = sdp_full + 64;
  auto wwait = [&](uint32_t mbar, uint32_t parity) { return warp_wait(mbar, parity, p.wait_ns); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int npair = (nwin + 1) >> 1;
  const int H = p.H, W = p.W, s = p.s;
  Cursor first;
  first.b = (int)(w_begin / p.nW);
  {
    const int w = (int)(w_begin - (int64_t)first.b * p.nW);
    first.wy = w / p.nWx;
    first.wx = w - first.wy * p.nWx;
  }

  // ---- set-up: tensor memory, barriers, zeroed operand blocks ------------------------
  if (warp == 0) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < kSTAGES; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 1);  // the gradient products' issuing thread
    }
    tc::mbar_init(sdp_full, 1);
    tc::mbar_init(sdp_free, 4);
    tc::mbar_init(pds_full, 4);
    tc::mbar_init(b_done, 1);
    tc::mbar_init(p_free, 1);
    tc::mbar_init(ds_free, 1);
    tc::mbar_init(acc_free, 4);
    tc::mbar_init(const_bar, 1);
    tc::mbar_init(drain_bar, 3);
    tc::mbar_init_fence();
  }
  // The stage tiles (rows past the loaded slots, and a pair's second window when it has
  // none, meet zero weights, so they must hold finite values) and the P / dS operand
  // blocks (the padded rows and keys stay zero) start zeroed.
  for (int e = tid; e < (kOFF_OPS + 2 * kOP) / 16; e += kTHREADS)
    reinterpret_cast<uint4*>(smem)[e] = make_uint4(0u, 0u, 0u, 0u);
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp >= 8) {
  tc::setmaxnreg_dec<128>();  // the control warpgroup: producer and MMA warps
  if (warp == kPROD_WARP) {
    // ==== producer: q, k, v and dO of pair n into stage n % kSTAGES ====================
    if (lane == 0) {
      tc::mbar_expect_tx(const_bar, kMASK_BYTES + kBIAS_BYTES);
      tc::bulk_copy(smem0 + kOFF_U, p.tables, kMASK_BYTES, const_bar);
      tc::bulk_copy(smem0 + kOFF_BIAS, p.tables + kMASK_BYTES + (size_t)h * kBIAS_BYTES, kBIAS_BYTES, const_bar);
    }
    const int g = lane & 15, w2 = lane >> 4;  // window of the pair, slot group 4g..4g+3
    int sly[4], slx[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = min(4 * g + q, kTN - 1);
      sly[q] = i / kTM;
      slx[q] = i % kTM;
    }
    const int colq = h * kHeadDim, colk = p.C + colq, colv = 2 * p.C + colq, colo = colq;
    const bool split_ok = ((kTM - s) & 1) == 0;
    auto kind = [&](const Cursor& c) {
      const bool wrap_x = c.wx * kTM + s + kTM > W, wrap_y = c.wy * kTM + s + kTM > H;
      return !wrap_x && !wrap_y ? 0 : (!wrap_x && split_ok ? 1 : 2);
    };
    Cursor cur = first;
    int issued = 0;
    for (int n = 0, st = 0; n < npair; ++n) {
      if (n >= kSTAGES && !wwait(empty_bar(st), ((n / kSTAGES) - 1) & 1)) {
        bad = 1;
        break;
      }
      issued = n + 1;
      const bool has_b = 2 * n + 1 < nwin;
      Cursor wa = cur, wb = cur;
      wb.next(p.nWy, p.nWx);
      const int k_a = kind(wa), k_b = has_b ? kind(wb) : 0;
      if (lane == 0)
        tc::mbar_expect_tx(full_bar(st), (k_a < 2 ? kBOX_TX : kG4_TX) + (has_b ? (k_b < 2 ? kBOX_TX : kG4_TX) : 0));
      __syncwarp();
      const Cursor me = w2 ? wb : wa;
      const int mk = w2 ? k_b : k_a;
      const uint32_t tile = smem0 + st * kSTAGE + w2 * kWIN;
      if (w2 == 0 || has_b) {
        if (mk < 2) {
          if (g == 0) {
            const int x = me.wx * kTM + s, y = me.wy * kTM + s;
            if (mk == 0) {
              tc::box_load(tile, &q_box, colq, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_K, &q_box, colk, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_V, &q_box, colv, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_O, &o_box, colo, x, y, me.b, full_bar(st));
            } else {
              const uint32_t bot = tile + (kTM - s) * kTM * kROW;
              tc::box_load(tile, &q_top, colq, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_K, &q_top, colk, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_V, &q_top, colv, x, y, me.b, full_bar(st));
              tc::box_load(tile + kOFF_O, &o_top, colo, x, y, me.b, full_bar(st));
              tc::box_load(bot, &q_bot, colq, x, 0, me.b, full_bar(st));
              tc::box_load(bot + kOFF_K, &q_bot, colk, x, 0, me.b, full_bar(st));
              tc::box_load(bot + kOFF_V, &q_bot, colv, x, 0, me.b, full_bar(st));
              tc::box_load(bot + kOFF_O, &o_bot, colo, x, 0, me.b, full_bar(st));
            }
          }
        } else if (g < kGROUPS) {
          int row[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            int y = me.wy * kTM + sly[q] + s, x = me.wx * kTM + slx[q] + s;
            y = y >= H ? y - H : y;
            x = x >= W ? x - W : x;
            row[q] = (me.b * H + y) * W + x;
          }
          const uint32_t base = tile + g * 4 * kROW;
          tc::gather4(base, &q_g4, colq, row[0], row[1], row[2], row[3], full_bar(st));
          tc::gather4(base + kOFF_K, &q_g4, colk, row[0], row[1], row[2], row[3], full_bar(st));
          tc::gather4(base + kOFF_V, &q_g4, colv, row[0], row[1], row[2], row[3], full_bar(st));
          tc::gather4(base + kOFF_O, &o_g4, colo, row[0], row[1], row[2], row[3], full_bar(st));
        }
      }
      cur.next(p.nWy, p.nWx);
      cur.next(p.nWy, p.nWx);
      st = st + 1 == kSTAGES ? 0 : st + 1;
    }
    // every load issued has landed before the CTA leaves, also when another role's wait
    // ran out before it consumed them
    for (int m = issued > kSTAGES ? issued - kSTAGES : 0; m < issued; ++m)
      tc::mbar_wait(full_bar(m % kSTAGES), (m / kSTAGES) & 1, p.wait_ns);
    tc::mbar_wait(const_bar, 0, p.wait_ns);
  } else {
    // ==== MMA issue: one thread per warp; the warp waits together ======================
    // S and dP of pair n (warp kA_WARP) run ahead of the gradient products of pair n - 1
    // (kDKV_WARP: dV and dK, kDQ_WARP: dQ); the tensor pipe takes them in issue order
    const uint32_t id_sq = tc::idesc_bf16(128, 128, false);
    const uint32_t id_mask = tc::idesc_bf16(128, 64, false);
    const uint32_t id_t = tc::idesc_bf16(128, 32, true, true);  // dV, dK: A and B MN-major
    const uint32_t id_q = tc::idesc_bf16(128, 32, true);        // dQ: A in tensor memory
    const uint32_t ops = smem0 + kOFF_OPS;
    auto wclass = [&](const Cursor& c) {
      return s > 0 ? ((c.wy == p.nWy - 1 ? 2 : 0) | (c.wx == p.nWx - 1 ? 1 : 0)) : 0;
    };
    if (warp == kA_WARP) {
      // S = Q K^T (+ mask) and dP = dO V^T of pair n once its tiles have landed and the
      // softmax warps have read the last pair's
      Cursor cur = first;
      const uint64_t du = tc::sdesc(smem0 + kOFF_U, 128, 256), dvc = tc::sdesc(smem0 + kOFF_VC, 128, 256);
      if (npair > 0 && !wwait(const_bar, 0)) bad = 1;
      for (int n = 0, st = 0; n < npair && !bad; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
        if (!wwait(full_bar(st), (n / kSTAGES) & 1) || (n > 0 && !wwait(sdp_free, (n - 1) & 1))) {
          bad = 1;
          break;
        }
        const int cls_a = wclass(cur);
        cur.next(p.nWy, p.nWx);
        const bool has_b = 2 * n + 1 < nwin;
        const int cls_b = has_b ? wclass(cur) : 0;
        cur.next(p.nWy, p.nWx);
        if (lane == 0) {
          tc::fence_after_sync();
          // descriptors as offsets from the stage's K-major one (addresses stay below 256 KB)
          const uint64_t d = tc::sdesc(smem0 + st * kSTAGE, 16, 512, kSW64);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            tc::mma_ss(tmem + kS_COL, tc::desc_add(d, kk * 32), tc::desc_add(d, kOFF_K + kk * 32), id_sq, kk > 0);
          if (cls_a) tc::mma_ss(tmem + kS_COL, du, tc::desc_add(dvc, (cls_a - 1) * kVC_BYTES), id_mask, true);
          if (cls_b) tc::mma_ss(tmem + kS_COL + 64, du, tc::desc_add(dvc, (cls_b - 1) * kVC_BYTES), id_mask, true);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            tc::mma_ss(tmem + kDP_COL, tc::desc_add(d, kOFF_O + kk * 32), tc::desc_add(d, kOFF_V + kk * 32), id_sq,
                       kk > 0);
          tc::commit(sdp_full);
        }
        __syncwarp();
      }
    } else if (warp == kGRAD_WARP) {
      // Per window: dV = P^T dO and dK = dS^T Q (A transposed from the shared operand
      // blocks), dQ = dS K (A from tensor memory), once the pair's P and dS are written and
      // the last pair's gradients have been read out. The A rows are the window's 64 rows
      // twice, hi halves and lo halves, so D row m and row m + 64 are two partial sums of
      // one gradient row. Issued in that order, with a commit after each kind, so that the
      // softmax warps may write the next pair's P once the dV products are done, its dS
      // once the dK products are.
      const uint64_t dops = tc::sdesc(ops, kBLK, 512, kSW64);
      for (int n = 0, st = 0; n < npair && !bad; ++n, st = st + 1 == kSTAGES ? 0 : st + 1) {
        if (!wwait(pds_full, n & 1) || (n > 0 && !wwait(acc_free, (n - 1) & 1))) {
          bad = 1;
          break;
        }
        if (lane == 0) {
          tc::fence_after_sync();
          // descriptors as offsets from the stage's MN-major one (addresses below 256 KB)
          const uint64_t d = tc::sdesc(smem0 + st * kSTAGE, kWIN, 512, kSW64);
#pragma unroll
          for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // the window's queries
              tc::mma_ss(tmem + kDV_COL + 32 * w, tc::desc_add(dops, w * 4 * kBLK + kk * 1024),
                         tc::desc_add(d, kOFF_O + (4 * w + kk) * 1024), id_t, kk > 0);
          tc::commit(p_free);
#pragma unroll
          for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // the window's queries
              tc::mma_ss(tmem + kDK_COL + 32 * w, tc::desc_add(dops, kOP + w * 4 * kBLK + kk * 1024),
                         tc::desc_add(d, (4 * w + kk) * 1024), id_t, kk > 0);
          tc::commit(ds_free);
#pragma unroll
          for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // the window's keys
              tc::mma_ts(tmem + kDQ_COL + 32 * w, tmem + kDSA_COL + 32 * w + kk * 8,
                         tc::desc_add(d, kOFF_K + (4 * w + kk) * 1024), id_q, kk > 0);
          tc::commit(b_done);
          tc::commit(empty_bar(st));
        }
        __syncwarp();
      }
    }
    // every MMA this thread issued has completed before the tensor memory is released
    if (lane == 0) tc::commit(drain_bar);
    __syncwarp();
    if (!wwait(drain_bar, 0)) bad = 1;
  }
  } else if (warp < 4) {
    // ==== softmax warps: thread r = row r of the pair (window w, slot i) ===============
    tc::setmaxnreg_inc<232>();
    const int w = tid >> 6, i = tid & 63;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    const float c_l2 = p.qk_scale_log2;
    const float* brow = sbias + i * kBIAS_STRIDE;
    unsigned char* ops = smem + kOFF_OPS;
    // the row's 64-byte rows in its window's operand blocks: hi halves in blocks 0-1 of
    // window a and 2-3 of window b, lo halves in the other two (keys 0-31, 32-63)
    const uint32_t hi_blk = (uint32_t)(4 * w + 2 * w) * kBLK, lo_blk = (uint32_t)(4 * w + 2 - 2 * w) * kBLK;
    // the other window's lo rows of dS, which this thread's lane holds in the dQ A operand
    const uint32_t oth_lo = (uint32_t)(4 - 2 * w) * kBLK;
    float dt[kTN];  // running sums of dS_ij over the CTA's windows (j = 0..48)
#pragma unroll
    for (int j = 0; j < kTN; ++j) dt[j] = 0.0f;

    // A wait that runs out marks the warp; the four warps leave the loop together at the
    // pair's named barrier, so that no warp is left waiting at a barrier.
    if (npair > 0 && !wwait(const_bar, 0)) bad = 1;
    for (int n = 0; n < npair; ++n) {
      const bool active = i < kTN && (w == 0 || 2 * n + 1 < nwin);

      // ---- S and dP rows of this pair ----------------------------------------------
      if (!bad && !wwait(sdp_full, n & 1)) bad = 1;
      tc::fence_after_sync();
      uint32_t sa[32], sb[16], sc1, pa[32], pb[16], pc1;
      {
        const uint32_t ts = trow + kS_COL + 64 * w, tp = trow + kDP_COL + 64 * w;
        tc::ld32_nowait(ts, sa);
        tc::ld16_nowait(ts + 32, sb);
        tc::ld1_nowait(ts + 48, sc1);
        tc::ld32_nowait(tp, pa);
        tc::ld16_nowait(tp + 32, pb);
        tc::ld1_nowait(tp + 48, pc1);
        tc::wait_ld_then();
        tc::dep32(sa);
        tc::dep16(sb);
        tc::dep1(sc1);
        tc::dep32(pa);
        tc::dep16(pb);
        tc::dep1(pc1);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sdp_free);

      // ---- P = softmax(scale q.k + bias + mask), D, dS -------------------------------
      float pr[kTN], dp[kTN];
#pragma unroll
      for (int j = 0; j < kTN; ++j) {
        pr[j] = __uint_as_float(j < 32 ? sa[j] : (j < 48 ? sb[j - 32] : sc1));
        dp[j] = __uint_as_float(j < 32 ? pa[j] : (j < 48 ? pb[j - 32] : pc1));
      }
      {
        const float4* b4 = reinterpret_cast<const float4*>(brow);
        const float2 c2 = make_float2(c_l2, c_l2);
#pragma unroll
        for (int q = 0; q < 12; ++q) {
          const float4 bb = b4[q];
          const float2 e0 = __ffma2_rn(make_float2(pr[4 * q], pr[4 * q + 1]), c2, make_float2(bb.x, bb.y));
          const float2 e1 = __ffma2_rn(make_float2(pr[4 * q + 2], pr[4 * q + 3]), c2, make_float2(bb.z, bb.w));
          pr[4 * q] = e0.x, pr[4 * q + 1] = e0.y, pr[4 * q + 2] = e1.x, pr[4 * q + 3] = e1.y;
        }
        pr[48] = fmaf(pr[48], c_l2, brow[48]);
      }
      float ma = pr[48], mb = pr[47];
#pragma unroll
      for (int q = 0; q < 46; q += 4) {
        ma = fmax3(ma, pr[q], pr[q + 1]);
        mb = fmax3(mb, pr[q + 2], pr[q + 3]);
      }
      ma = fmax3(ma, mb, pr[46]);
      float2 l2 = make_float2(0.0f, 0.0f);
      {
        const float2 nm = make_float2(-ma, -ma);
#pragma unroll
        for (int q = 0; q < 24; ++q) {
          const float2 d = __fadd2_rn(make_float2(pr[2 * q], pr[2 * q + 1]), nm);
          pr[2 * q] = fast_exp2(d.x);
          pr[2 * q + 1] = fast_exp2(d.y);
          l2 = __fadd2_rn(l2, make_float2(pr[2 * q], pr[2 * q + 1]));
        }
        pr[48] = fast_exp2(pr[48] - ma);
      }
      const float inv = active ? 1.0f / (l2.x + l2.y + pr[48]) : 0.0f;  // inactive rows: P = 0
      float2 D2 = make_float2(0.0f, 0.0f);
      {
        const float2 i2 = make_float2(inv, inv);
#pragma unroll
        for (int q = 0; q < 24; ++q) {
          const float2 v = __fmul2_rn(make_float2(pr[2 * q], pr[2 * q + 1]), i2);
          pr[2 * q] = v.x, pr[2 * q + 1] = v.y;
          D2 = __ffma2_rn(v, make_float2(dp[2 * q], dp[2 * q + 1]), D2);
        }
        pr[48] *= inv;
      }
      const float Dr = D2.x + D2.y + pr[48] * dp[48];
      // dS = P (dP - D) into dp; running sums
      {
        const float2 nD = make_float2(-Dr, -Dr);
#pragma unroll
        for (int q = 0; q < 24; ++q) {
          const float2 v = __fmul2_rn(make_float2(pr[2 * q], pr[2 * q + 1]),
                                      __fadd2_rn(make_float2(dp[2 * q], dp[2 * q + 1]), nD));
          dp[2 * q] = v.x, dp[2 * q + 1] = v.y;
          const float2 t2 = __fadd2_rn(make_float2(dt[2 * q], dt[2 * q + 1]), v);
          dt[2 * q] = t2.x, dt[2 * q + 1] = t2.y;
        }
        dp[48] = pr[48] * (dp[48] - Dr);
        dt[48] += dp[48];
      }
      // P and dS as bf16 hi/lo, keys 8c..8c+7 of each 16-byte chunk (keys >= 49 zero)
      uint32_t ph[28], pl[28], sh[32], sl[32];
#pragma unroll
      for (int q = 0; q < 24; ++q) {
        split2(pr[2 * q], pr[2 * q + 1], ph[q], pl[q]);
        split2(dp[2 * q], dp[2 * q + 1], sh[q], sl[q]);
      }
      split2(pr[48], 0.0f, ph[24], pl[24]);
      split2(dp[48], 0.0f, sh[24], sl[24]);
#pragma unroll
      for (int q = 25; q < 28; ++q) ph[q] = pl[q] = 0u;
#pragma unroll
      for (int q = 25; q < 32; ++q) sh[q] = sl[q] = 0u;

      // ---- the last pair's gradient products are done: write this pair's operands -----
      // (rows past the window's 49 slots and keys 56-63 are never written: they keep the
      // zeros of the set-up); P once the last pair's dV products are done, dS once its dK
      // products are, the tensor-memory rows once all its products are
      const uint32_t* mats[4] = {ph, pl, sh, sl};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (m == 0 && !bad && n > 0 && !wwait(p_free, (n - 1) & 1)) bad = 1;
        if (m == 2 && !bad && n > 0 && !wwait(ds_free, (n - 1) & 1)) bad = 1;
        if (i < kTN) {
          unsigned char* dst = ops + (m >> 1) * kOP + ((m & 1) ? lo_blk : hi_blk);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
#pragma unroll
            for (int c = 0; c < (a ? 3 : 4); ++c) {
              const int q = 16 * a + 4 * c;  // words 4c.. of key atom a: keys 32a + 8c ..
              *reinterpret_cast<uint4*>(dst + a * kBLK + swz(i, c)) =
                  make_uint4(mats[m][q], mats[m][q + 1], mats[m][q + 2], mats[m][q + 3]);
            }
          }
        }
      }
      // dQ's A operand: lane r holds its own window's dS hi row and the other window's dS lo
      // row of the same slot (written by the thread 64 lanes away)
      if (!bad && n > 0 && !wwait(b_done, (n - 1) & 1)) bad = 1;
      tc::st_x32(trow + kDSA_COL + 32 * w, sh);
      if (bar_or(1, 128, bad)) {
        bad = 1;
        break;
      }
      {
        uint32_t o[32];
        const unsigned char* src = ops + kOP + oth_lo;
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + a * kBLK + swz(i, c));
            o[16 * a + 4 * c] = v.x, o[16 * a + 4 * c + 1] = v.y, o[16 * a + 4 * c + 2] = v.z, o[16 * a + 4 * c + 3] = v.w;
          }
        tc::st_x32(trow + kDSA_COL + 32 * (1 - w), o);
      }
      tc::wait_st();
      tc::fence_proxy_async();  // the operand rows to the tensor core's reads
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(pds_full);
    }
    // all products have completed, so the operand blocks are free
    if (!bad && npair > 0 && !wwait(b_done, (npair - 1) & 1)) bad = 1;

    // ---- fold the per-(i, j) dS sums into this CTA's table-gradient partial ----------
    // Window a's threads store their rows, window b's add theirs to the same slot's row;
    // then table entry (dy, dx) sums row si, column si - (7 dy + dx) over the slots si
    // whose partner lies in the window.
    float* sdt = reinterpret_cast<float*>(ops);  // [64][49]
    if (w == 0) {
#pragma unroll
      for (int j = 0; j < kTN; ++j) sdt[i * kTN + j] = i < kTN ? dt[j] : 0.0f;
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    if (w == 1 && i < kTN) {
#pragma unroll
      for (int j = 0; j < kTN; ++j) sdt[i * kTN + j] += dt[j];
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    for (int rr = tid; rr < kR; rr += 128) {
      const int dy = rr / (2 * kTM - 1) - (kTM - 1), dx = rr % (2 * kTM - 1) - (kTM - 1);
      const int y0 = max(0, dy), y1 = min(kTM, kTM + dy), x0 = max(0, dx), x1 = min(kTM, kTM + dx);
      const int off = dy * kTM + dx;
      float acc0 = 0.0f, acc1 = 0.0f;
      for (int yi = y0; yi < y1; ++yi) {
        const float* rowp = sdt + (yi * kTM) * (kTN + 1) - off;  // element (si, si - off) at si * 50 - off
        int xi = x0;
        for (; xi + 1 < x1; xi += 2) {
          acc0 += rowp[xi * (kTN + 1)];
          acc1 += rowp[(xi + 1) * (kTN + 1)];
        }
        if (xi < x1) acc0 += rowp[xi * (kTN + 1)];
      }
      const float acc = acc0 + acc1;
      p.partial[(int64_t)blockIdx.x * kR + rr] = acc;
    }
  } else {
    // ==== epilogue warps: thread r = row r of the pair (lane quadrant warp % 4) =========
    // Lane r holds, per gradient, its own window's hi partial sum of row r and the other
    // window's lo partial sum of the same slot. The lo partials go (as bf16: they are
    // ~2^-8 of the row) to the thread 64 lanes away through shared memory; each thread
    // adds its partner's to its own in fp32, rounds once and stores its row.
    tc::setmaxnreg_dec<136>();
    const int r = tid - 128, w = r >> 6, i = r & 63;
    const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    unsigned char* xch = smem + kOFF_XCH;
    const int cols[3] = {kDQ_COL, kDK_COL, kDV_COL};
    Cursor cur = first;
    for (int n = 0; n < npair; ++n) {
      Cursor c = cur;
      if (w) c.next(p.nWy, p.nWx);
      const bool active = i < kTN && (w == 0 || 2 * n + 1 < nwin);
      if (!bad && !wwait(b_done, n & 1)) bad = 1;
      tc::fence_after_sync();
      // the other window's partials, scaled and packed, to the partner's rows
#pragma unroll
      for (int t3 = 0; t3 < 3; ++t3) {
        uint32_t x[32];
        tc::ld32_nowait(trow + cols[t3] + 32 * (1 - w), x);
        tc::wait_ld_then();
        tc::dep32(x);
        const float m = t3 < 2 ? p.scale : 1.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w4[u] = pack_bf16(__uint_as_float(x[8 * q + 2 * u]) * m, __uint_as_float(x[8 * q + 2 * u + 1]) * m);
          *reinterpret_cast<uint4*>(xch + t3 * kXCH + swz(r ^ 64, q)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      uint32_t own[3][32];
#pragma unroll
      for (int t3 = 0; t3 < 3; ++t3) tc::ld32_nowait(trow + cols[t3] + 32 * w, own[t3]);
      tc::wait_ld_then();
#pragma unroll
      for (int t3 = 0; t3 < 3; ++t3) tc::dep32(own[t3]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_free);
      if (bar_or(2, 128, bad)) {
        bad = 1;
        break;
      }
      // own + partner, one rounding, into the thread's own row
#pragma unroll
      for (int t3 = 0; t3 < 3; ++t3) {
        const float m = t3 < 2 ? p.scale : 1.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4* row = reinterpret_cast<uint4*>(xch + t3 * kXCH + swz(r, q));
          const uint4 pv = *row;
          const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w4[u] = pack_bf16(fmaf(__uint_as_float(own[t3][8 * q + 2 * u]), m, __uint_as_float(pw[u] << 16)),
                              fmaf(__uint_as_float(own[t3][8 * q + 2 * u + 1]), m, __uint_as_float(pw[u] & 0xffff0000u)));
          *row = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      int yy = c.wy * kTM + i / kTM + s, xx = c.wx * kTM + i % kTM + s;
      yy = yy >= H ? yy - H : yy;
      xx = xx >= W ? xx - W : xx;
      const long long tok = ((long long)c.b * H + yy) * W + xx;
      __syncwarp();
      // the warp's 32 rows, four lanes to a 64-byte row (eight rows per store instruction)
      const int rl = lane >> 2, ch = lane & 3;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int src = rl + 8 * k;
        const long long tk = __shfl_sync(0xffffffffu, tok, src);
        const bool act = __shfl_sync(0xffffffffu, active ? 1 : 0, src) != 0;
        if (act) {
          uint4* dst = reinterpret_cast<uint4*>(p.dqkv + tk * 3 * p.C + h * kHeadDim) + ch;
#pragma unroll
          for (int t3 = 0; t3 < 3; ++t3)
            dst[t3 * (p.C / 8)] = *reinterpret_cast<const uint4*>(xch + t3 * kXCH + swz(32 * (warp & 3) + src, ch));
        }
      }
      // every row has been stored before the next pair's partials are written
      asm volatile("bar.sync 2, 128;\n" ::: "memory");
      cur.next(p.nWy, p.nWx);
      cur.next(p.nWy, p.nWx);
    }
  }
  if (bad) atomicOr(p.err, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

// ---- host side ---------------------------------------------------------------------

cudaError_t launch_dtable_reduce(const float* partial, int R, int nH, int chunks, float* dtable, cudaStream_t st);

// 7 x 7 windows with bf16 activations, tokens addressed by 32-bit tensor-map rows.
bool bwd_tc_applies(const Plan& pl) {
  return pl.M == kTM && pl.dtype == SWIN_WATTN_BF16 && (int64_t)pl.B * pl.H * pl.W < ((int64_t)1 << 31);
}

// One CTA of twelve warps per SM (it holds all of the tensor memory), one wave.
cudaError_t bwd_tc_config(const Plan& pl, BwdLaunch* L) {
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bwd_tc_kernel, kTHREADS, kSMEM);
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
  L->partial_rows = L->grid;
  L->tc = true;
  return cudaSuccess;
}

cudaError_t bwd_tc_launch(const Plan& pl, const BwdLaunch& L, const void* qkv, const void* dout, void* dqkv,
                          float* dtable, cudaStream_t st) {
  CUtensorMap qm[4], om[4];
  cudaError_t e = make_act_maps(pl, qkv, pl.B, 3 * pl.C, &qm[0], &qm[1], &qm[2], &qm[3]);
  if (e == cudaSuccess) e = make_act_maps(pl, dout, pl.B, pl.C, &om[0], &om[1], &om[2], &om[3]);
  if (e != cudaSuccess) return e;
  BwdTcParams p;
  p.dqkv = reinterpret_cast<__nv_bfloat16*>(dqkv);
  p.tables = pl.tc_tables;
  p.partial = pl.dt_partial;
  p.err = pl.err;
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
  p.qk_scale_log2 = kLog2e / kInvScale;
  p.scale = 1.0f / kInvScale;
  p.wait_ns = wait_limit_ns();
  e = launch_pdl(bwd_tc_kernel, dim3(L.grid), dim3(L.threads), L.smem, st, qm[0], qm[1], qm[2], qm[3], om[0], om[1],
                 om[2], om[3], p);
  if (e != cudaSuccess) return e;
  return launch_dtable_reduce(pl.dt_partial, kR, pl.nH, L.chunks, dtable, st);
}

}  // namespace swin
