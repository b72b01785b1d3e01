// Fused (shifted-)window attention forward on the fifth-generation tensor cores
// (tcgen05 + tensor memory, TMA gathers) for 7x7 windows and bf16 tensors.
//
// The same single fused pass as the mma.sync kernel (roll, partition, Q K^T, bias, mask,
// softmax, P V, reverse and un-roll in one kernel: NVIDIA Swin talk transcript, uticex.com
// article 1598, sections 2 and 3; Baidu AIAK-Training talk, jxzklqfsx.com article 743345,
// section 2), laid out for tcgen05 and split over specialised warps:
//
// * A CTA owns one head and a range of windows, taken two at a time (a pair). The two
//   windows' query rows, each padded from 49 to 64, stack into M = 128: lane r of tensor
//   memory holds query row r.
// * The producer warp (5) brings the pair's q/k/v head slices with TMA: a window that
//   does not wrap around the image border is one 7 x 7-token box per tensor (the rolled
//   window is a plain rectangle of the unrolled image), one that wraps at the bottom only
//   is two row bands; the last window column of a shifted layer goes by tile::gather4
//   loads, each fetching the 64-byte head slice of four arbitrary tokens, so the wrap is
//   nothing but the token indices handed to the copy engine. The copies land in 64-byte-swizzled tiles that the tensor core reads as
//   they are, three pairs ahead, and complete on the stage's mbarrier.
// * The MMA warp (4) issues, from one thread: S = Q K^T as two M128 N128 K16 MMAs (both
//   windows' keys side by side; the off-diagonal blocks are never read), one M128 N64 K16
//   MMA per boundary window that adds the shift mask (the rank-4 product of a one-hot
//   region matrix U and a per-class matrix V), then O = P V as four M128 N80 K16 MMAs
//   whose B operand is [v of window a | v of window b | a ones column]: row r's output
//   sits in columns 32 * window .. + 31 and its row sum (of the very bf16 P that weighted
//   V) in column 64.
// * Row warps (0..3): thread r loads its 49 logits from tensor memory, adds the relative
//   position bias, takes max and exp2, writes the bf16 row of P to tensor memory (the A
//   operand of P V); one pair later (its P V ran meanwhile) it normalises its row of O and
//   stores it at the token the row was read from. The MMA thread issues the next pair's
//   Q K^T as soon as S has been read out, ahead of the current pair's P V.
//
// The bias image of the CTA's head and the mask operands are built once per plan and
// arrive with one bulk copy. Hand-offs go through mbarriers (stage full / empty, S full /
// free, P full, O full / free), so the gathers, the tensor core and the softmax of
// consecutive pairs overlap. Every wait is bounded (1 s): a role whose wait runs out sets
// the plan's error word and stops; the others then run out in turn, and the CTA releases
// its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kTM = 7, kTN = 49;
constexpr int kGROUPS = (kTN + 3) / 4;         // gather4 row groups per window tile (13)
constexpr int kMMA_WARP = 4, kPROD_WARP = 5;
constexpr int kTHREADS = 6 * 32;
constexpr int kROW_BYTES = 64;                 // one token's 32 bf16 head channels
constexpr int kWIN_TILE = 64 * kROW_BYTES;     // 64 slot rows of one window (4 KB)
// stage: q_a q_b | k_a k_b | v_a v_b ones (64-byte swizzled rows; ones is constant)
constexpr int kOFF_K = 2 * kWIN_TILE;
constexpr int kOFF_V = 4 * kWIN_TILE;
constexpr int kSTAGE = 7 * kWIN_TILE;          // 28672 B
constexpr int kSTAGES = 3;
constexpr int kBIAS_STRIDE = 52;               // floats per bias row (13 x 16 B)
constexpr int kBIAS_BYTES = 64 * kBIAS_STRIDE * 4;
constexpr int kU_BYTES = 128 * 16 * 2;         // U: 128 rows x K16 (core-matrix layout)
constexpr int kVC_BYTES = 64 * 16 * 2;         // V of one boundary class: 64 keys x K16
constexpr int kMASK_BYTES = kU_BYTES + 3 * kVC_BYTES;
constexpr int kOFF_U = kSTAGES * kSTAGE;
constexpr int kOFF_VC = kOFF_U + kU_BYTES;
constexpr int kOFF_BIAS = kOFF_U + kMASK_BYTES;
constexpr int kOFF_BAR = kOFF_BIAS + kBIAS_BYTES;
constexpr int kNBAR = 2 * kSTAGES + 7;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + alignment slack
constexpr uint32_t kG4_TX = 3 * kGROUPS * 4 * kROW_BYTES;  // bytes of one window's gather4 loads
constexpr uint32_t kBOX_TX = 3 * kTN * kROW_BYTES;           // bytes of one window's box loads
// Tensor memory: S [0, 128) (keys of window a, keys of window b), P [128, 160) (bf16
// pairs over the row's own 64 keys), O [160, 240) (window a, window b, row sums).
constexpr int kTMEM_COLS = 256;
constexpr int kS_COL = 0, kP_COL = 128, kO_COL = 160;
constexpr uint32_t kSW64 = 4;                  // descriptor layout: 64-byte swizzle

static_assert(kSMEM * 3 > 233472, "at most two CTAs per SM: each holds half the tensor memory");
static_assert(kOFF_U % 1024 == 0 && kSTAGE % 1024 == 0, "swizzled tiles stay 512-byte aligned");

// Byte offset of bf16 element (r, k) in a K16 tile (U, or a class V), core-matrix layout.
__device__ __forceinline__ uint32_t k16_off(int r, int k) {
  return (r >> 3) * 256 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

// A bounded wait whose outcome is the same for the whole warp.
__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, limit_ns)) != 0;
}

struct TcParams {
  __nv_bfloat16* out;
  const unsigned char* tables;  // plan: U | V of classes 1..3 | bias image per head
  int* err;                     // plan error word (bit 0: a wait ran out)
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;
  int chunks;
  float qk_scale_log2;  // hd^-0.5 * log2(e)
  uint64_t wait_ns;     // bound of each wait
  int fault;            // armed fault site (fault-injection build only)
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

__global__ void __launch_bounds__(kTHREADS, 1) fwd_tc_kernel(const __grid_constant__ CUtensorMap qkv_map,
                                                              const __grid_constant__ CUtensorMap box_map,
                                                              const __grid_constant__ CUtensorMap top_map,
                                                              const __grid_constant__ CUtensorMap bot_map,
                                                              const TcParams p) {
  // The 64-byte swizzle is a function of the shared-memory address: tiles sit on
  // 1024-byte boundaries of the address space (the launch adds the slack).
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const float* sbias = reinterpret_cast<const float*>(smem + kOFF_BIAS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 8 * kNBAR);
  // The next kernel may be scheduled now; everything this one reads (activations, and the
  // plan's tables, which the previous kernel may just have rebuilt) waits for the previous
  // kernel to complete.
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem0 + kOFF_BAR;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto empty_bar = [&](int st) { return bar0 + 8 * (kSTAGES + st); };
  const uint32_t s_full = bar0 + 8 * (2 * kSTAGES), s_free = s_full + 8, p_full = s_full + 16;
  const uint32_t o_full = s_full + 24, o_free = s_full + 32, const_bar = s_full + 40;
  const uint32_t drain_bar = s_full + 48;  // the MMA thread's last commit before it leaves
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

  // ---- set-up: tensor memory, barriers, constant shared data ------------------------
  if (warp == 0) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < kSTAGES; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_free, 4);
    tc::mbar_init(p_full, 4);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(o_free, 4);
    tc::mbar_init(const_bar, 1);
    tc::mbar_init(drain_bar, 1);
    tc::mbar_init_fence();
  }
  // Stage tiles start zeroed: slot rows 52..63 are never written by the gathers. The
  // ones tile of every stage holds 1.0 in column 0 of each (swizzled) key row.
  for (int e = tid; e < kSTAGES * kSTAGE / 16; e += kTHREADS) {
    const int st = e / (kSTAGE / 16), off = (e % (kSTAGE / 16)) * 16;
    const int r = (off - (kOFF_V + 2 * kWIN_TILE)) / kROW_BYTES;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (off >= kOFF_V + 2 * kWIN_TILE && ((off >> 4) & 3) == ((r >> 1) & 3)) v.x = 0x3F80u;
    *reinterpret_cast<uint4*>(smem + st * kSTAGE + off) = v;
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp == kPROD_WARP) {
    // ==== producer: TMA gathers of pair n into stage n % kSTAGES =======================
    if (lane == 0) {
      // this plan's mask operands and this head's bias image
      tc::mbar_expect_tx(const_bar, kMASK_BYTES + kBIAS_BYTES);
      tc::bulk_copy(smem0 + kOFF_U, p.tables, kMASK_BYTES, const_bar);
      tc::bulk_copy(smem0 + kOFF_BIAS, p.tables + kMASK_BYTES + (size_t)h * kBIAS_BYTES, kBIAS_BYTES, const_bar);
    }
    // lane: window (lane >> 4) of the pair, slot group g = lane & 15 (slots 4g..4g+3)
    const int g = lane & 15, w2 = lane >> 4;
    int sly[4], slx[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = min(4 * g + q, kTN - 1);  // slots past 48 repeat slot 48 (padding rows)
      sly[q] = i / kTM;
      slx[q] = i % kTM;
    }
    const int colq = h * kHeadDim, colk = p.C + colq, colv = 2 * p.C + colq;
    Cursor cur = first;
    // How a window's tiles are fetched: 0, one 7 x 7 box per tensor (the window does not
    // wrap around the image border); 1, two boxes, rows [0, 7 - s) and [7 - s, 7) (it
    // wraps at the bottom border only and the second box starts on a 128-byte boundary);
    // 2, gather4 loads (it wraps at the right border).
    const bool split_ok = ((kTM - s) & 1) == 0;
    auto kind = [&](const Cursor& c) {
      const bool wrap_x = c.wx * kTM + s + kTM > W, wrap_y = c.wy * kTM + s + kTM > H;
      return !wrap_x && !wrap_y ? 0 : (!wrap_x && split_ok ? 1 : 2);
    };
    int issued = 0;  // pairs whose loads were issued
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
      const uint32_t tile = smem0 + st * kSTAGE + w2 * kWIN_TILE;
      if (w2 == 0 || has_b) {
        if (mk == 0) {
          if (g == 0) {
            const int x = me.wx * kTM + s, y = me.wy * kTM + s;
            tc::box_load(tile, &box_map, colq, x, y, me.b, full_bar(st));
            tc::box_load(tile + kOFF_K, &box_map, colk, x, y, me.b, full_bar(st));
            tc::box_load(tile + kOFF_V, &box_map, colv, x, y, me.b, full_bar(st));
          }
        } else if (mk == 1) {
          if (g == 0) {
            const int x = me.wx * kTM + s, y = me.wy * kTM + s;
            const uint32_t bot = tile + (kTM - s) * kTM * kROW_BYTES;
            tc::box_load(tile, &top_map, colq, x, y, me.b, full_bar(st));
            tc::box_load(tile + kOFF_K, &top_map, colk, x, y, me.b, full_bar(st));
            tc::box_load(tile + kOFF_V, &top_map, colv, x, y, me.b, full_bar(st));
            tc::box_load(bot, &bot_map, colq, x, 0, me.b, full_bar(st));
            tc::box_load(bot + kOFF_K, &bot_map, colk, x, 0, me.b, full_bar(st));
            tc::box_load(bot + kOFF_V, &bot_map, colv, x, 0, me.b, full_bar(st));
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
          const uint32_t base = tile + g * 4 * kROW_BYTES;
          tc::gather4(base, &qkv_map, colq, row[0], row[1], row[2], row[3], full_bar(st));
          tc::gather4(base + kOFF_K, &qkv_map, colk, row[0], row[1], row[2], row[3], full_bar(st));
          tc::gather4(base + kOFF_V, &qkv_map, colv, row[0], row[1], row[2], row[3], full_bar(st));
        }
      }
      cur.next(p.nWy, p.nWx);
      cur.next(p.nWy, p.nWx);
      st = st + 1 == kSTAGES ? 0 : st + 1;
    }
    // every load issued has landed before the CTA leaves, also when another role's wait
    // ran out before it consumed them (the latest phase of each stage completes with its
    // bytes; older phases have completed)
    for (int m = issued > kSTAGES ? issued - kSTAGES : 0; m < issued; ++m)
      tc::mbar_wait(full_bar(m % kSTAGES), (m / kSTAGES) & 1, p.wait_ns);
    tc::mbar_wait(const_bar, 0, p.wait_ns);  // and the constant operands
  } else if (warp == kMMA_WARP) {
    // ==== MMA issue: one thread; the warp waits together ==============================
    const uint32_t idesc_qk = tc::idesc_bf16(128, 128, false);
    const uint32_t idesc_mask = tc::idesc_bf16(128, 64, false);
    const uint32_t idesc_pv = tc::idesc_bf16(128, 80, true);
    Cursor cur = first;  // first window of the next pair whose Q K^T is issued
    auto wclass = [&](const Cursor& c) {
      return s > 0 ? ((c.wy == p.nWy - 1 ? 2 : 0) | (c.wx == p.nWx - 1 ? 1 : 0)) : 0;
    };
    auto issue_qk = [&](int n) {
      const int st = n % kSTAGES;
      const int cls_a = wclass(cur);
      cur.next(p.nWy, p.nWx);
      const bool has_b = 2 * n + 1 < nwin;
      const int cls_b = has_b ? wclass(cur) : 0;
      if (has_b) cur.next(p.nWy, p.nWx);
      if (lane == 0) {
        tc::fence_after_sync();
        const uint32_t base = smem0 + st * kSTAGE;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          tc::mma_ss(tmem + kS_COL, tc::sdesc(base + kk * 32, 16, 512, kSW64),
                     tc::sdesc(base + kOFF_K + kk * 32, 16, 512, kSW64), idesc_qk, kk > 0);
        if (cls_a)
          tc::mma_ss(tmem + kS_COL, tc::sdesc(smem0 + kOFF_U, 128, 256),
                     tc::sdesc(smem0 + kOFF_VC + (cls_a - 1) * kVC_BYTES, 128, 256), idesc_mask, true);
        if (cls_b)
          tc::mma_ss(tmem + kS_COL + 64, tc::sdesc(smem0 + kOFF_U, 128, 256),
                     tc::sdesc(smem0 + kOFF_VC + (cls_b - 1) * kVC_BYTES, 128, 256), idesc_mask, true);
        tc::commit(s_full);
      }
      __syncwarp();
    };
    if (npair > 0) {
      if (wwait(const_bar, 0) && wwait(full_bar(0), 0))
        issue_qk(0);
      else
        bad = 1;
    }
    // Q K^T of pair n + 1 as soon as its tiles have landed and the row warps have read S
    // of pair n out (early in their softmax of pair n), then P V of pair n once its P is
    // written and O of pair n - 1 has been read out: the row warps find S of the next pair
    // ready, and P V runs while they work on the next pair.
    for (int n = 0; n < npair && !bad; ++n) {
      if (n + 1 < npair) {
        const int st1 = (n + 1) % kSTAGES;
        if (!wwait(full_bar(st1), ((n + 1) / kSTAGES) & 1) || !wwait(s_free, n & 1)) {
          bad = 1;
          break;
        }
        issue_qk(n + 1);
      }
      if (!wwait(p_full, n & 1) || (n > 0 && !wwait(o_free, (n - 1) & 1))) {
        bad = 1;
        break;
      }
      if (lane == 0) {
        tc::fence_after_sync();
        const uint32_t vbase = smem0 + (n % kSTAGES) * kSTAGE + kOFF_V;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_ts(tmem + kO_COL, tmem + kP_COL + 8 * kk,
                     tc::sdesc(vbase + kk * 2 * 8 * kROW_BYTES, kWIN_TILE, 8 * kROW_BYTES, kSW64), idesc_pv, kk > 0);
        tc::commit(o_full);
        tc::commit(empty_bar(n % kSTAGES));
      }
      __syncwarp();
    }
    // every MMA this thread issued has completed before the tensor memory is released
    if (lane == 0) tc::commit(drain_bar);
    __syncwarp();
    if (!wwait(drain_bar, 0)) bad = 1;
  } else {
    // ==== row warps: softmax of row r, then its output ================================
    const int win = tid >> 6, i = tid & 63;  // window of the pair (warp-uniform) and slot
    const int ly = i / kTM, lx = i % kTM;
    const float c_l2 = p.qk_scale_log2;
    const float* brow = sbias + i * kBIAS_STRIDE;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
    Cursor cur = first, prev = first;  // the pair being computed; the pair whose O is stored
    bool prev_active = false;
    if (npair > 0 && !wwait(const_bar, 0)) bad = 1;
    // Pair n's softmax, then pair n - 1's output (its P V ran meanwhile), then pair n's P.
    for (int n = 0; n <= npair && !bad; ++n) {
      Cursor me = cur;
      if (win) me.next(p.nWy, p.nWx);
      const bool active = n < npair && i < kTN && (win == 0 || 2 * n + 1 < nwin);
      uint32_t pw[32];
      if (n < npair) {
        if (!wwait(s_full, n & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t sa[32], sb[16], sc;
        tc::ld49_wait(trow + kS_COL + 64 * win, sa, sb, sc);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free);

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
      if (n > 0) {
        // ---- pair n - 1: its row of O / the row sum, at the token the row was read from
        if (!wwait(o_full, (n - 1) & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        uint32_t o[32], osum;
        tc::ld32_1_wait(trow + kO_COL + 32 * win, trow + kO_COL + 64, o, osum);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
        if (prev_active) {
          const float inv = 1.0f / __uint_as_float(osum);
          const float2 i2 = make_float2(inv, inv);
          int yy = prev.wy * kTM + ly + s, xx = prev.wx * kTM + lx + s;
          yy = yy >= H ? yy - H : yy;
          xx = xx >= W ? xx - W : xx;
          const int64_t tok = ((int64_t)prev.b * H + yy) * W + xx;
          uint4* dst = reinterpret_cast<uint4*>(p.out + tok * p.C + h * kHeadDim);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w4[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 v = __fmul2_rn(
                  make_float2(__uint_as_float(o[8 * q + 2 * u]), __uint_as_float(o[8 * q + 2 * u + 1])), i2);
              w4[u] = pack_bf16(v.x, v.y);
            }
            dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      if (n < npair) {
        // P's previous contents were consumed: this thread waited for O of pair n - 1
        tc::st_x32(trow + kP_COL, pw);
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
#ifdef SWIN_WATTN_FAULT_INJECTION
        // armed: row warp 0 withholds its arrival for the first pair, so the MMA thread's
        // bounded wait for P runs out
        if (!(p.fault == kFaultFwdTcgen05 && warp == 0 && n == 0))
#endif
          if (lane == 0) tc::mbar_arrive(p_full);
        prev = me;
        prev_active = active;
        cur.next(p.nWy, p.nWx);
        cur.next(p.nWy, p.nWx);
      }
    }
  }
  if (bad) atomicOr(p.err, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

// The plan's constant operands of fwd_tc_kernel: U (query region one-hot, -100), V of the
// three boundary classes (core-matrix K16 layout), and per head the bias image
// bias[i][j] * log2(e) in rows of kBIAS_STRIDE floats (zero outside 49 x 49).
__global__ void tc_tables_kernel(const float* __restrict__ dense, int nH, int H, int W, int s,
                                 unsigned char* __restrict__ tables) {
  const int nU = 128 * 8, nV = 3 * 64 * 8, nB = nH * 64 * kBIAS_STRIDE;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nU + nV + nB; e += gridDim.x * blockDim.x) {
    if (e < nU) {
      const int r = e >> 3, k = 2 * (e & 7), i = r & 63;
      uint32_t w = 0u;
      if (s > 0 && i < kTN && k < 8) {
        const int c = (i / kTM >= kTM - s ? 2 : 0) | (i % kTM >= kTM - s ? 1 : 0);
        w = (((k & 3) == c) ? kMaskUBits : 0u) | (((k + 1) & 3) == c ? kMaskUBits << 16 : 0u);
      }
      *reinterpret_cast<uint32_t*>(tables + k16_off(r, k)) = w;
    } else if (e < nU + nV) {
      const int f = e - nU, cls = 1 + (f >> 9), j = (f >> 3) & 63, k = 2 * (f & 7);
      uint32_t w = 0u;
      if (s > 0) w = mask_v_bits(cls, j, k, H, W, kTM, s) | (mask_v_bits(cls, j, k + 1, H, W, kTM, s) << 16);
      *reinterpret_cast<uint32_t*>(tables + kU_BYTES + (cls - 1) * kVC_BYTES + k16_off(j, k)) = w;
    } else {
      const int f = e - nU - nV, hh = f / (64 * kBIAS_STRIDE), r = f % (64 * kBIAS_STRIDE);
      const int i = r / kBIAS_STRIDE, j = r % kBIAS_STRIDE;
      reinterpret_cast<float*>(tables + kMASK_BYTES)[f] =
          (i < kTN && j < kTN) ? dense[((int64_t)hh * kTN + i) * kTN + j] * kLog2e : 0.0f;
    }
  }
}

}  // namespace

// ---- host side ---------------------------------------------------------------------

// Tokens are addressed by 32-bit row coordinates of the tensor map.
bool fwd_tc_applies(const Plan& pl) {
  return pl.M == kTM && pl.dtype == SWIN_WATTN_BF16 && (int64_t)pl.B * pl.H * pl.W < ((int64_t)1 << 31);
}

size_t tc_tables_bytes(const Plan& pl) {
  return pl.M == kTM ? (size_t)kMASK_BYTES + (size_t)pl.nH * kBIAS_BYTES : 0;
}

cudaError_t launch_tc_tables(const Plan& pl, cudaStream_t st) {
  if (pl.tc_tables == nullptr) return cudaSuccess;
  const int64_t n = 128 * 8 + 3 * 64 * 8 + (int64_t)pl.nH * 64 * kBIAS_STRIDE;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 1024);
  tc_tables_kernel<<<grid, 256, 0, st>>>(pl.dense_bias, pl.nH, pl.H, pl.W, pl.s, pl.tc_tables);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The q/k/v tensor [batch, H, W, 3C] (bf16) as tensor maps, all with 32-channel (one
// head) boxes, 64-byte swizzled in shared memory:
//   gather  [tokens, 3C], one-token rows, for tile::gather4 loads;
//   box     [B, H, W, 3C], 7 x 7 tokens: a window that does not wrap;
//   top/bot the same with 7 x (7 - s) and 7 x s tokens: the two row bands of a window that
//           wraps at the bottom border only.
cudaError_t make_qkv_maps(const Plan& pl, const void* qkv, int batch, CUtensorMap* gather, CUtensorMap* box,
                          CUtensorMap* top, CUtensorMap* bot) {
  return make_act_maps(pl, qkv, batch, 3 * pl.C, gather, box, top, bot);
}

// The same maps for any [batch, H, W, channels] bf16 activation (qkv: 3C; dO: C).
cudaError_t make_act_maps(const Plan& pl, const void* act, int batch, int channels, CUtensorMap* gather,
                          CUtensorMap* box, CUtensorMap* top, CUtensorMap* bot) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const void* qkv = act;
  const int64_t tokens = (int64_t)batch * pl.H * pl.W;
  const cuuint64_t row = (cuuint64_t)channels * 2;
  const cuuint64_t dims[2] = {(cuuint64_t)channels, (cuuint64_t)tokens};
  const cuuint64_t strides[1] = {row};
  const cuuint32_t gbox[2] = {kHeadDim, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  if (encode(gather, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, gbox, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const cuuint64_t bdims[4] = {(cuuint64_t)channels, (cuuint64_t)pl.W, (cuuint64_t)pl.H, (cuuint64_t)batch};
  const cuuint64_t bstrides[3] = {row, row * pl.W, row * pl.W * pl.H};
  const cuuint32_t heights[3] = {kTM, (cuuint32_t)(pl.s > 0 ? kTM - pl.s : kTM), (cuuint32_t)(pl.s > 0 ? pl.s : kTM)};
  CUtensorMap* maps[3] = {box, top, bot};
  for (int m = 0; m < 3; ++m) {
    const cuuint32_t bbox[4] = {kHeadDim, kTM, heights[m], 1};
    if (encode(maps[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(qkv), bdims, bstrides, bbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

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
  CUtensorMap map, box_map, top_map, bot_map;
  cudaError_t e = make_qkv_maps(pl, qkv, batch, &map, &box_map, &top_map, &bot_map);
  if (e != cudaSuccess) return e;
  TcParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.tables = pl.tc_tables;
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
  p.wait_ns = wait_limit_ns();
  p.fault = fault_site();
  return launch_pdl(fwd_tc_kernel, dim3(L.grid), dim3(L.threads), L.smem, st, map, box_map, top_map, bot_map, p);
}

}  // namespace swin
