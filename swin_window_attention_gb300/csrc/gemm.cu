// The two matrix products around the attention, on the fifth-generation tensor cores.
//
// Producer (in front of the attention): LayerNorm over the C channels of each token, then
// qkv = LN(x) W^T + b (W [3C, C] bf16, b [3C] fp32), written as the [tokens, 3C] bf16
// tensor the attention reads. The NVIDIA Swin talk (uticex.com article 1598, section 2
// "training optimisation") lists LayerNorm and the qkv GEMM among the operations fused
// around the window attention, and its section 3 fuses the qkv GEMM with its bias; the
// cyclic shift and the window partition that the talk fuses with them are already folded
// into the attention's loads here, so this kernel writes qkv in plain token order.
//
// The normalisation is moved to the other side of the product:
//   LN(x) W^T + b = rstd * (x W'^T) - rstd * mean * u + v,
//   W'[n][c] = bf16(gamma_c W[n][c]),  u_n = sum_c W'[n][c],  v_n = sum_c beta_c W[n][c] + b_n,
// so the tensor cores consume the raw bf16 x tiles as they arrive and the epilogue applies
// the row statistics (u is summed from the rounded W', so the mean cancels exactly against
// the rounded weights). W', u and v depend on the weights alone: the talk's section 3 says
// inference may transform the qkv weight and bias ahead of time, so they are built once by
// qkv_prepare_launch (or on every call by qkv_proj_launch). The mean and
// 1 / sqrt(var + eps) of each token come from one of two places:
// * when every token tile is one work item (many tokens), statistics warps sum them from
//   the x tiles already staged for the product, at no extra memory traffic;
// * when the output channels of a token tile are split over several work items (few
//   tokens, wide C), gemm_prep_kernel computes them first in one coalesced pass over x,
//   so that no work item repeats the sums.
//
// Consumer (after the attention): y = residual + O Wp^T + bp (O the attention output
// [tokens, C] bf16, Wp [C, C] bf16, bp [C] fp32, the residual [tokens, C] bf16), the
// output projection with the bias and residual addition that the same talk's section 3
// fuses into one vectorised elementwise pass (its half2 example) moved into the product's
// epilogue, so the projection's output never goes to memory before the residual is added.
//
// Both are one kernel, gemm_kernel<MODE>: a dense contraction (2 K N flops per token for
// K input and N output channels). One persistent CTA per SM walks work items (128 tokens,
// the MMA's M, times a group of output-channel tiles of N <= 256), with specialised warps
// whose pipelines run on across items:
// * copy warp: TMA loads of activation chunks [128 tokens x 64 channels] and weight
//   chunks [N tile x 64 channels], 128-byte swizzled, into a ring of as many stages as
//   the rest of the shared memory holds (3 to 8); channels past C in the last chunk
//   arrive as zeros and add nothing;
// * MMA warp, one thread: per chunk four M128 N<=256 K16 tcgen05.mma (A = the activation
//   chunk, B = the weight chunk) into one of two tensor-memory accumulators;
// * statistics warps (four, producer with statistics on chip): thread r sums its token
//   row's x and x^2, shifted by the row's first value, over the chunks of an item's first
//   output tile and publishes mean and rstd;
// * epilogue warps (eight, two per tensor-memory lane quadrant, taking alternate
//   32-channel slices): thread r forms rstd * acc - rstd * mean * u + v (producer) or
//   acc + bp + residual (consumer) for its token row and rounds it to bf16 into one of
//   the warp's own 64-byte-swizzled staging tiles [32 rows x 32 channels], which the
//   warp's first lane writes out with a TMA store (two or three tiles per warp rotate; no
//   barrier beyond the warp), while the next output tile accumulates. The consumer's
//   residual slice arrives in that staging tile by a TMA load one slice ahead; u and v
//   (bp) of a warp's slices are staged per output tile in its corner of shared memory.
// Every wait is bounded (1 s); a wait that runs out sets the caller's status word (when
// one is given) and the CTA leaves after releasing its tensor memory.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kBM = 128;                       // tokens per work item
constexpr int kKC = 64;                        // channels per K chunk: one 128-byte row
constexpr int kSC = 32;                        // output channels per stored slice
constexpr int kMaxNT = 256;                    // output channels per N tile
constexpr int kMaxC = 1536;
constexpr int kMaxSTAGES = 8;
constexpr int kXCH = kBM * 128;                // x chunk
// Epilogues: the producer with statistics from the prep pass or summed on chip, and the
// consumer.
enum GemmMode { kLnPrepStats = 0, kLnChipStats = 1, kBiasResidual = 2 };

// Warp roles: [statistics warps 0..3 when on chip], 8 epilogue warps, MMA, copy.
template <int MODE>
struct Roles {
  static constexpr int kEPI0 = MODE == kLnChipStats ? 4 : 0;
  static constexpr int kMMA = kEPI0 + 8, kCOPY = kMMA + 1;
  static constexpr int kTHREADS = (kCOPY + 1) * 32;
};
// Shared memory, from a 1024-byte aligned base: the stage ring (stages x stage_bytes),
// [mean and rstd: 2 buffers x 128 x float2, with in-kernel statistics], per epilogue warp
// its staging tiles of 32 rows x 64 bytes [and its u/v corner], the mbarriers and the
// tensor-memory address.
constexpr int kSTATS_BYTES = 2 * kBM * 8;
// Staging tiles per epilogue warp: three where the epilogue paces the kernel, so that a
// store has two slices' time to read its tile before the tile is needed again (for the
// consumer the residual arrives by TMA in the tile the result is then written over and
// stored from, one slice ahead); two for the producer with the statistics pass (few
// tokens, wide C: the tensor cores pace it, and the ring keeps the shared memory).
template <int MODE>
__host__ __device__ constexpr int out_bufs() { return MODE == 0 ? 2 : 3; }
// per epilogue warp: the staging tiles, then (where the epilogue paces the kernel) u and
// v of its slices of the current output tile (up to 4 slices x 32 channels x 2 floats)
template <int MODE>
__host__ __device__ constexpr int uv_warp_bytes() { return MODE == 0 ? 0 : 4 * 64 * 4; }
template <int MODE>
__host__ __device__ constexpr int out_bytes() { return 8 * (out_bufs<MODE>() * 32 * 64 + uv_warp_bytes<MODE>()); }
constexpr int kRBAR0 = 2 * kMaxSTAGES + 8;  // consumer: residual-load barriers, 3 per epilogue warp
constexpr int kDRAIN = kRBAR0 + 8 * 3;      // the MMA thread's last commit before it leaves
constexpr int kNBAR = kDRAIN + 1;
template <int MODE>
__host__ __device__ constexpr int tail_bytes() { return out_bytes<MODE>() + 8 * kNBAR + 8 + 1024; }  // + alignment slack
// More than half of an SM's shared memory: one CTA per SM, so the 512-column tensor
// memory allocation never waits for another CTA of this kernel.
constexpr int kMinSMEM = 120 * 1024;
constexpr int kTMEM_COLS = 512;                // two accumulators of up to 256 columns
constexpr uint32_t kSW128 = 2;  // descriptor layout: 128-byte swizzle

struct GemmParams {
  __nv_bfloat16* out;              // [T, N]
  const float* u;                  // [N] producer: row sums of W'
  const float* v;                  // [N] producer: beta W^T + b; consumer: bp
  const float2* stats;             // [T] (mean, rstd), producer with the prep pass
  int* status;                     // optional: bit 0 set when a bounded wait ran out
  uint64_t wait_ns;                // bound of each wait
  int fault;                       // armed fault site (fault-injection build only)
  // producer with 8-bit output: 1 / scale of q, k and v (output channel n belongs to
  // tensor n / K), and the optional per-tensor max |value| (float bits, atomically max-ed)
  float f8_inv[3];
  unsigned int* f8_amax;
  int T, K, N, NT, tiles_per_item, n_tt, n_items;
  int stages, stage_bytes;  // the ring: stages x (x chunk + NT x 128 bytes), 1024-byte multiples
  int off_stats, off_out, off_bar;
  float eps;
};

__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, limit_ns)) != 0;
}

// Two fp32 values rounded to OCP FP8 E4M3 (nearest even, saturated to +-448): `lo` in the
// low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int MODE, bool F8>
__global__ void __launch_bounds__(Roles<MODE>::kTHREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                const __grid_constant__ CUtensorMap out_map, const __grid_constant__ CUtensorMap res_map,
                const GemmParams p) {
  using R = Roles<MODE>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  pdl_launch_dependents();
  const uint32_t smem0 = smem_u32(smem);
  float2* sstats = reinterpret_cast<float2*>(smem + p.off_stats);  // [2][128] (mean, rstd)
  const uint32_t bar0 = smem0 + p.off_bar;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto empty_bar = [&](int st) { return bar0 + 8 * (kMaxSTAGES + st); };
  auto dfull_bar = [&](int b) { return bar0 + 8 * (2 * kMaxSTAGES + b); };
  auto dfree_bar = [&](int b) { return bar0 + 8 * (2 * kMaxSTAGES + 2 + b); };
  auto sfull_bar = [&](int b) { return bar0 + 8 * (2 * kMaxSTAGES + 4 + b); };
  auto sfree_bar = [&](int b) { return bar0 + 8 * (2 * kMaxSTAGES + 6 + b); };
  const int stages = p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.off_bar + 8 * kNBAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = p.N / p.NT;
  const int kcn = (p.K + kKC - 1) / kKC;
  // Work item i: token tile i % n_tt, output-channel tiles [j0, j0 + ntile) of group i / n_tt.
  auto item_tiles = [&](int i, int& t0, int& j0, int& ntile) {
    t0 = (i % p.n_tt) * kBM;
    j0 = (i / p.n_tt) * p.tiles_per_item;
    ntile = min(p.tiles_per_item, n_tiles - j0);  // >= 1 by construction
  };

  if (warp == R::kMMA) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < stages; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), MODE == kLnChipStats ? 1 + 4 : 1);  // the MMA commit [and the statistics warps]
    }
    if constexpr (MODE == kBiasResidual)
      for (int b = 0; b < 8 * 3; ++b) tc::mbar_init(bar0 + 8 * (kRBAR0 + b), 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(dfull_bar(b), 1);
      tc::mbar_init(dfree_bar(b), 8);
      tc::mbar_init(sfull_bar(b), 4);
      tc::mbar_init(sfree_bar(b), 8);
    }
    tc::mbar_init(bar0 + 8 * kDRAIN, 1);
    tc::mbar_init_fence();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // The prologue above touches only this CTA's shared and tensor memory, so it may overlap
  // the previous kernel on the stream; every global read comes after this wait.
  pdl_wait();
  int bad = 0;

  if (warp == R::kCOPY) {
    // ==== copies: x chunk and W' chunk of each step into the next ring stage ==========
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, first = 1;  // ring phase; the first pass needs no free stage
      for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x) {
        int t0, j0, ntile;
        item_tiles(it, t0, j0, ntile);
        for (int s_ = 0; s_ < ntile * kcn; ++s_) {
          if (!first && !tc::mbar_wait(empty_bar(st), ph ^ 1, p.wait_ns)) {
            bad = 1;
            break;
          }
          const int kc = s_ % kcn, n0 = (j0 + s_ / kcn) * p.NT;
          const uint32_t base = smem0 + st * p.stage_bytes;
          tc::mbar_expect_tx(full_bar(st), p.stage_bytes);
          tc::tile_load_2d(base, &x_map, kc * kKC, t0, full_bar(st));
          tc::tile_load_2d(base + kXCH, &w_map, kc * kKC, n0, full_bar(st));
          if (++st == stages) {
            st = 0;
            ph ^= 1;
            first = 0;
          }
        }
      }
      // every load issued has landed before the CTA leaves, also when another role's wait
      // ran out before it consumed them (a stage's last phase has completed already unless
      // its bytes are still coming)
      for (int s2 = 0; s2 < (first ? st : stages); ++s2)
        tc::mbar_wait(full_bar(s2), s2 < st ? ph : ph ^ 1, p.wait_ns);
    }
    __syncwarp();
  } else if (warp == R::kMMA) {
    // ==== MMA issue: one thread; the warp waits together ==============================
    const uint32_t idesc = tc::idesc_bf16(128, p.NT, false);
    int st = 0, g = 0;  // ring stage and output-tile counter
    uint32_t ph = 0;    // ring phase
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      for (int jj = 0; jj < ntile && !bad; ++jj, ++g) {
        const int buf = g & 1;
        if (g >= 2 && !warp_wait(dfree_bar(buf), ((g >> 1) - 1) & 1, p.wait_ns)) {
          bad = 1;
          break;
        }
        for (int kc = 0; kc < kcn; ++kc) {
          if (!warp_wait(full_bar(st), ph, p.wait_ns)) {
            bad = 1;
            break;
          }
          if (lane == 0) {
            tc::fence_after_sync();
            const uint32_t a = smem0 + st * p.stage_bytes, w = a + kXCH;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ss(tmem + buf * kMaxNT, tc::sdesc(a + kk * 32, 16, 1024, kSW128),
                         tc::sdesc(w + kk * 32, 16, 1024, kSW128), idesc, kc > 0 || kk > 0);
            tc::commit(empty_bar(st));
#ifdef SWIN_WATTN_FAULT_INJECTION
            // armed: the first output tile's accumulator is never announced, so the
            // epilogue's bounded wait for it runs out
            if (!(p.fault == kFaultGemm && g == 0))
#endif
              if (kc == kcn - 1) tc::commit(dfull_bar(buf));
          }
          __syncwarp();
          if (++st == stages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
    }
    // every MMA this thread issued has completed before the tensor memory is released
    if (lane == 0) tc::commit(bar0 + 8 * kDRAIN);
    __syncwarp();
    if (!warp_wait(bar0 + 8 * kDRAIN, 0, p.wait_ns)) bad = 1;
  } else if (warp < R::kEPI0) {
    // ==== statistics warps: shifted sums of row r over the item's first output tile =====
    const int r = tid;
    int st = 0, k = 0;  // ring stage and item counter
    uint32_t ph = 0;    // ring phase
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x, ++k) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      float shift = 0.0f;
      float2 sh2 = make_float2(0.0f, 0.0f), s1v = make_float2(0.0f, 0.0f), s2v = make_float2(0.0f, 0.0f);
      for (int s_ = 0; s_ < ntile * kcn; ++s_) {
        if (!warp_wait(full_bar(st), ph, p.wait_ns)) {
          bad = 1;
          break;
        }
        if (s_ < kcn) {
          const unsigned char* xc = smem + st * p.stage_bytes;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (s_ * kKC + c * 8 >= p.K) break;  // zero fill past C (C is a multiple of 8)
            const uint4 w4 = *reinterpret_cast<const uint4*>(xc + r * 128 + ((c ^ (r & 7)) << 4));
            const uint32_t in[4] = {w4.x, w4.y, w4.z, w4.w};
            if (s_ == 0 && c == 0) {
              shift = bf16_lo(in[0]);
              sh2 = make_float2(-shift, -shift);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 a = __fadd2_rn(make_float2(bf16_lo(in[u]), bf16_hi(in[u])), sh2);
              s1v = __fadd2_rn(s1v, a);
              s2v = __ffma2_rn(a, a, s2v);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty_bar(st));
        if (++st == stages) {
          st = 0;
          ph ^= 1;
        }
        if (s_ == kcn - 1) {
          // mean = shift + s1 / C; var = s2 / C - (s1 / C)^2 (shifted sums)
          const float m1 = (s1v.x + s1v.y) / p.K;
          const float var = fmaxf((s2v.x + s2v.y) / p.K - m1 * m1, 0.0f);
          const int sb = k & 1;
          if (k >= 2 && !warp_wait(sfree_bar(sb), ((k >> 1) - 1) & 1, p.wait_ns)) {
            bad = 1;
            break;
          }
          sstats[sb * kBM + r] = make_float2(shift + m1, rsqrtf(var + p.eps));
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(sfull_bar(sb));
        }
      }
    }
  } else {
    // ==== epilogue warps: rstd * acc - rstd * mean * u + v or acc + bp + residual, bf16,
    //      staged TMA stores ===========================================================
    constexpr int NB = out_bufs<MODE>();
    const int ew = warp - R::kEPI0, quad = ew & 3, parity = ew >> 2;
    const int row = quad * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
    unsigned char* wstage = smem + p.off_out + ew * (NB * 32 * 64 + uv_warp_bytes<MODE>());
    float* wuv = reinterpret_cast<float*>(wstage + NB * 32 * 64);  // [slice i][u 32 | v 32]
    const bool has_slices = parity * kSC < p.NT;  // at N tile 32 the second warp of a quadrant idles
    // Consumer: the residual of the warp's slices arrives by TMA, one slice ahead, in the
    // staging tile the slice's result is written over. The warp's slices in order: items
    // it, their output tiles jj, channel offsets c0 = parity * 32 + 64 i.
    const uint32_t rbar0 = bar0 + 8 * (kRBAR0 + 3 * ew);
    int nx_it = blockIdx.x, nx_jj = 0, nx_c0 = parity * kSC;  // the next slice to request
    int issued = 0;                                           // residual loads requested
    auto request_next = [&]() {
      if (!has_slices || nx_it >= p.n_items) return;
      int t0_, j0_, nt_;
      item_tiles(nx_it, t0_, j0_, nt_);
      if (lane == 0) {
        const uint32_t rb = rbar0 + 8 * (issued % 3);
        tc::mbar_expect_tx(rb, 32 * 64);
        tc::tile_load_2d(smem_u32(wstage + (issued % 3) * (32 * 64)), &res_map, (j0_ + nx_jj) * p.NT + nx_c0,
                         t0_ + quad * 32, rb);
      }
      ++issued;
      nx_c0 += 2 * kSC;
      if (nx_c0 >= p.NT) {
        nx_c0 = parity * kSC;
        if (++nx_jj >= nt_) {
          nx_jj = 0;
          nx_it += gridDim.x;
        }
      }
    };
    if constexpr (MODE == kBiasResidual) request_next();
    int g = 0, k = 0, m = 0;  // output tiles, items, slices stored by this warp
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x, ++k) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      float2 ms = make_float2(0.0f, 1.0f);
      if constexpr (MODE == kLnChipStats) {
        const int sb = k & 1;
        if (!warp_wait(sfull_bar(sb), (k >> 1) & 1, p.wait_ns)) {
          bad = 1;
          break;
        }
        ms = sstats[sb * kBM + row];
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(sfree_bar(sb));
      } else if constexpr (MODE == kLnPrepStats) {
        ms = t0 + row < p.T ? p.stats[t0 + row] : make_float2(0.0f, 0.0f);
      }
      const float rstd = ms.y, nmr = -ms.x * ms.y;
      const float2 r2 = make_float2(rstd, rstd), nm2 = make_float2(nmr, nmr);
      for (int jj = 0; jj < ntile; ++jj, ++g) {
        const int buf = g & 1;
        const int n0 = (j0 + jj) * p.NT;
        // u and v (bp for the consumer) of the warp's slices of this tile: one coalesced
        // word per lane and slice, loaded while the accumulator is still being summed and
        // kept in the warp's corner of shared memory for broadcast reads (with the
        // statistics pass the tensor cores pace the kernel: broadcast reads from global)
        if constexpr (MODE != kLnPrepStats) {
          float ut[4], vt[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = parity * kSC + 2 * kSC * i;
            ut[i] = vt[i] = 0.0f;
            if (c < p.NT) {
              vt[i] = __ldg(p.v + n0 + c + lane);
              if constexpr (MODE != kBiasResidual) ut[i] = __ldg(p.u + n0 + c + lane);
            }
          }
          __syncwarp();  // the previous tile's reads of the corner are done
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wuv[64 * i + lane] = ut[i];
            wuv[64 * i + 32 + lane] = vt[i];
          }
          __syncwarp();
        }
        if (!warp_wait(dfull_bar(buf), (g >> 1) & 1, p.wait_ns)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        int si = 0;  // the warp's slice index within the tile
        for (int c0 = parity * kSC; c0 < p.NT; c0 += 2 * kSC, ++m, ++si) {
          unsigned char* so = wstage + (m % NB) * (32 * 64);
          if constexpr (MODE == kBiasResidual) {
            if (m >= 2) {
              if (lane == 0) tc::bulk_wait_read<1>();  // the store of slice m - 2 has read its tile
              __syncwarp();
            }
            request_next();  // the residual of slice m + 1, into the tile of slice m - 2
          } else if (m >= NB) {
            if (lane == 0) tc::bulk_wait_read<NB - 1>();  // the store of slice m - NB has read its tile
            __syncwarp();
          }
          // 8-bit output: this slice's tensor scale, the row's max |value|, packed words
          [[maybe_unused]] const int f8t = (n0 + c0) / p.K;
          [[maybe_unused]] const float f8inv = f8t == 0 ? p.f8_inv[0] : (f8t == 1 ? p.f8_inv[1] : p.f8_inv[2]);
          [[maybe_unused]] float f8max = 0.0f;
          [[maybe_unused]] uint32_t f8w[4];
          const float4* u4s = MODE == kLnPrepStats ? reinterpret_cast<const float4*>(p.u + n0 + c0)
                                                   : reinterpret_cast<const float4*>(wuv + 64 * si);
          const float4* v4s = MODE == kLnPrepStats ? reinterpret_cast<const float4*>(p.v + n0 + c0) : u4s + 8;
          uint32_t a[32];
          tc::ld32_wait(trow + buf * kMaxNT + c0, a);
          if constexpr (MODE == kBiasResidual) {
            if (!warp_wait(rbar0 + 8 * (m % 3), (m / 3) & 1, p.wait_ns)) {
              bad = 1;
              break;
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4* sp = reinterpret_cast<uint4*>(so + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
            uint4 rw = make_uint4(0, 0, 0, 0);
            if constexpr (MODE == kBiasResidual) rw = *sp;  // the residual's 8 channels of this row
            const uint32_t rr[4] = {rw.x, rw.y, rw.z, rw.w};
            const float4 vA = v4s[2 * c], vB = v4s[2 * c + 1];  // broadcast reads
            const float vv[8] = {vA.x, vA.y, vA.z, vA.w, vB.x, vB.y, vB.z, vB.w};
            float uu[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if constexpr (MODE != kBiasResidual) {
              const float4 uA = u4s[2 * c], uB = u4s[2 * c + 1];
              uu[0] = uA.x, uu[1] = uA.y, uu[2] = uA.z, uu[3] = uA.w;
              uu[4] = uB.x, uu[5] = uB.y, uu[6] = uB.z, uu[7] = uB.w;
            }
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 8 * c + 2 * q;
              const float2 a0 = make_float2(__uint_as_float(a[e]), __uint_as_float(a[e + 1]));
              const float2 v2 = make_float2(vv[2 * q], vv[2 * q + 1]);
              float2 y;
              if constexpr (MODE == kBiasResidual) {
                // (acc + bp) + residual, as the definition adds them
                y = __fadd2_rn(__fadd2_rn(a0, v2), make_float2(bf16_lo(rr[q]), bf16_hi(rr[q])));
              } else {
                y = __ffma2_rn(a0, r2, __ffma2_rn(nm2, make_float2(uu[2 * q], uu[2 * q + 1]), v2));
              }
              if constexpr (F8) {
                f8max = fmax3(f8max, fabsf(y.x), fabsf(y.y));
                const float2 z = __fmul2_rn(y, make_float2(f8inv, f8inv));
                o[q] = e4m3x2(z.x, z.y);  // channels 8c + 2q, +1 as two bytes
              } else {
                o[q] = pack_bf16(y.x, y.y);
              }
            }
            if constexpr (F8) {
              // 8 bytes of this row: its 32-byte row holds 16-byte chunk c >> 1 at position
              // (c >> 1) ^ ((row >> 2) & 1) (the copy engine's 32-byte swizzle)
              f8w[2 * (c & 1)] = o[0] | (o[1] << 16);
              f8w[2 * (c & 1) + 1] = o[2] | (o[3] << 16);
              if (c & 1)
                *reinterpret_cast<uint4*>(so + lane * 32 + (((c >> 1) ^ ((lane >> 2) & 1)) << 4)) =
                    make_uint4(f8w[0], f8w[1], f8w[2], f8w[3]);
            } else {
              *sp = make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
          if constexpr (F8) {
            if (p.f8_amax != nullptr) {
              const unsigned int mx = __reduce_max_sync(0xffffffffu, __float_as_uint(f8max));
              if (lane == 0) atomicMax(p.f8_amax + f8t, mx);
            }
          }
          tc::fence_proxy_async();  // the staging tile to the copy engine
          __syncwarp();
          if (lane == 0) {
            tc::tile_store_2d(&out_map, n0 + c0, t0 + quad * 32, smem_u32(so));
            tc::bulk_commit();
          }
        }
        if (bad) break;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(dfree_bar(buf));
      }
    }
    if constexpr (MODE == kBiasResidual) {
      // after a timeout: let the residual loads still in flight land before the CTA leaves
      for (int q = m; q < issued; ++q) warp_wait(rbar0 + 8 * (q % 3), (q / 3) & 1, p.wait_ns);
    }
    if (lane == 0) tc::bulk_wait_all();
  }
  if (bad && p.status != nullptr) atomicOr(p.status, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == R::kMMA) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

// The producer's preparation. Blocks [0, fold_blocks): W'[n][c] = bf16(gamma_c W[n][c]),
// u_n = sum_c W'[n][c], v_n = sum_c beta_c W[n][c] + b_n, one warp per output channel n.
// Blocks from fold_blocks on (when stats is given): (mean, 1 / sqrt(var + eps)) of each
// token's C channels, four tokens per warp with their loads in flight together; shifted
// sums (by the row's first value) in fp32, reduced across the warp.
__global__ void gemm_prep_kernel(const __nv_bfloat16* __restrict__ w, const float* __restrict__ gamma,
                                const float* __restrict__ beta, const float* __restrict__ b, int C, int N,
                                __nv_bfloat16* __restrict__ wf, float* __restrict__ u, float* __restrict__ v,
                                int fold_blocks, const __nv_bfloat16* __restrict__ x, int T, float eps,
                                float2* __restrict__ stats) {
  pdl_wait();  // x and the weights may come from the previous kernel on the stream
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  if ((int)blockIdx.x < fold_blocks) {
    // gamma and beta staged once per block, read back as float4 (8 channels per lane)
    __shared__ __align__(16) float sg[kMaxC], sb[kMaxC];
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      sg[c] = gamma[c];
      sb[c] = beta[c];
    }
    __syncthreads();
    for (int n = blockIdx.x * wpb + wib; n < N; n += fold_blocks * wpb) {
      const uint4* wr = reinterpret_cast<const uint4*>(w + (int64_t)n * C);
      uint4* fr = reinterpret_cast<uint4*>(wf + (int64_t)n * C);
      float su_ = 0.0f, sv_ = 0.0f;
#pragma unroll 4
      for (int c8 = lane; c8 < C / 8; c8 += 32) {  // 8 channels per lane and step
        const uint4 w4 = wr[c8];
        const float4 g0 = reinterpret_cast<const float4*>(sg)[2 * c8], g1 = reinterpret_cast<const float4*>(sg)[2 * c8 + 1];
        const float4 b0 = reinterpret_cast<const float4*>(sb)[2 * c8], b1 = reinterpret_cast<const float4*>(sb)[2 * c8 + 1];
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const uint32_t in[4] = {w4.x, w4.y, w4.z, w4.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float w0 = bf16_lo(in[k]), w1 = bf16_hi(in[k]);
          const __nv_bfloat16 f0 = __float2bfloat16_rn(gg[2 * k] * w0);
          const __nv_bfloat16 f1 = __float2bfloat16_rn(gg[2 * k + 1] * w1);
          su_ += __bfloat162float(f0) + __bfloat162float(f1);
          sv_ = fmaf(bb[2 * k], w0, fmaf(bb[2 * k + 1], w1, sv_));
          o[k] = (uint32_t)__bfloat16_as_ushort(f0) | ((uint32_t)__bfloat16_as_ushort(f1) << 16);
        }
        fr[c8] = make_uint4(o[0], o[1], o[2], o[3]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        su_ += __shfl_xor_sync(0xffffffffu, su_, o);
        sv_ += __shfl_xor_sync(0xffffffffu, sv_, o);
      }
      if (lane == 0) {
        u[n] = su_;
        v[n] = sv_ + b[n];
      }
    }
    return;
  }
  const int sblocks = gridDim.x - fold_blocks;
  for (int64_t t0 = ((int64_t)(blockIdx.x - fold_blocks) * wpb + wib) * 4; t0 < T; t0 += (int64_t)sblocks * wpb * 4) {
    const int nr = T - t0 < 4 ? (int)(T - t0) : 4;
    float shift[4];
    float2 s1[4], s2[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      shift[r] = r < nr ? __bfloat162float(x[(t0 + r) * C]) : 0.0f;
      s1[r] = make_float2(0.0f, 0.0f);
      s2[r] = make_float2(0.0f, 0.0f);
    }
    for (int c = lane; c < C / 8; c += 32) {
      uint4 w4[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        w4[r] = r < nr ? reinterpret_cast<const uint4*>(x + (t0 + r) * C)[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t in[4] = {w4[r].x, w4[r].y, w4[r].z, w4[r].w};
        const float2 sh2 = make_float2(-shift[r], -shift[r]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 a = __fadd2_rn(make_float2(bf16_lo(in[k]), bf16_hi(in[k])), sh2);
          s1[r] = __fadd2_rn(s1[r], a);
          s2[r] = __ffma2_rn(a, a, s2[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float a1 = s1[r].x + s1[r].y, a2 = s2[r].x + s2[r].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
        a2 += __shfl_xor_sync(0xffffffffu, a2, o);
      }
      if (lane == 0 && r < nr) {
        const float m1 = a1 / C;  // mean = shift + m1; var = a2 / C - m1^2
        stats[t0 + r] = make_float2(shift[r] + m1, rsqrtf(fmaxf(a2 / C - m1 * m1, 0.0f) + eps));
      }
    }
  }
}

}  // namespace

// Prepared producer weights: W' [3C, C] bf16, u and v [3C] fp32, each part 256-byte
// aligned. The one-call workspace adds the token statistics [T] (mean, rstd).
static size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }
size_t qkv_prepared_bytes(int C) { return align256((size_t)3 * C * C * 2) + 2 * align256((size_t)3 * C * 4); }
size_t qkv_stats_bytes(int64_t T) { return align256((size_t)T * 8); }
size_t qkv_workspace_bytes(int C, int64_t T) { return qkv_prepared_bytes(C) + qkv_stats_bytes(T); }

namespace {

// Output-channel tile: the largest multiple of 32 up to 256 that divides N (a multiple of
// 32).
int gemm_tile(int N) {
  for (int nt = kMaxNT; nt >= 32; nt -= 32)
    if (N % nt == 0) return nt;
  return 0;
}

// Work items: token tiles times groups of output-channel tiles; one persistent CTA per SM
// walks them. With many tokens (at least four token tiles per SM) each token tile is one
// item, so its statistics can be summed on chip. Otherwise the group size is the one
// that minimises the tiles of the busiest SM, ceil(items / SMs) x tiles per item (every
// output tile costs the same), preferring larger groups on a tie.
struct ItemPlan {
  int sms, smem_max, NT, n_tt, per, n_items;
  bool one_item_per_token_tile;
};

cudaError_t plan_items(int T, int N, ItemPlan* ip) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ip->sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ip->smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  ip->NT = gemm_tile(N);
  if (ip->NT == 0) return cudaErrorInvalidValue;
  ip->n_tt = (T + kBM - 1) / kBM;
  const int n_tiles = N / ip->NT;
  int per = n_tiles;
  if (ip->n_tt < 4 * ip->sms) {
    int64_t best = -1;
    for (int q = n_tiles; q >= 1; --q) {
      const int64_t items = (int64_t)ip->n_tt * ((n_tiles + q - 1) / q);
      const int64_t cost = (items + ip->sms - 1) / ip->sms * q;
      if (best < 0 || cost < best) {
        best = cost;
        per = q;
      }
    }
  }
  const int groups = (n_tiles + per - 1) / per;
  ip->per = per;
  ip->n_items = ip->n_tt * groups;
  ip->one_item_per_token_tile = groups == 1;
  return cudaSuccess;
}

// A row-major [outer, inner] tensor of bf16 (or of bytes with `bytes`) for the copy engine.
cudaError_t encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* map, const void* base, int inner,
                      int outer, int box_inner, int box_outer, CUtensorMapSwizzle swz, CUtensorMapL2promotion l2,
                      bool bytes = false) {
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * (bytes ? 1 : 2)};
  const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  const cuuint32_t es[2] = {1, 1};
  return encode(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

// F8: the producer's output is OCP FP8 E4M3 bytes [T, N] (32-byte-swizzled staging tiles of
// 32 rows x 32 channels, stored by the copy engine).
template <int MODE, bool F8 = false>
cudaError_t launch_gemm(const ItemPlan& ip, GemmParams p, const void* a, const void* w, cudaStream_t st,
                        const void* residual = nullptr) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap a_map, w_map, out_map;
  cudaError_t e = encode_2d(encode, &a_map, a, p.K, p.T, kKC, kBM, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e == cudaSuccess)
    e = encode_2d(encode, &w_map, w, p.K, p.N, kKC, ip.NT, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (e == cudaSuccess)
    e = encode_2d(encode, &out_map, p.out, p.N, p.T, kSC, 32, F8 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, F8);
  CUtensorMap res_map = out_map;  // read only by the consumer
  if (e == cudaSuccess && residual != nullptr)
    e = encode_2d(encode, &res_map, residual, p.N, p.T, kSC, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
  if (e != cudaSuccess) return e;
  p.NT = ip.NT;
  p.tiles_per_item = ip.per;
  p.n_tt = ip.n_tt;
  p.n_items = ip.n_items;
  p.stage_bytes = kXCH + ip.NT * 128;
  constexpr int kStatsBytes = MODE == kLnChipStats ? kSTATS_BYTES : 0;
  const int fixed = kStatsBytes + tail_bytes<MODE>();
  p.stages = std::min(kMaxSTAGES, (ip.smem_max - fixed) / p.stage_bytes);
  if (p.stages < 2) return cudaErrorInvalidConfiguration;
  p.off_stats = p.stages * p.stage_bytes;
  p.off_out = p.off_stats + kStatsBytes;
  p.off_bar = p.off_out + out_bytes<MODE>();
  const int smem = std::max(kMinSMEM, p.stages * p.stage_bytes + fixed);
  e = cudaFuncSetAttribute(gemm_kernel<MODE, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(gemm_kernel<MODE, F8>, dim3(std::min(ip.n_items, ip.sms)), dim3(Roles<MODE>::kTHREADS), smem,
                    st, a_map, w_map, out_map, res_map, p);
}

GemmParams base_params(void* out, int T, int K, int N, int* status) {
  GemmParams p{};
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.status = status;
  p.wait_ns = wait_limit_ns();
  p.fault = fault_site();
  p.T = T;
  p.K = K;
  p.N = N;
  return p;
}

}  // namespace

namespace {

struct Prepared {
  __nv_bfloat16* wf;
  float* u;
  float* v;
};

Prepared prepared_parts(void* prepared, int C) {
  unsigned char* p = static_cast<unsigned char*>(prepared);
  const int N = 3 * C;
  Prepared r;
  r.wf = reinterpret_cast<__nv_bfloat16*>(p);
  r.u = reinterpret_cast<float*>(p + align256((size_t)N * C * 2));
  r.v = reinterpret_cast<float*>(p + align256((size_t)N * C * 2) + align256((size_t)N * 4));
  return r;
}

// The fold (when w is given) and the token statistics (when the product will not sum them
// on chip) in one launch, then the product.
cudaError_t qkv_run(const void* x, const float* gamma, const float* beta, const void* w, const float* b,
                    const Prepared& pw, float2* stats, void* out, int T, int C, float eps, int* status,
                    cudaStream_t st, const float* f8_scales = nullptr, unsigned int* f8_amax = nullptr) {
  const int N = 3 * C;
  ItemPlan ip;
  cudaError_t e = plan_items(T, N, &ip);
  if (e != cudaSuccess) return e;
  const bool chip_stats = ip.one_item_per_token_tile;  // each token tile is one item: sum on chip
  const int fold_blocks = w != nullptr ? (N + 7) / 8 : 0;
  const int stat_blocks = chip_stats ? 0 : (int)std::min<int64_t>(((int64_t)T + 31) / 32, 16 * ip.sms);
  if (fold_blocks + stat_blocks > 0) {
    e = launch_pdl(gemm_prep_kernel, dim3(fold_blocks + stat_blocks), dim3(256), 0, st,
                   reinterpret_cast<const __nv_bfloat16*>(w), gamma, beta, b, C, N, pw.wf, pw.u, pw.v, fold_blocks,
                   reinterpret_cast<const __nv_bfloat16*>(x), T, eps, stats);
    if (e != cudaSuccess) return e;
  }
  GemmParams p = base_params(out, T, C, N, status);
  p.u = pw.u;
  p.v = pw.v;
  p.eps = eps;
  if (f8_scales != nullptr) {
    for (int t = 0; t < 3; ++t) p.f8_inv[t] = 1.0f / f8_scales[t];
    p.f8_amax = f8_amax;
    if (chip_stats) return launch_gemm<kLnChipStats, true>(ip, p, x, pw.wf, st);
    p.stats = stats;
    return launch_gemm<kLnPrepStats, true>(ip, p, x, pw.wf, st);
  }
  if (chip_stats) return launch_gemm<kLnChipStats>(ip, p, x, pw.wf, st);
  p.stats = stats;
  return launch_gemm<kLnPrepStats>(ip, p, x, pw.wf, st);
}

}  // namespace

// Producer, one call: the weights are folded into the workspace, then the product. Two
// launches (the prep kernel, the product).
cudaError_t qkv_proj_launch(const void* x, const float* gamma, const float* beta, const void* w, const float* b,
                            void* out, int T, int C, float eps, void* workspace, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % 32 != 0 || C < 32 || C > kMaxC) return cudaErrorInvalidValue;
  float2* stats = reinterpret_cast<float2*>(static_cast<unsigned char*>(workspace) + qkv_prepared_bytes(C));
  return qkv_run(x, gamma, beta, w, b, prepared_parts(workspace, C), stats, out, T, C, eps, status, st);
}

// Producer weights prepared ahead of time: W', u and v into `prepared`. One launch.
cudaError_t qkv_prepare_launch(const float* gamma, const float* beta, const void* w, const float* b, int C,
                               void* prepared, cudaStream_t st) {
  if (C % 32 != 0 || C < 32 || C > kMaxC) return cudaErrorInvalidValue;
  const int N = 3 * C;
  const Prepared pw = prepared_parts(prepared, C);
  return launch_pdl(gemm_prep_kernel, dim3((N + 7) / 8), dim3(256), 0, st, reinterpret_cast<const __nv_bfloat16*>(w),
                    gamma, beta, b, C, N, pw.wf, pw.u, pw.v, (N + 7) / 8, static_cast<const __nv_bfloat16*>(nullptr), 0,
                    0.0f, static_cast<float2*>(nullptr));
}

// Producer on prepared weights: [the token statistics,] the product.
cudaError_t qkv_proj_prepared_launch(const void* x, const void* prepared, void* out, int T, int C, float eps,
                                     void* stats_workspace, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % 32 != 0 || C < 32 || C > kMaxC) return cudaErrorInvalidValue;
  return qkv_run(x, nullptr, nullptr, nullptr, nullptr, prepared_parts(const_cast<void*>(prepared), C),
                 static_cast<float2*>(stats_workspace), out, T, C, eps, status, st);
}

// Producer on prepared weights with OCP FP8 E4M3 output: qkv8 = satfinite(qkv / scale_t)
// for the tensor t (q, k, v) of each channel, and optionally max |qkv_t| into amax[t].
cudaError_t qkv_proj_fp8_launch(const void* x, const void* prepared, void* out8, int T, int C, float eps,
                                const float scales[3], unsigned int* amax, void* stats_workspace, int* status,
                                cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % 32 != 0 || C < 32 || C > kMaxC) return cudaErrorInvalidValue;
  return qkv_run(x, nullptr, nullptr, nullptr, nullptr, prepared_parts(const_cast<void*>(prepared), C),
                 static_cast<float2*>(stats_workspace), out8, T, C, eps, status, st, scales, amax);
}

// Launches of one producer call for T tokens of C channels with or without the fold.
int qkv_launches(int T, int C, bool fold) {
  ItemPlan ip;
  if (T <= 0 || plan_items(T, 3 * C, &ip) != cudaSuccess) return 0;
  return 1 + ((fold || !ip.one_item_per_token_tile) ? 1 : 0);
}

// Consumer: y = residual + O Wp^T + bp. One launch.
cudaError_t proj_residual_launch(const void* o, const void* wp, const float* bp, const void* residual, void* y,
                                 int T, int C, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % 32 != 0 || C < 32 || C > kMaxC) return cudaErrorInvalidValue;
  ItemPlan ip;
  cudaError_t e = plan_items(T, C, &ip);
  if (e != cudaSuccess) return e;
  GemmParams p = base_params(y, T, C, C, status);
  p.v = bp;
  return launch_gemm<kBiasResidual>(ip, p, o, wp, st, residual);
}

}  // namespace swin
