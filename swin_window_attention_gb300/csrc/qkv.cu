// The producer step in front of the attention: LayerNorm over the C channels of each
// token, then qkv = LN(x) W^T + b (W [3C, C] bf16, b [3C] fp32), written as the
// [tokens, 3C] bf16 tensor the attention reads. The NVIDIA Swin talk (uticex.com article
// 1598, section 2 "training optimisation") lists LayerNorm and the qkv GEMM among the
// operations fused around the window attention; the cyclic shift and the window
// partition that the talk fuses with them are already folded into the attention's
// loads here, so this kernel writes qkv in plain token order.
//
// The normalisation is moved to the other side of the product:
//   LN(x) W^T + b = rstd * (x W'^T) - rstd * mean * u + v,
//   W'[n][c] = bf16(gamma_c W[n][c]),  u_n = sum_c W'[n][c],  v_n = sum_c beta_c W[n][c] + b_n,
// so the tensor cores consume the raw bf16 x tiles as they arrive, the row statistics are
// summed from the same tiles while the MMAs run, and the epilogue applies them (u is
// summed from the rounded W', so the mean cancels exactly against the rounded weights).
// qkv_fold_kernel builds W', u and v once per call.
//
// A dense contraction (2 * 3C * C flops per token) on the fifth-generation tensor cores.
// One persistent CTA per SM walks work items (128 tokens, the MMA's M, times a group of
// output-channel tiles of N <= 256), with specialised warps whose pipelines run on across
// items:
// * copy warp (13): TMA loads of x chunks [128 tokens x 32 channels] and W' chunks
//   [N tile x 32 channels], 64-byte swizzled, six stages deep;
// * MMA warp (12), one thread: per chunk two M128 N<=256 K16 tcgen05.mma (A = the x chunk,
//   B = the W' chunk) into one of two tensor-memory accumulators;
// * statistics warps (0..3): thread r sums its token row's x and x^2 (shifted by the row's
//   first value) over the chunks of an item's first output tile, then publishes mean and
//   1 / sqrt(var + eps);
// * epilogue warps (4..11, two per tensor-memory lane quadrant, each taking 16 of every
//   32 channels): thread r forms rstd * acc - rstd * mean * u + v and rounds to bf16 into
//   a 64-byte-swizzled staging tile that one thread writes out with a TMA store (two
//   staging tiles alternate), while the next output tile accumulates.
// Every wait is bounded (1 s); a wait that runs out sets the caller's status word (when
// one is given) and the CTA leaves after releasing its tensor memory.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kBM = 128;                       // tokens per work item
constexpr int kKC = 32;                        // channels per K chunk: one 64-byte row
constexpr int kMaxNT = 256;                    // output channels per N tile
constexpr int kMaxC = 1536;
constexpr int kSTAGES = 6;
constexpr int kXCH = kBM * 64;                 // x chunk
constexpr int kWCH = kMaxNT * 64;              // W' chunk
constexpr int kSTAGE = kXCH + kWCH;            // 24 KB
constexpr int kTHREADS = 14 * 32;
constexpr int kEPI_WARP0 = 4, kEPI_THREADS = 256, kMMA_WARP = 12, kCOPY_WARP = 13;
constexpr int kOFF_UV = kSTAGES * kSTAGE;              // u, v: 2 x 3 kMaxC floats
constexpr int kOFF_STATS = kOFF_UV + 6 * kMaxC * 4;    // mean, rstd: 2 buffers x 128 x 2 floats
constexpr int kOFF_OUT = kOFF_STATS + 2 * kBM * 8;     // 2 staging tiles of 128 rows x 64 B
constexpr int kOFF_BAR = kOFF_OUT + 2 * kBM * 64;
constexpr int kNBAR = 2 * kSTAGES + 8;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + alignment slack
constexpr int kTMEM_COLS = 512;                // two accumulators of up to 256 columns
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kSW64 = 4;

// More than half of the SM's shared memory: one CTA per SM, so the 512-column tensor
// memory allocation never waits.
static_assert(kSMEM > 233472 / 2 && kSMEM <= 232448, "one CTA per SM");

struct QkvParams {
  __nv_bfloat16* out;     // [T, 3C]
  const float* u;         // [3C]
  const float* v;         // [3C]
  int* status;            // optional: bit 0 set when a bounded wait ran out
  int T, C, N, NT, tiles_per_item, n_tt, n_items;
  float eps;
};

__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, kWaitLimitNs)) != 0;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kTHREADS, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                    const __grid_constant__ CUtensorMap out_map, const QkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t smem0 = smem_u32(smem);
  float* su = reinterpret_cast<float*>(smem + kOFF_UV);
  float* sv = su + 3 * kMaxC;
  float2* sstats = reinterpret_cast<float2*>(smem + kOFF_STATS);  // [2][128] (mean, rstd)
  const uint32_t bar0 = smem0 + kOFF_BAR;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto empty_bar = [&](int st) { return bar0 + 8 * (kSTAGES + st); };
  auto dfull_bar = [&](int b) { return bar0 + 8 * (2 * kSTAGES + b); };
  auto dfree_bar = [&](int b) { return bar0 + 8 * (2 * kSTAGES + 2 + b); };
  auto sfull_bar = [&](int b) { return bar0 + 8 * (2 * kSTAGES + 4 + b); };
  auto sfree_bar = [&](int b) { return bar0 + 8 * (2 * kSTAGES + 6 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 8 * kNBAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = p.N / p.NT;
  const int kcn = p.C / kKC;
  // Work item i: token tile i % n_tt, output-channel tiles [j0, j0 + ntile) of group i / n_tt.
  auto item_tiles = [&](int i, int& t0, int& j0, int& ntile) {
    t0 = (i % p.n_tt) * kBM;
    j0 = (i / p.n_tt) * p.tiles_per_item;
    ntile = min(p.tiles_per_item, n_tiles - j0);  // >= 1 by construction
  };

  if (warp == kMMA_WARP) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < kSTAGES; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(empty_bar(st), 1 + 4);  // the MMA commit and the four statistics warps
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(dfull_bar(b), 1);
      tc::mbar_init(dfree_bar(b), 8);
      tc::mbar_init(sfull_bar(b), 4);
      tc::mbar_init(sfree_bar(b), 8);
    }
    tc::mbar_init_fence();
  }
  for (int c = tid; c < p.N; c += kTHREADS) {
    su[c] = p.u[c];
    sv[c] = p.v[c];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp == kCOPY_WARP) {
    // ==== copies: x chunk and W' chunk of step q into stage q % kSTAGES ==============
    if (lane == 0) {
      int q = 0, st = 0;
      for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x) {
        int t0, j0, ntile;
        item_tiles(it, t0, j0, ntile);
        for (int s_ = 0; s_ < ntile * kcn; ++s_, ++q) {
          if (q >= kSTAGES && !tc::mbar_wait(empty_bar(st), ((q / kSTAGES) - 1) & 1, kWaitLimitNs)) {
            bad = 1;
            break;
          }
          const int kc = s_ % kcn, n0 = (j0 + s_ / kcn) * p.NT;
          const uint32_t base = smem0 + st * kSTAGE;
          tc::mbar_expect_tx(full_bar(st), kXCH + p.NT * 64);
          tc::tile_load_2d(base, &x_map, kc * kKC, t0, full_bar(st));
          tc::tile_load_2d(base + kXCH, &w_map, kc * kKC, n0, full_bar(st));
          st = st + 1 == kSTAGES ? 0 : st + 1;
        }
      }
    }
    __syncwarp();
  } else if (warp == kMMA_WARP) {
    // ==== MMA issue: one thread; the warp waits together ==============================
    const uint32_t idesc = tc::idesc_bf16(128, p.NT, false);
    int q = 0, st = 0, g = 0;  // global step and output-tile counters
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      for (int jj = 0; jj < ntile && !bad; ++jj, ++g) {
        const int buf = g & 1;
        if (g >= 2 && !warp_wait(dfree_bar(buf), ((g >> 1) - 1) & 1)) {
          bad = 1;
          break;
        }
        for (int kc = 0; kc < kcn; ++kc, ++q) {
          if (!warp_wait(full_bar(st), (q / kSTAGES) & 1)) {
            bad = 1;
            break;
          }
          if (lane == 0) {
            tc::fence_after_sync();
            const uint32_t a = smem0 + st * kSTAGE, w = a + kXCH;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              tc::mma_ss(tmem + buf * kMaxNT, tc::sdesc(a + kk * 32, 16, 512, kSW64),
                         tc::sdesc(w + kk * 32, 16, 512, kSW64), idesc, kc > 0 || kk > 0);
            tc::commit(empty_bar(st));
            if (kc == kcn - 1) tc::commit(dfull_bar(buf));
          }
          __syncwarp();
          st = st + 1 == kSTAGES ? 0 : st + 1;
        }
      }
    }
  } else if (warp < kEPI_WARP0) {
    // ==== statistics warps: shifted sums of row r over the item's first output tile =====
    const int r = tid;
    int q = 0, st = 0, k = 0;  // global step and item counters
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x, ++k) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      float shift = 0.0f;
      float2 sh2 = make_float2(0.0f, 0.0f), s1v = make_float2(0.0f, 0.0f), s2v = make_float2(0.0f, 0.0f);
      for (int s_ = 0; s_ < ntile * kcn; ++s_, ++q) {
        if (!warp_wait(full_bar(st), (q / kSTAGES) & 1)) {
          bad = 1;
          break;
        }
        if (s_ < kcn) {
          const unsigned char* xc = smem + st * kSTAGE;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 w4 = *reinterpret_cast<const uint4*>(xc + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
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
        st = st + 1 == kSTAGES ? 0 : st + 1;
        if (s_ == kcn - 1) {
          // mean = shift + s1 / C; var = s2 / C - (s1 / C)^2 (shifted sums)
          const float m1 = (s1v.x + s1v.y) / p.C;
          const float var = fmaxf((s2v.x + s2v.y) / p.C - m1 * m1, 0.0f);
          const int sb = k & 1;
          if (k >= 2 && !warp_wait(sfree_bar(sb), ((k >> 1) - 1) & 1)) {
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
    // ==== epilogue warps: rstd * acc - rstd * mean * u + v, bf16, staged TMA stores =====
    const int ew = warp - kEPI_WARP0, row = (ew & 3) * 32 + lane, half = ew >> 2;  // 16-channel half
    const int et = ew * 32 + lane;  // 0 .. 255
    const uint32_t trow = tmem + ((uint32_t)((ew & 3) * 32) << 16);
    unsigned char* stage_out = smem + kOFF_OUT;
    int g = 0, k = 0, m = 0;  // output tiles, items, 32-channel slices
    for (int it = blockIdx.x; it < p.n_items && !bad; it += gridDim.x, ++k) {
      int t0, j0, ntile;
      item_tiles(it, t0, j0, ntile);
      const int sb = k & 1;
      if (!warp_wait(sfull_bar(sb), (k >> 1) & 1)) {
        bad = 1;
        break;
      }
      const float2 ms = sstats[sb * kBM + row];
      const float rstd = ms.y, nmr = -ms.x * ms.y;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(sfree_bar(sb));
      const float2 r2 = make_float2(rstd, rstd), nm2 = make_float2(nmr, nmr);
      for (int jj = 0; jj < ntile; ++jj, ++g) {
        const int buf = g & 1;
        if (!warp_wait(dfull_bar(buf), (g >> 1) & 1)) {
          bad = 1;
          break;
        }
        tc::fence_after_sync();
        const int n0 = (j0 + jj) * p.NT;
        for (int c0 = 0; c0 < p.NT; c0 += 32, ++m) {
          unsigned char* so = stage_out + (m & 1) * (kBM * 64);
          if (m >= 2) {
            if (et == 0) tc::bulk_wait_read<1>();  // the store of slice m - 2 has read its tile
            asm volatile("bar.sync 1, %0;\n" ::"n"(kEPI_THREADS) : "memory");
          }
          uint32_t a[16];
          tc::ld16_wait(trow + buf * kMaxNT + c0 + 16 * half, a);
          const float4* uu = reinterpret_cast<const float4*>(su + n0 + c0 + 16 * half);
          const float4* vv = reinterpret_cast<const float4*>(sv + n0 + c0 + 16 * half);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[4];
#pragma unroll
            for (int w2 = 0; w2 < 2; ++w2) {
              const float4 u4 = uu[2 * c + w2], v4 = vv[2 * c + w2];
              const int e = 8 * c + 4 * w2;
              const float2 c0v = __ffma2_rn(nm2, make_float2(u4.x, u4.y), make_float2(v4.x, v4.y));
              const float2 c1v = __ffma2_rn(nm2, make_float2(u4.z, u4.w), make_float2(v4.z, v4.w));
              const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(a[e]), __uint_as_float(a[e + 1])), r2, c0v);
              const float2 y1 =
                  __ffma2_rn(make_float2(__uint_as_float(a[e + 2]), __uint_as_float(a[e + 3])), r2, c1v);
              o[2 * w2] = pack_bf16(y0.x, y0.y);
              o[2 * w2 + 1] = pack_bf16(y1.x, y1.y);
            }
            const int chunk = 2 * half + c;
            *reinterpret_cast<uint4*>(so + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
          tc::fence_proxy_async();  // the staging tile to the copy engine
          asm volatile("bar.sync 1, %0;\n" ::"n"(kEPI_THREADS) : "memory");
          if (et == 0) {
            tc::tile_store_2d(&out_map, n0 + c0, t0, smem_u32(so));
            tc::bulk_commit();
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(dfree_bar(buf));
      }
    }
    if (et == 0) tc::bulk_wait_all();
  }
  if (bad && p.status != nullptr) atomicOr(p.status, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMMA_WARP) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

// W'[n][c] = bf16(gamma_c W[n][c]); u_n = sum_c W'[n][c]; v_n = sum_c beta_c W[n][c] + b_n.
// One warp per output channel n.
__global__ void qkv_fold_kernel(const __nv_bfloat16* __restrict__ w, const float* __restrict__ gamma,
                                const float* __restrict__ beta, const float* __restrict__ b, int C, int N,
                                __nv_bfloat16* __restrict__ wf, float* __restrict__ u, float* __restrict__ v) {
  const int lane = threadIdx.x & 31;
  for (int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); n < N; n += gridDim.x * (blockDim.x >> 5)) {
    float su_ = 0.0f, sv_ = 0.0f;
    for (int c = lane; c < C; c += 32) {
      const float wv = __bfloat162float(w[(int64_t)n * C + c]);
      const __nv_bfloat16 f = __float2bfloat16_rn(gamma[c] * wv);
      wf[(int64_t)n * C + c] = f;
      su_ += __bfloat162float(f);
      sv_ = fmaf(beta[c], wv, sv_);
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
}

}  // namespace

// Workspace of one call: W' [3C, C] bf16, then u and v [3C] fp32, each 256-byte aligned.
size_t qkv_workspace_bytes(int C) {
  const size_t wf = ((size_t)3 * C * C * 2 + 255) & ~(size_t)255;
  const size_t uv = ((size_t)3 * C * 4 + 255) & ~(size_t)255;
  return wf + 2 * uv;
}

// Output-channel tile: the largest multiple of 32 up to 256 that divides 3C (C is a
// multiple of 32, so 96 always qualifies).
static int qkv_tile(int N) {
  for (int nt = kMaxNT; nt >= 32; nt -= 32)
    if (N % nt == 0) return nt;
  return 0;
}

cudaError_t qkv_proj_launch(const void* x, const float* gamma, const float* beta, const void* w, const float* b,
                            void* out, int T, int C, float eps, void* workspace, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % kKC != 0 || C < kKC || C > kMaxC) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const int N = 3 * C, NT = qkv_tile(N);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  __nv_bfloat16* wf = reinterpret_cast<__nv_bfloat16*>(ws);
  float* u = reinterpret_cast<float*>(ws + (((size_t)N * C * 2 + 255) & ~(size_t)255));
  float* v = u + ((((size_t)N * 4 + 255) & ~(size_t)255) / 4);
  qkv_fold_kernel<<<(N + 7) / 8, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(w), gamma, beta, b, C, N, wf,
                                               u, v);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap x_map, w_map;
  const cuuint32_t es[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {kKC, kBM};
    if (encode(&x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
    const cuuint32_t box[2] = {kKC, (cuuint32_t)NT};
    if (encode(&w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wf, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap out_map;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
    const cuuint32_t box[2] = {kKC, kBM};
    if (encode(&out_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  // Work items: token tiles times groups of output-channel tiles, at least four per SM
  // when the channel tiles allow it; one persistent CTA per SM walks them.
  const int n_tt = (T + kBM - 1) / kBM, n_tiles = N / NT;
  int groups = (4 * sms + n_tt - 1) / n_tt;
  groups = groups < 1 ? 1 : (groups > n_tiles ? n_tiles : groups);
  const int per = (n_tiles + groups - 1) / groups;
  groups = (n_tiles + per - 1) / per;
  const int n_items = n_tt * groups;
  QkvParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.u = u;
  p.v = v;
  p.status = status;
  p.T = T;
  p.C = C;
  p.N = N;
  p.NT = NT;
  p.tiles_per_item = per;
  p.n_tt = n_tt;
  p.n_items = n_items;
  p.eps = eps;
  return launch_pdl(qkv_gemm_kernel, dim3(n_items < sms ? n_items : sms), dim3(kTHREADS), kSMEM, st, x_map, w_map,
                    out_map, p);
}

}  // namespace swin
