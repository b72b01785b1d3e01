// The producer step in front of the attention: LayerNorm over the C channels of each
// token, then qkv = LN(x) W^T + b (W [3C, C] bf16, b [3C] fp32), written as the
// [tokens, 3C] bf16 tensor the attention reads. The NVIDIA Swin talk (uticex.com article
// 1598, section 2 "training optimisation") lists LayerNorm and the qkv GEMM among the
// operations fused around the window attention; the cyclic shift and the window
// partition that the talk fuses with them are already folded into the attention's
// loads here, so this kernel writes qkv in plain token order.
//
// A dense contraction (2 * 3C * C flops per token), so it runs on the fifth-generation
// tensor cores. A CTA owns 128 tokens (the MMA's M) and a range of output-channel tiles
// (N <= 256 each), with specialised warps:
// * copy warp (9): TMA loads of x chunks [128 tokens x 32 channels] and W chunks
//   [N tile x 32 channels], 64-byte swizzled, four stages deep;
// * normalising warps (0..3): thread r owns token row r: a first pass over its row in
//   global memory gives the mean and 1 / sqrt(var + eps) (fp32, two passes); then each x
//   chunk is turned into the bf16 A operand (x - mean) * rstd * gamma + beta in place
//   next to it, in the same swizzled layout;
// * MMA warp (8), one thread: per chunk two M128 N<=256 K16 tcgen05.mma into one of two
//   tensor-memory accumulators (N tile j uses columns 256 * (j & 1) onward);
// * epilogue warps (4..7): thread r (tensor-memory lane r) adds the bias, rounds to bf16
//   and stores its token's row of the N tile, while the next tile accumulates.
// Every wait is bounded (1 s); a wait that runs out sets the caller's status word (when
// one is given) and the CTA leaves after releasing its tensor memory.
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace swin {

namespace {

constexpr int kBM = 128;                       // tokens per CTA
constexpr int kKC = 32;                        // channels per K chunk: one 64-byte row
constexpr int kMaxNT = 256;                    // output channels per N tile
constexpr int kMaxC = 1536;
constexpr int kSTAGES = 4;
constexpr int kXCH = kBM * 64;                 // raw x chunk
constexpr int kACH = kBM * 64;                 // normalised A chunk
constexpr int kWCH = kMaxNT * 64;              // W chunk
constexpr int kSTAGE = kXCH + kACH + kWCH;     // 32 KB
constexpr int kTHREADS = 10 * 32;
constexpr int kEPI_WARP0 = 4, kMMA_WARP = 8, kCOPY_WARP = 9;
constexpr int kOFF_GB = kSTAGES * kSTAGE;              // gamma, beta: 2 x kMaxC floats
constexpr int kOFF_BIAS = kOFF_GB + 2 * kMaxC * 4;     // bias of the CTA's channel range
constexpr int kOFF_BAR = kOFF_BIAS + 3 * kMaxC * 4;
constexpr int kNBAR = 3 * kSTAGES + 4;
constexpr int kSMEM = kOFF_BAR + 8 * kNBAR + 8 + 1024;  // + alignment slack
constexpr int kTMEM_COLS = 512;                // two accumulators of up to 256 columns
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kSW64 = 4;

// More than half of the SM's shared memory: one CTA per SM, so the 512-column tensor
// memory allocation never waits.
static_assert(kSMEM > 233472 / 2, "one CTA per SM");

struct QkvParams {
  const __nv_bfloat16* x;  // [T, C], for the statistics pass
  __nv_bfloat16* out;      // [T, 3C]
  const float* gamma;
  const float* beta;
  const float* bias;
  int* status;  // optional: bit 0 set when a bounded wait ran out
  int T, C, N, NT, tiles_per_cta, n_tt;
  float eps;
};

__device__ __forceinline__ bool warp_wait(uint32_t mbar, uint32_t parity) {
  return __all_sync(0xffffffffu, tc::mbar_wait(mbar, parity, kWaitLimitNs)) != 0;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kTHREADS, 1)
    qkv_ln_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                       const QkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  pdl_launch_dependents();
  pdl_wait();
  const uint32_t smem0 = smem_u32(smem);
  float* sgamma = reinterpret_cast<float*>(smem + kOFF_GB);
  float* sbeta = sgamma + kMaxC;
  float* sbias = reinterpret_cast<float*>(smem + kOFF_BIAS);
  const uint32_t bar0 = smem0 + kOFF_BAR;
  auto full_bar = [&](int st) { return bar0 + 8 * st; };
  auto afull_bar = [&](int st) { return bar0 + 8 * (kSTAGES + st); };
  auto empty_bar = [&](int st) { return bar0 + 8 * (2 * kSTAGES + st); };
  auto dfull_bar = [&](int b) { return bar0 + 8 * (3 * kSTAGES + b); };
  auto dfree_bar = [&](int b) { return bar0 + 8 * (3 * kSTAGES + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOFF_BAR + 8 * kNBAR);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tt = blockIdx.x % p.n_tt, ng = blockIdx.x / p.n_tt;
  const int t0 = tt * kBM;
  const int n_tiles = p.N / p.NT;
  const int j0 = ng * p.tiles_per_cta;
  const int ntile = min(p.tiles_per_cta, n_tiles - j0);  // >= 1 by construction
  const int kcn = p.C / kKC;
  const int steps = ntile * kcn;

  if (warp == kMMA_WARP) tc::tmem_alloc<kTMEM_COLS>(smem_u32(tmem_slot));
  if (tid == 0) {
    for (int st = 0; st < kSTAGES; ++st) {
      tc::mbar_init(full_bar(st), 1);
      tc::mbar_init(afull_bar(st), 4);
      tc::mbar_init(empty_bar(st), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(dfull_bar(b), 1);
      tc::mbar_init(dfree_bar(b), 4);
    }
    tc::mbar_init_fence();
  }
  for (int c = tid; c < p.C; c += kTHREADS) {
    sgamma[c] = p.gamma[c];
    sbeta[c] = p.beta[c];
  }
  for (int c = tid; c < ntile * p.NT; c += kTHREADS) sbias[c] = p.bias[j0 * p.NT + c];
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int bad = 0;

  if (warp == kCOPY_WARP) {
    // ==== copies: x chunk and W chunk of step q into stage q % kSTAGES ===============
    if (lane == 0) {
      for (int q = 0, st = 0; q < steps; ++q) {
        if (q >= kSTAGES && !tc::mbar_wait(empty_bar(st), ((q / kSTAGES) - 1) & 1, kWaitLimitNs)) {
          bad = 1;
          break;
        }
        const int kc = q % kcn, n0 = (j0 + q / kcn) * p.NT;
        const uint32_t base = smem0 + st * kSTAGE;
        tc::mbar_expect_tx(full_bar(st), kXCH + p.NT * 64);
        tc::tile_load_2d(base, &x_map, kc * kKC, t0, full_bar(st));
        tc::tile_load_2d(base + kXCH + kACH, &w_map, kc * kKC, n0, full_bar(st));
        st = st + 1 == kSTAGES ? 0 : st + 1;
      }
    }
    __syncwarp();
  } else if (warp == kMMA_WARP) {
    // ==== MMA issue: one thread; the warp waits together ==============================
    const uint32_t idesc = tc::idesc_bf16(128, p.NT, false);
    for (int q = 0, st = 0; q < steps && !bad; ++q) {
      const int jj = q / kcn, kc = q % kcn, buf = jj & 1;
      if (kc == 0 && jj >= 2 && !warp_wait(dfree_bar(buf), ((jj >> 1) - 1) & 1)) {
        bad = 1;
        break;
      }
      if (!warp_wait(full_bar(st), (q / kSTAGES) & 1) || !warp_wait(afull_bar(st), (q / kSTAGES) & 1)) {
        bad = 1;
        break;
      }
      if (lane == 0) {
        tc::fence_after_sync();
        const uint32_t a = smem0 + st * kSTAGE + kXCH, w = a + kACH;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          tc::mma_ss(tmem + buf * kMaxNT, tc::sdesc(a + kk * 32, 16, 512, kSW64), tc::sdesc(w + kk * 32, 16, 512, kSW64),
                     idesc, kc > 0 || kk > 0);
        tc::commit(empty_bar(st));
        if (kc == kcn - 1) tc::commit(dfull_bar(buf));
      }
      __syncwarp();
      st = st + 1 == kSTAGES ? 0 : st + 1;
    }
  } else if (warp < kEPI_WARP0) {
    // ==== normalising warps: statistics of row r, then the A chunks ====================
    const int r = tid, t = t0 + r;
    float mean = 0.0f, rstd = 0.0f;
    if (t < p.T) {
      const uint4* xr = reinterpret_cast<const uint4*>(p.x + (int64_t)t * p.C);
      float s1 = 0.0f;
      for (int c = 0; c < p.C / 8; ++c) {
        const uint4 v = xr[c];
        s1 += bf16_lo(v.x) + bf16_hi(v.x) + bf16_lo(v.y) + bf16_hi(v.y) + bf16_lo(v.z) + bf16_hi(v.z) +
              bf16_lo(v.w) + bf16_hi(v.w);
      }
      mean = s1 / p.C;
      float s2 = 0.0f;
      for (int c = 0; c < p.C / 8; ++c) {
        const uint4 v = xr[c];
        const float e[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                            bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
#pragma unroll
        for (int u = 0; u < 8; ++u) s2 = fmaf(e[u] - mean, e[u] - mean, s2);
      }
      rstd = rsqrtf(s2 / p.C + p.eps);
    }
    const float2 rs2 = make_float2(rstd, rstd), nmr = make_float2(-mean * rstd, -mean * rstd);
    for (int q = 0, st = 0; q < steps; ++q) {
      if (!warp_wait(full_bar(st), (q / kSTAGES) & 1)) {
        bad = 1;
        break;
      }
      const int c0 = (q % kcn) * kKC;
      unsigned char* xc = smem + st * kSTAGE;
      unsigned char* ac = xc + kXCH;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t off = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
        const uint4 v = *reinterpret_cast<const uint4*>(xc + off);
        const float4 g0 = *reinterpret_cast<const float4*>(sgamma + c0 + 8 * c);
        const float4 g1 = *reinterpret_cast<const float4*>(sgamma + c0 + 8 * c + 4);
        const float4 b0 = *reinterpret_cast<const float4*>(sbeta + c0 + 8 * c);
        const float4 b1 = *reinterpret_cast<const float4*>(sbeta + c0 + 8 * c + 4);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // (x - mean) * rstd = x * rstd - mean * rstd, then * gamma + beta
          const float2 z = __ffma2_rn(make_float2(bf16_lo(in[u]), bf16_hi(in[u])), rs2, nmr);
          const float2 y = __ffma2_rn(z, make_float2(gg[2 * u], gg[2 * u + 1]), make_float2(bb[2 * u], bb[2 * u + 1]));
          o[u] = pack_bf16(y.x, y.y);
        }
        *reinterpret_cast<uint4*>(ac + off) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      tc::fence_proxy_async();  // the A chunk to the tensor core
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(afull_bar(st));
      st = st + 1 == kSTAGES ? 0 : st + 1;
    }
  } else {
    // ==== epilogue warps: bias, bf16, store (thread = tensor-memory lane = token row) ====
    const int r = (warp - kEPI_WARP0) * 32 + lane, t = t0 + r;
    const uint32_t trow = tmem + ((uint32_t)((warp - kEPI_WARP0) * 32) << 16);
    for (int jj = 0; jj < ntile; ++jj) {
      const int buf = jj & 1;
      if (!warp_wait(dfull_bar(buf), (jj >> 1) & 1)) {
        bad = 1;
        break;
      }
      tc::fence_after_sync();
      const int n0 = (j0 + jj) * p.NT;
      for (int c0 = 0; c0 < p.NT; c0 += 16) {
        uint32_t v[16];
        tc::ld16_wait(trow + buf * kMaxNT + c0, v);
        const float* bs = sbias + jj * p.NT + c0;
        uint32_t o[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float2 y = __fadd2_rn(make_float2(__uint_as_float(v[2 * u]), __uint_as_float(v[2 * u + 1])),
                                      make_float2(bs[2 * u], bs[2 * u + 1]));
          o[u] = pack_bf16(y.x, y.y);
        }
        if (t < p.T) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)t * p.N + n0 + c0);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(dfree_bar(buf));
    }
  }
  if (bad && p.status != nullptr) atomicOr(p.status, 1);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMMA_WARP) tc::tmem_dealloc<kTMEM_COLS>(tmem);
}

}  // namespace

// Output-channel tile: the largest multiple of 16 up to 256 that divides 3C (C is a
// multiple of 32, so 96 always qualifies).
static int qkv_tile(int N) {
  for (int nt = kMaxNT; nt >= 16; nt -= 16)
    if (N % nt == 0) return nt;
  return 0;
}

cudaError_t qkv_proj_launch(const void* x, const float* gamma, const float* beta, const void* w, const float* b,
                            void* out, int T, int C, float eps, int* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (C % kKC != 0 || C < kKC || C > kMaxC) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  const int N = 3 * C, NT = qkv_tile(N);
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
    if (encode(&w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(qkv_ln_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSMEM);
  if (e != cudaSuccess) return e;
  // Token tiles times groups of output-channel tiles, enough CTAs for every SM twice.
  const int n_tt = (T + kBM - 1) / kBM, n_tiles = N / NT;
  int groups = (2 * sms + n_tt - 1) / n_tt;
  groups = groups < 1 ? 1 : (groups > n_tiles ? n_tiles : groups);
  const int per = (n_tiles + groups - 1) / groups;
  groups = (n_tiles + per - 1) / per;
  QkvParams p;
  p.x = reinterpret_cast<const __nv_bfloat16*>(x);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.gamma = gamma;
  p.beta = beta;
  p.bias = b;
  p.status = status;
  p.T = T;
  p.C = C;
  p.N = N;
  p.NT = NT;
  p.tiles_per_cta = per;
  p.n_tt = n_tt;
  p.eps = eps;
  return launch_pdl(qkv_ln_gemm_kernel, dim3(n_tt * groups), dim3(kTHREADS), kSMEM, st, x_map, w_map, p);
}

}  // namespace swin
