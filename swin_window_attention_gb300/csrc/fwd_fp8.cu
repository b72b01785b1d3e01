// Fused (shifted-)window attention forward on 8-bit operands, 7x7 windows.
//
// The pages take the Swin GEMMs to low precision for inference (NVIDIA Swin talk
// transcript, uticex.com article 1598, section 3: INT8 with PTQ or QAT); here the same
// direction is applied to the attention's own operands. q, k and v arrive as OCP FP8 E4M3
// values with one scale per tensor (q = sq q8, k = sk k8, v = sv v8), so the qkv tensor
// is 3C bytes per token instead of 6C. The arithmetic after decoding is that of the bf16
// forward (fwd.cu), applied to the decoded values:
// * S = Q8 K8^T on the 8-bit tensor-core MMA (m16n8k32 e4m3: products exact in fp32,
//   fp32 accumulation), the accumulator seeded with bias / (scale sq sk) (the head's bias
//   fragments rescaled once per CTA in shared memory) and the shift mask
//   added as the same rank-4 bf16 MMA with its -100 rescaled by 1 / (sq sk);
// * P = softmax(scale sq sk S) in fp32, rounded to fp16 (11 significant bits);
// * O = P V8 on the fp16 MMA after V8 is widened to fp16 in shared memory (exact), with
//   the row sums of the same fp16 P from a ones tile; out = sv O / rowsum, bf16.
// The shift, partition, reverse and un-roll are the addressing of the bf16 forward.
#include <cuda_fp16.h>

#include "common.cuh"

namespace swin {

namespace {

struct Fp8Params {
  const unsigned char* qkv;   // [B, H, W, 3C] e4m3
  __nv_bfloat16* out;         // [B, H, W, C]
  const float4* bias_frag;    // plan fragments [nH][WARPS][NT][32] (bias / scale)
  const uint32_t* mask_frag;  // plan boundary-class mask V fragments, or null
  int H, W, C, nH, s, nWy, nWx, nW;
  int64_t total_windows;  // B * nW
  int chunks;             // window ranges per head
  float inv_sqsk;         // 1 / (sq sk)
  float c_l2;             // scale sq sk log2(e)
  float sv;
  uint32_t mask_u;        // bf16 bits of -100 / (sq sk)
  int* err;
};

constexpr int kM = 7;
using G7 = Geo<kM>;
constexpr int kRows = G7::NPAD;            // 64 rows per tile
constexpr int kT8 = kRows * 32;            // an 8-bit tile: 32 bytes per row
constexpr int kStage8 = 3 * kT8;           // q8, k8, v8
constexpr int kStages8 = 3;
constexpr int kV16 = kRows * 64;           // v widened to fp16 (the bf16 tile layout)
constexpr int kStg = G7::WARPS * 16 * 64;  // per-warp output staging, 16 rows x 64 bytes
constexpr int kSmem8 = G7::BIAS_BYTES + G7::MASK_BYTES + kStages8 * kStage8 + kV16 + kStg;

// Byte offset of 16-byte chunk c (0, 1) of row r in an 8-bit tile, XOR-swizzled so that
// the 8 rows of an ldmatrix phase hit distinct banks.
__device__ __forceinline__ uint32_t tile8_off(int r, int c) {
  return (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
}

// D = A(16x32 e4m3, row) * B(32x8 e4m3, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_e4m3_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_8(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  ldsm_x4(addr, r0, r1, r2, r3);  // 8x8 b16 matrices: 8 rows of 16 bytes, any element type
}

// Two fp32 -> packed f16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four e4m3 values (bytes 0..3 of w) -> two f16x2 words (exact).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__global__ void __launch_bounds__(G7::THREADS, 5) fwd_fp8_kernel(const Fp8Params p) {
  constexpr int N = G7::N, NT = G7::NT, KT = G7::KT, THREADS = G7::THREADS;
  extern __shared__ __align__(128) unsigned char smem[];
  pdl_launch_dependents();
  pdl_wait();
  float4* sbias = reinterpret_cast<float4*>(smem);
  uint32_t* smask = reinterpret_cast<uint32_t*>(smem + G7::BIAS_BYTES);
  unsigned char* stiles = smem + G7::BIAS_BYTES + G7::MASK_BYTES;
  unsigned char* sv16 = stiles + kStages8 * kStage8;
  unsigned char* sstg = sv16 + kV16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int h = blockIdx.x % p.nH;
  const int chunk = blockIdx.x / p.nH;
  const int64_t w_begin = p.total_windows * chunk / p.chunks;
  const int nwin = (int)(p.total_windows * (chunk + 1) / p.chunks - w_begin);
  const int C3 = 3 * p.C, H = p.H, W = p.W, s = p.s;

  // This thread's gather slot (the same for q, k and v): 16-byte chunk c of window slot i.
  constexpr int TCH = N * 2;  // chunks per tensor
  const bool has_slot = tid < TCH;
  const int slot_i = has_slot ? tid >> 1 : 0, slot_c = tid & 1;
  const uint32_t ld_soff = tile8_off(slot_i, slot_c);
  const int ld_ly = slot_i / kM, ld_lx = slot_i % kM, ld_chan = h * kHeadDim + slot_c * 16;

  int lb, lwy, lwx;  // cursor of the next window to load
  {
    lb = (int)(w_begin / p.nW);
    const int w = (int)(w_begin - (int64_t)lb * p.nW);
    lwy = w / p.nWx;
    lwx = w - lwy * p.nWx;
  }
  int cb = lb, cwy = lwy, cwx = lwx;  // cursor of the window being computed
  const uint32_t tiles_u32 = smem_u32(stiles);

  auto issue = [&](uint32_t stage_off) {
    if (has_slot) {
      const int y0 = lwy * kM + s, x0 = lwx * kM + s;
      int64_t rel = (int64_t)ld_ly * W + ld_lx;  // token offset from the window's first token
      if (ld_ly >= H - y0) rel -= (int64_t)H * W;
      if (ld_lx >= W - x0) rel -= W;
      const unsigned char* src = p.qkv + ((((int64_t)lb * H + y0) * W + x0) + rel) * C3 + ld_chan;
#pragma unroll
      for (int tt = 0; tt < 3; ++tt) cp_async_16(tiles_u32 + stage_off + tt * kT8 + ld_soff, src + tt * p.C);
    }
    if (++lwx == p.nWx) {
      lwx = 0;
      if (++lwy == p.nWy) {
        lwy = 0;
        ++lb;
      }
    }
  };

  // This head's bias fragments and the class mask fragments travel with window 0.
  {
    const unsigned char* bsrc = reinterpret_cast<const unsigned char*>(p.bias_frag) + (size_t)h * G7::BIAS_BYTES;
    for (int e = tid; e < G7::BIAS_BYTES / 16; e += THREADS) cp_async_16(smem_u32(smem + e * 16), bsrc + e * 16);
    if (p.mask_frag != nullptr) {
      const unsigned char* msrc = reinterpret_cast<const unsigned char*>(p.mask_frag);
      for (int e = tid; e < G7::MASK_BYTES / 16; e += THREADS)
        cp_async_16(smem_u32(smem + G7::BIAS_BYTES + e * 16), msrc + e * 16);
    }
  }
#pragma unroll
  for (int st = 0; st < kStages8 - 1; ++st) {
    if (st < nwin) issue(st * kStage8);
    cp_async_commit();
  }
  // Padded rows N..NPAD-1 of every 8-bit tile are zero (loads never touch them).
  for (int e = tid; e < kStages8 * 3 * (kRows - N) * 2; e += THREADS) {
    const int c = e & 1, r = (e >> 1) % (kRows - N), tile = (e >> 1) / (kRows - N);
    *reinterpret_cast<uint4*>(stiles + tile * kT8 + tile8_off(N + r, c)) = make_uint4(0u, 0u, 0u, 0u);
  }

  const float4* bfrag = sbias + warp * NT * 32 + lane;
  const float r_sc = p.inv_sqsk, c_l2 = p.c_l2;
  const int os0 = warp * 16 + g, os1 = os0 + 8;
  const int oly0 = os0 / kM, olx0 = os0 % kM, oly1 = os1 / kM, olx1 = os1 % kM;
  // U operand of the shift-mask MMA with -100 / (sq sk) in place of -100.
  uint32_t mu0, mu1;
  {
    const uint32_t u0 = mask_u_frag(os0, t, kM, s), u1 = mask_u_frag(os1, t, kM, s);
    const uint32_t lo = p.mask_u, hi = p.mask_u << 16;
    mu0 = ((u0 & 0xffffu) ? lo : 0u) | ((u0 >> 16) ? hi : 0u);
    mu1 = ((u1 & 0xffffu) ? lo : 0u) | ((u1 >> 16) ? hi : 0u);
  }
  const uint32_t ones = 0x3C003C00u;  // f16 1.0, 1.0
  // ldmatrix lane parts: Q (A of m16n8k32: rows 0-7 / 8-15 x bytes 0-15 / 16-31), K (B of
  // two key tiles: keys 0-7 of tile 2i / 2i+1 x bytes 0-15 / 16-31), V16 as in fwd.cu.
  const int mi = lane >> 3, r8 = lane & 7, r16 = r8 + ((mi & 1) << 3);
  const uint32_t q_off = tile8_off(warp * 16 + ((mi & 1) << 3) + r8, mi >> 1);
  const int k_row = ((mi >> 1) << 3) + r8, k_chk = mi & 1;
  const uint32_t v_off0 = tile_off(r16, mi >> 1), v_off1 = tile_off(r16, 2 + (mi >> 1));
  const uint32_t st_off0 = tile_off(r8 + ((mi & 1) << 3), mi >> 1);
  const uint32_t st_off1 = tile_off(r8 + ((mi & 1) << 3), 2 + (mi >> 1));
  unsigned char* wstg = sstg + warp * (16 * 64);

  uint32_t cur_off = 0, nxt_off = (kStages8 - 1) * kStage8;
  for (int it = 0; it < nwin; ++it) {
    cp_async_wait<kStages8 - 2>();
    __syncthreads();  // this window's tiles are in; every warp is done with the last one
    if (it == 0) {
      // the head's bias fragments (bias / scale) to accumulator units, once per CTA
      for (int e = tid; e < G7::BIAS_BYTES / 16; e += THREADS) {
        const float4 v = sbias[e];
        sbias[e] = make_float4(v.x * r_sc, v.y * r_sc, v.z * r_sc, v.w * r_sc);
      }
      __syncthreads();
    }
    if (it + kStages8 - 1 < nwin) issue(nxt_off);
    cp_async_commit();
    nxt_off = nxt_off + kStage8 == kStages8 * kStage8 ? 0 : nxt_off + kStage8;
    const int b = cb, wy = cwy, wx = cwx;
    if (++cwx == p.nWx) {
      cwx = 0;
      if (++cwy == p.nWy) {
        cwy = 0;
        ++cb;
      }
    }
    const uint32_t tb = tiles_u32 + cur_off;
    const unsigned char* v8 = stiles + cur_off + 2 * kT8;
    cur_off = cur_off + kStage8 == kStages8 * kStage8 ? 0 : cur_off + kStage8;

    // ---- v8 -> fp16 tile: one 16-byte chunk (16 channels of a key row) per thread ------
    {
      const int r = tid >> 1, c = tid & 1;  // 128 threads, 64 rows x 2 chunks
      const uint4 w = *reinterpret_cast<const uint4*>(v8 + tile8_off(r, c));
      uint32_t f[8];
      e4m3x4_to_f16(w.x, f[0], f[1]);
      e4m3x4_to_f16(w.y, f[2], f[3]);
      e4m3x4_to_f16(w.z, f[4], f[5]);
      e4m3x4_to_f16(w.w, f[6], f[7]);
      *reinterpret_cast<uint4*>(sv16 + tile_off(r, 2 * c)) = make_uint4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<uint4*>(sv16 + tile_off(r, 2 * c + 1)) = make_uint4(f[4], f[5], f[6], f[7]);
    }

    // ---- S = Q8 K8^T + bias / (scale sq sk) --------------------------------------------
    uint32_t qa0, qa1, qa2, qa3;
    ldsm_x4_8(tb + q_off, qa0, qa1, qa2, qa3);
    float sacc[NT][4];
#pragma unroll
    for (int np = 0; np < (NT + 1) / 2; ++np) {
      uint32_t b0, b1, b2, b3;  // key tiles 2np (b0, b1) and 2np + 1 (b2, b3)
      ldsm_x4_8(tb + kT8 + tile8_off(np * 16 + k_row, k_chk), b0, b1, b2, b3);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nt = 2 * np + u;
        if (nt < NT) {
          const float4 bb = bfrag[nt * 32];
          mma_e4m3_c(sacc[nt], qa0, qa1, qa2, qa3, u ? b2 : b0, u ? b3 : b1, bb.x, bb.y, bb.z, bb.w);
        }
      }
    }
    // ---- shift mask (boundary windows only) ------------------------------------------
    if (p.mask_frag != nullptr && (wy == p.nWy - 1 || wx == p.nWx - 1)) {
      const int cls = (wy == p.nWy - 1 ? 2 : 0) | (wx == p.nWx - 1 ? 1 : 0);
      const uint4* mv = reinterpret_cast<const uint4*>(smask) + (cls - 1) * (G7::NTP / 4) * 32 + lane;
#pragma unroll
      for (int q4 = 0; q4 < G7::NTP / 4; ++q4) {
        const uint4 v = mv[q4 * 32];
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (q4 * 4 + u < NT) mma_bf16(sacc[q4 * 4 + u], mu0, mu1, 0u, 0u, vw[u], 0u);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m0 = fmax3(m0, sacc[nt][0], sacc[nt][1]);
      m1 = fmax3(m1, sacc[nt][2], sacc[nt][3]);
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    const float2 c2 = make_float2(c_l2, c_l2);
    const float2 nm0 = make_float2(-m0 * c_l2, -m0 * c_l2), nm1 = make_float2(-m1 * c_l2, -m1 * c_l2);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float2 e0 = __ffma2_rn(make_float2(sacc[nt][0], sacc[nt][1]), c2, nm0);
      const float2 e1 = __ffma2_rn(make_float2(sacc[nt][2], sacc[nt][3]), c2, nm1);
      sacc[nt][0] = fast_exp2(e0.x);
      sacc[nt][1] = fast_exp2(e0.y);
      sacc[nt][2] = fast_exp2(e1.x);
      sacc[nt][3] = fast_exp2(e1.y);
    }
    __syncthreads();  // every thread's part of the fp16 v tile is in

    // ---- O = P V16, row sums from the ones tile ----------------------------------------
    float o[4][4], lsum[4];
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const uint32_t a0 = pack_f16(sacc[2 * kk][0], sacc[2 * kk][1]);
      const uint32_t a1 = pack_f16(sacc[2 * kk][2], sacc[2 * kk][3]);
      uint32_t a2 = 0u, a3 = 0u;
      if (2 * kk + 1 < NT) {
        a2 = pack_f16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        a3 = pack_f16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
      }
      uint32_t v0, v1, v2, v3, w0, w1, w2, w3;
      ldsm_x4_t(smem_u32(sv16) + v_off0 + kk * 1024, v0, v1, v2, v3);
      ldsm_x4_t(smem_u32(sv16) + v_off1 + kk * 1024, w0, w1, w2, w3);
      if (kk == 0) {
#pragma unroll
        for (int nd = 0; nd < 4; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.0f;
        lsum[0] = lsum[1] = lsum[2] = lsum[3] = 0.0f;
      }
      mma_f16(o[0], a0, a1, a2, a3, v0, v1);
      mma_f16(o[1], a0, a1, a2, a3, v2, v3);
      mma_f16(o[2], a0, a1, a2, a3, w0, w1);
      mma_f16(o[3], a0, a1, a2, a3, w2, w3);
      mma_f16(lsum, a0, a1, a2, a3, ones, ones);
    }

    // ---- normalise (x sv) and store at the gathered token positions -------------------
    const float inv0 = p.sv / lsum[0], inv1 = p.sv / lsum[2];
    const int y0 = wy * kM + s, x0 = wx * kM + s;
    int ya = y0 + oly0, xa = x0 + olx0, yb = y0 + oly1, xb = x0 + olx1;
    ya = ya >= H ? ya - H : ya;
    xa = xa >= W ? xa - W : xa;
    yb = yb >= H ? yb - H : yb;
    xb = xb >= W ? xb - W : xb;
    const int64_t img = (int64_t)b * H * W;
    const int64_t tok0 = img + ya * W + xa, tok1 = img + yb * W + xb;
    const float2 i0 = make_float2(inv0, inv0), i1 = make_float2(inv1, inv1);
    uint32_t ow[4][2];
#pragma unroll
    for (int nd = 0; nd < 4; ++nd) {
      const float2 a = __fmul2_rn(make_float2(o[nd][0], o[nd][1]), i0);
      const float2 c = __fmul2_rn(make_float2(o[nd][2], o[nd][3]), i1);
      ow[nd][0] = pack_bf16(a.x, a.y);
      ow[nd][1] = pack_bf16(c.x, c.y);
    }
    stsm_x4(smem_u32(wstg) + st_off0, ow[0][0], ow[0][1], ow[1][0], ow[1][1]);
    stsm_x4(smem_u32(wstg) + st_off1, ow[2][0], ow[2][1], ow[3][0], ow[3][1]);
    __syncwarp();
    __nv_bfloat16* outp = p.out + h * kHeadDim + t * 8;
    if (os0 < N) *reinterpret_cast<uint4*>(outp + tok0 * p.C) = *reinterpret_cast<const uint4*>(wstg + tile_off(g, t));
    if (os1 < N)
      *reinterpret_cast<uint4*>(outp + tok1 * p.C) = *reinterpret_cast<const uint4*>(wstg + tile_off(g + 8, t));
    __syncwarp();  // the staging rows are read before the next window overwrites them
  }
  cp_async_wait<0>();
}

}  // namespace

bool fwd_fp8_applies(const Plan& pl) { return pl.M == kM && pl.dtype == SWIN_WATTN_BF16; }

// One wave of CTAs: one head and a contiguous window range per CTA, as the bf16 forward.
cudaError_t fwd_fp8_launch(const Plan& pl, const void* qkv8, float sq, float sk, float sv, void* out,
                           cudaStream_t st) {
  if (!fwd_fp8_applies(pl)) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem8);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fwd_fp8_kernel, G7::THREADS, kSmem8);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t total = (int64_t)pl.B * pl.nW;
  int64_t chunks = ((int64_t)pl.num_sms * occ) / pl.nH;
  if (chunks < 1) chunks = 1;
  if (chunks > total) chunks = total;
  Fp8Params p;
  p.qkv = static_cast<const unsigned char*>(qkv8);
  p.out = static_cast<__nv_bfloat16*>(out);
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
  p.total_windows = total;
  p.chunks = (int)chunks;
  const float sqsk = sq * sk;
  p.inv_sqsk = 1.0f / sqsk;
  p.c_l2 = kLog2e / kInvScale * sqsk;
  p.sv = sv;
  p.mask_u = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(kMaskValue / sqsk));
  p.err = pl.err;
  return launch_pdl(fwd_fp8_kernel, dim3((unsigned)(chunks * pl.nH)), dim3(G7::THREADS), kSmem8, st, p);
}

}  // namespace swin
