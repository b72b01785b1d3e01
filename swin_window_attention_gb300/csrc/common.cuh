// Shared device helpers and the plan structure of the swin_wattn library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/swin_wattn.h"

namespace swin {

constexpr uint32_t kPlanMagic = 0x5357414eu;  // "SWAN"
constexpr int kHeadDim = 32;
constexpr float kMaskValue = -100.0f;
constexpr float kLog2e = 1.4426950408889634f;
// 1 / scale = sqrt(hd) for hd = 32: the kernels accumulate z = q.k + (bias + mask) / scale
// in the MMA, so that the logit is scale * z.
constexpr float kInvScale = 5.6568542494923802f;


struct Plan {
  uint32_t magic;
  int B, H, W, C, nH, M, s, dtype;
  int N, nWy, nWx, nW;
  int device;
  int num_sms;
  float* dense_bias;  // [nH, N, N], owned
  float* mask;        // [nW, N, N], owned; null when s == 0
  float* dt_partial;  // backward reduction scratch, owned
  int dt_partial_rows;
  // Per-head dense bias in the kernels' mma-fragment order, log2(e)-scaled, -inf in
  // padded key columns: [nH][WARPS][NT][32 lanes] float4. Owned.
  float4* bias_frag;
  // Shift-mask B fragments of the three boundary window classes (see mask_v_word):
  // [3 classes][NTP / 4][32 lanes][4] uint32. Owned; null when s == 0.
  uint32_t* mask_frag;
  // Constant operands of the tcgen05 forward (7x7 windows): mask U, class V and the bias
  // image per head. Owned; null for other window sizes.
  unsigned char* tc_tables;
  // The tables no longer match the bias (built lazily before the next tcgen05 forward).
  bool tc_stale;
  // Device error word written by kernels with bounded waits (bit 0: a wait ran out).
  // Owned.
  int* err;
  // Forward and backward kernel requests: SWIN_WATTN_KERNEL_AUTO, _MMA_SYNC or _TCGEN05.
  int fwd_kernel;
  int bwd_kernel;
};

// ---- bounded waits and the fault-injection build ---------------------------------
//
// Every device-side wait on an mbarrier gives up after wait_limit_ns() (1 s) and the
// kernel reports SWIN_WATTN_ERR_TIMEOUT through an error word. The fault-injection build
// (compiled with SWIN_WATTN_FAULT_INJECTION, libswin_wattn_debug.so) can shorten that
// limit and arm one site that withholds a single mbarrier arrival, so that one wait runs
// out and the error path runs; the default build contains no injection code and its
// fault site is always kFaultNone.
enum FaultSite { kFaultNone = 0, kFaultFwdMmaSync = 1, kFaultFwdTcgen05 = 2, kFaultGemm = 3 };
uint64_t wait_limit_ns();
int fault_site();

// ---- geometry shared by every kernel that touches a window -----------------------

// Original-grid token index (b*H + y)*W + x read by slot i of window w in batch b.
// Rolled (y, x) = (wy*M + i/M, wx*M + i%M) reads original ((y+s) mod H, (x+s) mod W).
__device__ __forceinline__ int64_t gather_token(int b, int wy, int wx, int i, int M, int s,
                                                int H, int W) {
  int y = wy * M + i / M + s;
  int x = wx * M + i % M + s;
  if (y >= H) y -= H;
  if (x >= W) x -= W;
  return ((int64_t)b * H + y) * W + x;
}

// Relative position index of local positions i, j in an M x M window.
__device__ __forceinline__ int rel_index(int i, int j, int M) {
  return (i / M - j / M + M - 1) * (2 * M - 1) + (i % M - j % M + M - 1);
}

// Shift-region label of a rolled coordinate pair (per axis [0,L-M), [L-M,L-s), [L-s,L)).
__device__ __forceinline__ int region_1d(int c, int L, int M, int s) {
  return c < L - M ? 0 : (c < L - s ? 1 : 2);
}
__device__ __forceinline__ int region_label(int ry, int rx, int H, int W, int M, int s) {
  return 3 * region_1d(ry, H, M, s) + region_1d(rx, W, M, s);
}

// ---- PTX wrappers ----------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// Every cp.async of this thread, committed to a group or not, has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + C with separate C inputs (no register copy to seed the accumulator).
__device__ __forceinline__ void mma_bf16_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1, float c0,
                                           float c1, float c2, float c3) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
        "f"(c3));
}

// Programmatic dependent launch: let the next kernel in the stream be scheduled (its
// CTAs take SMs as this kernel's CTAs leave), and wait until the previous kernel has
// completed and its memory is visible (a no-op when this kernel was launched without
// the programmatic attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Four 8x8 bf16 matrices from mma C-fragment pairs to shared rows (lanes 8i..8i+7 give
// the row addresses of matrix i).
__device__ __forceinline__ void stsm_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                        uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

__device__ __forceinline__ void stsm_x2(uint32_t addr, uint32_t r0, uint32_t r1) {
  asm volatile("stmatrix.sync.aligned.m8n8.x2.shared.b16 [%0], {%1,%2};\n" ::"r"(addr), "r"(r0),
               "r"(r1)
               : "memory");
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// a - b on a pair with one packed FFMA2 (a + (-1) * b).
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

// (a, b) = hi + lo with hi the bf16x2 rounding of (a, b) and lo the bf16x2 rounding of
// the residual: the pair carries ~16 significant bits of each value into a bf16 MMA.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  const float2 r = fsub2(make_float2(a, b), make_float2(__uint_as_float(hi << 16),
                                                                    __uint_as_float(hi & 0xffff0000u)));
  lo = pack_bf16(r.x, r.y);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk c (0..3) of row r in a [rows][32 x bf16] shared tile,
// XOR-swizzled so that 8 consecutive rows of one chunk column hit distinct banks.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// ---- window tiles -------------------------------------------------------------------

// Compile-time geometry of one window-head tile for window size M (hd = 32).
template <int M_>
struct Geo {
  static constexpr int M = M_;
  static constexpr int N = M * M;
  static constexpr int MT = (N + 15) / 16;  // query row tiles = warps per CTA
  static constexpr int NT = (N + 7) / 8;    // key n8 tiles of S
  static constexpr int KT = MT;             // k16 steps of P.V
  static constexpr int NPAD = MT * 16;      // rows of the shared q/k/v tiles
  static constexpr int WARPS = MT;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int NTP = (NT + 3) & ~3;      // key tiles rounded to whole uint4 loads
  static constexpr int CHUNKS = 3 * N * 4;       // 16-byte bf16 chunks per window-head
  static constexpr int CH_ITERS = (CHUNKS + THREADS - 1) / THREADS;
  static constexpr int TILE_BYTES = NPAD * 64;
  static constexpr int STAGE_BYTES = 3 * TILE_BYTES;
  static constexpr int BIAS_BYTES = WARPS * NT * 32 * 16;
  static constexpr int MASK_BYTES = 3 * NTP * 32 * 4;
  static_assert(NT * 8 <= NPAD, "key tiles must fit the padded tile");
};

// ---- the shift mask as one extra k16 MMA per key tile -------------------------------
//
// In a boundary window (class 1: last window column, 2: last window row, 3: both) slot
// i = (ly, lx) lies in the local region c(i) = 2 [ly >= M - s] + [lx >= M - s], and the
// region labels of query slot i and key slot j differ exactly when mism(c(i), j) does,
// where mism(c, j) compares j with any slot of region c. The mask in z units,
// -100 * sqrt(hd) * mism(c(i), j), is therefore the k16 product U V^T with
//   U[i][4e + c] = -100 * [c == c(i)],   V[j][4e + c] = part_e * mism(c, j),   e = 0, 1,
// part_0 = bf16(sqrt(hd)), part_1 = bf16(sqrt(hd) - part_0), and k-slots 8..15 zero. One
// c is set per row, so an accumulator receives -100 * (part_0 + part_1) (within 2e-4 of
// -100 * sqrt(hd); every product is exact in fp32) or nothing.
constexpr uint32_t kMaskUBits = 0xC2C8u;       // bf16 of -100
constexpr float kMaskPartHi = 5.65625f;        // bf16 of sqrt(32)
constexpr uint32_t kMaskPartHiBits = 0x40B5u;  // its bit pattern

// U fragment word of query row r for lane column t (k-slots 2t, 2t+1); zero for padding.
__device__ __forceinline__ uint32_t mask_u_frag(int r, int t, int M, int s) {
  if (r >= M * M) return 0u;
  const int c = ((r / M) >= M - s ? 2 : 0) | ((r % M) >= M - s ? 1 : 0);
  return (((2 * t) & 3) == c ? kMaskUBits : 0u) | (((2 * t + 1) & 3) == c ? kMaskUBits << 16 : 0u);
}

// mism(c, j) in a window of boundary class cls: do key slot j and the slots of local
// region c carry different region labels?
__device__ __forceinline__ bool mask_mismatch(int cls, int c, int j, int H, int W, int M, int s) {
  const int y0 = (cls & 2) ? (H / M - 1) * M : 0, x0 = (cls & 1) ? (W / M - 1) * M : 0;
  const int lj = region_label(y0 + j / M, x0 + j % M, H, W, M, s);
  const int lc = region_label(y0 + ((c & 2) ? M - 1 : 0), x0 + ((c & 1) ? M - 1 : 0), H, W, M, s);
  return lc != lj;
}

// bf16 bit pattern of V[j][k] (k < 8) for class cls; zero for padded keys.
__device__ __forceinline__ uint32_t mask_v_bits(int cls, int j, int k, int H, int W, int M, int s) {
  if (j >= M * M || k >= 8 || !mask_mismatch(cls, k & 3, j, H, W, M, s)) return 0u;
  return k < 4 ? kMaskPartHiBits : (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(kInvScale - kMaskPartHi));
}

// V fragment word (b0 of key tile nt: k-slots 2t, 2t+1 of key j = 8 nt + g) of class cls.
__device__ __forceinline__ uint32_t mask_v_word(int cls, int lane, int nt, int H, int W, int M, int s) {
  const int j = nt * 8 + (lane >> 2), t = lane & 3;
  return mask_v_bits(cls, j, 2 * t, H, W, M, s) | (mask_v_bits(cls, j, 2 * t + 1, H, W, M, s) << 16);
}

// Word e of the [3 classes][NTP / 4][32 lanes][4] mask fragment array.
template <int M>
__device__ __forceinline__ uint32_t mask_frag_word(int e, int H, int W, int s) {
  using G = Geo<M>;
  const int cls = 1 + e / (G::NTP * 32), r = e % (G::NTP * 32);
  const int nt = (r >> 7) * 4 + (r & 3), lane = (r >> 2) & 31;
  return nt < G::NT ? mask_v_word(cls, lane, nt, H, W, M, s) : 0u;
}

// One 16-byte bf16 chunk (8 channels) of a token's head slice into shared memory: a
// cp.async for bf16 sources; fp32 sources are read, rounded to bf16 (nearest even) and
// stored.
template <typename TIO>
__device__ __forceinline__ void load_chunk(uint32_t dst, const TIO* src);

template <>
__device__ __forceinline__ void load_chunk<__nv_bfloat16>(uint32_t dst, const __nv_bfloat16* src) {
  cp_async_16(dst, src);
}

template <>
__device__ __forceinline__ void load_chunk<float>(uint32_t dst, const float* src) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(src));
  const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
  const uint32_t w0 = pack_bf16(a.x, a.y), w1 = pack_bf16(a.z, a.w);
  const uint32_t w2 = pack_bf16(b.x, b.y), w3 = pack_bf16(b.z, b.w);
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst), "r"(w0), "r"(w1), "r"(w2),
               "r"(w3)
               : "memory");
}

// Launch `kernel` on `st` with programmatic stream serialisation: it may start while the
// previous kernel of the stream drains; it calls pdl_wait() before touching activations.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct FwdLaunch {
  int grid = 0, threads = 0, smem = 0, chunks = 0;
  int ctas_per_sm = 0;
  bool tc = false;   // the tcgen05 kernel (fwd_tc.cu) rather than the mma.sync one
  bool tma = false;  // mma.sync kernel: tiles by the copy engine (7x7 windows, bf16)
};
struct BwdLaunch {
  int grid = 0, threads = 0, smem = 0, chunks = 0, partial_rows = 0;
  bool tc = false;  // the tcgen05 kernel (bwd_tc.cu) rather than the mma.sync one
};

}  // namespace swin
