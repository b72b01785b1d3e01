// Preprocessing kernels: dense relative-position bias and shift mask, plus the debug
// dumps of the index maps.
//
// The bias lookup is moved out of the attention and done once (NVIDIA Swin talk
// transcript, uticex.com article 1598, section 3 "inference optimisation"); the mask
// and bias then reach the fused attention as tensors (same transcript, section 2).
#include "common.cuh"

namespace swin {

// mask[w, i, j] = 0 if the region labels of slots i and j of window w agree, else -100.
__global__ void build_mask_kernel(int H, int W, int M, int s, float* __restrict__ mask) {
  const int N = M * M, nWx = W / M, nW = (H / M) * nWx;
  const int64_t total = (int64_t)nW * N * N;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(e / ((int64_t)N * N));
    const int ij = (int)(e % ((int64_t)N * N));
    const int i = ij / N, j = ij % N;
    const int wy = w / nWx, wx = w % nWx;
    const int li = region_label(wy * M + i / M, wx * M + i % M, H, W, M, s);
    const int lj = region_label(wy * M + j / M, wx * M + j % M, H, W, M, s);
    mask[e] = (li == lj) ? 0.0f : kMaskValue;
  }
}

__global__ void gather_map_kernel(int H, int W, int M, int s, int32_t* __restrict__ out) {
  const int N = M * M, nWx = W / M, nW = (H / M) * nWx;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nW * N; e += gridDim.x * blockDim.x) {
    const int w = e / N, i = e % N;
    out[e] = (int32_t)gather_token(0, w / nWx, w % nWx, i, M, s, H, W);
  }
}

__global__ void relidx_kernel(int M, int32_t* __restrict__ out) {
  const int N = M * M;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < N * N; e += gridDim.x * blockDim.x)
    out[e] = rel_index(e / N, e % N, M);
}

// The bias in the order the attention kernels consume it (lane (g, t) of warp wp, key
// tile nt: rows 16wp+g, +8; columns 8nt+2t, +1), so that a CTA stages its head's block with
// plain 16-byte copies, read straight from the table (the same value the dense bias
// holds). It is stored divided by the softmax scale (it seeds the q.k accumulators), -inf
// in padded key columns and 0 in padded query rows. In the same launch: the shift-mask V
// fragments of the three boundary classes (mask_frag_word, from the region labels the
// dense mask uses), when mask_frag is given, and the dense bias
// dense[h, i, j] = table[idx(i, j), h], when dense is given.
template <int M>
__global__ void bias_tables_kernel(const float* __restrict__ table, int nH, int H, int W, int s,
                                   float4* __restrict__ bias_frag, uint32_t* __restrict__ mask_frag,
                                   float* __restrict__ dense) {
  using G = Geo<M>;
  constexpr int N = G::N, NT = G::NT;
  const int per_head = G::WARPS * NT * 32;
  const int64_t nbias = (int64_t)nH * per_head;
  const int64_t nmask = mask_frag ? G::MASK_BYTES / 4 : 0;
  const int64_t ndense = dense ? (int64_t)nH * N * N : 0;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nbias + nmask + ndense;
       e += (int64_t)gridDim.x * blockDim.x) {
    if (e < nbias) {
      const int h = (int)(e / per_head), f = (int)(e % per_head);
      const int ln = f & 31, nt = (f >> 5) % NT, wp = (f >> 5) / NT;
      const int r0 = wp * 16 + (ln >> 2), c0 = nt * 8 + 2 * (ln & 3);
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + 8 * (q >> 1), c = c0 + (q & 1);
        v[q] = c >= N ? -INFINITY : (r >= N ? 0.0f : table[(int64_t)rel_index(r, c, M) * nH + h] * kInvScale);
      }
      bias_frag[e] = make_float4(v[0], v[1], v[2], v[3]);
    } else if (e < nbias + nmask) {
      mask_frag[e - nbias] = mask_frag_word<M>((int)(e - nbias), H, W, s);
    } else {
      const int64_t d = e - nbias - nmask;
      const int h = (int)(d / (N * N)), ij = (int)(d % (N * N));
      dense[d] = table[(int64_t)rel_index(ij / N, ij % N, M) * nH + h];
    }
  }
}

static int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 4096) g = 4096;
  return (int)g;
}

cudaError_t launch_build_mask(int H, int W, int M, int s, float* mask, cudaStream_t st) {
  const int64_t n = (int64_t)(H / M) * (W / M) * M * M * M * M;
  build_mask_kernel<<<grid_for(n, 256), 256, 0, st>>>(H, W, M, s, mask);
  return cudaGetLastError();
}

size_t bias_frag_bytes(int M, int nH) {
  switch (M) {
    case 4: return (size_t)nH * Geo<4>::BIAS_BYTES;
    case 7: return (size_t)nH * Geo<7>::BIAS_BYTES;
    case 12: return (size_t)nH * Geo<12>::BIAS_BYTES;
    default: return 0;
  }
}

size_t mask_frag_bytes(int M) {
  switch (M) {
    case 4: return Geo<4>::MASK_BYTES;
    case 7: return Geo<7>::MASK_BYTES;
    case 12: return Geo<12>::MASK_BYTES;
    default: return 0;
  }
}

// Bias fragments from `table` for window size M, with the class mask fragments when
// `mask_frag` is given and the dense bias when `dense` is given: one launch.
cudaError_t launch_bias_frags(int M, const float* table, int nH, int H, int W, int s, float4* bias_frag,
                              uint32_t* mask_frag, float* dense, cudaStream_t st) {
  const int64_t n = (int64_t)bias_frag_bytes(M, nH) / 16 + (mask_frag ? mask_frag_bytes(M) / 4 : 0) +
                    (dense ? (int64_t)nH * M * M * M * M : 0);
  const int grid = grid_for(n, 256);
  switch (M) {
    case 4:
      bias_tables_kernel<4><<<grid, 256, 0, st>>>(table, nH, H, W, s, bias_frag, mask_frag, dense);
      break;
    case 7:
      bias_tables_kernel<7><<<grid, 256, 0, st>>>(table, nH, H, W, s, bias_frag, mask_frag, dense);
      break;
    case 12:
      bias_tables_kernel<12><<<grid, 256, 0, st>>>(table, nH, H, W, s, bias_frag, mask_frag, dense);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// The plan's bias fragments and dense bias from `table` [and its mask fragments], one
// launch.
cudaError_t launch_bias_tables(const Plan& p, const float* table, bool with_mask, cudaStream_t st) {
  uint32_t* mask = with_mask && p.s > 0 ? p.mask_frag : nullptr;
  return launch_bias_frags(p.M, table, p.nH, p.H, p.W, p.s, p.bias_frag, mask, p.dense_bias, st);
}

cudaError_t launch_gather_map(int H, int W, int M, int s, int32_t* out, cudaStream_t st) {
  gather_map_kernel<<<grid_for((int64_t)H * W, 256), 256, 0, st>>>(H, W, M, s, out);
  return cudaGetLastError();
}

cudaError_t launch_relidx(int M, int32_t* out, cudaStream_t st) {
  relidx_kernel<<<grid_for((int64_t)M * M * M * M, 256), 256, 0, st>>>(M, out);
  return cudaGetLastError();
}

}  // namespace swin
