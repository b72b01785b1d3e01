// Preprocessing kernels: dense relative-position bias and shift mask, plus the debug
// dumps of the index maps.
//
// The bias lookup is moved out of the attention and done once (NVIDIA Swin talk
// transcript, uticex.com article 1598, section 3 "inference optimisation"); the mask
// and bias then reach the fused attention as tensors (same transcript, section 2).
#include "common.cuh"

namespace swin {

// dense[h, i, j] = table[idx(i, j), h]
__global__ void expand_bias_kernel(const float* __restrict__ table, int nH, int M,
                                   float* __restrict__ dense) {
  const int N = M * M;
  const int64_t total = (int64_t)nH * N * N;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int h = (int)(e / ((int64_t)N * N));
    const int ij = (int)(e % ((int64_t)N * N));
    const int i = ij / N, j = ij % N;
    dense[e] = table[(int64_t)rel_index(i, j, M) * nH + h];
  }
}

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

static int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 4096) g = 4096;
  return (int)g;
}

cudaError_t launch_expand_bias(const float* table, int nH, int M, float* dense,
                               cudaStream_t st) {
  const int64_t n = (int64_t)nH * M * M * M * M;
  expand_bias_kernel<<<grid_for(n, 256), 256, 0, st>>>(table, nH, M, dense);
  return cudaGetLastError();
}

cudaError_t launch_build_mask(int H, int W, int M, int s, float* mask, cudaStream_t st) {
  const int64_t n = (int64_t)(H / M) * (W / M) * M * M * M * M;
  build_mask_kernel<<<grid_for(n, 256), 256, 0, st>>>(H, W, M, s, mask);
  return cudaGetLastError();
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
