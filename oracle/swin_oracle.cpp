// Reference oracle for Swin (shifted-)window multi-head attention, fp64, CPU only.
//
// TEST INFRASTRUCTURE. This file is the slow, plain statement of what the GPU path
// computes. Only the test suite, the smoke check and the CPU-baseline leg of the bench
// load it. The library under swin_window_attention_gb300/ never links, includes or calls
// it, and it shares no code with that library.
//
// Sources, cited by page and section:
//  * NVIDIA "visual large-model training and inference optimisation" talk, full
//    transcript (uticex.com, article 1598), section 1 "Swin Transformer introduction":
//    attention only among the tokens of each non-overlapping window; a window shift to
//    bridge window borders; a relative position bias added to the attention logits.
//  * same transcript, section 2 "training optimisation": shift, partition and reverse
//    are pure index mappings (a roll, then a split into windows, and their inverses);
//    mask and bias enter the attention as tensors.
//  * same transcript, section 3 "inference optimisation": the bias lookup is done once,
//    ahead of the attention, as a dense per-head tensor.
//  * Baidu AIAK-Training talk (jxzklqfsx.com, article 743345), section 2, the fused
//    WindowAttention case: the module is two matrix products around a softmax; the
//    backward recomputes the forward's intermediates.
// The pages print no formula, listing or worked value for these steps. Where they are
// silent, the readings used are the plain ones, each stated at the function that takes
// it:
//  R1 roll direction: the rolled grid reads the original token at (y+s, x+s) mod (H, W).
//  R2 windows are taken row-major over (H/M, W/M); tokens row-major inside a window.
//  R3 qkv channel c of a token is t*C + h*hd + d with t in {q, k, v}.
//  R4 output channel of a token is h*hd + d.
//  R5 relative index of local positions i=(yi,xi), j=(yj,xj) is
//     (yi-yj+M-1)*(2M-1) + (xi-xj+M-1), a row of the [(2M-1)^2, nH] table.
//  R6 shift-mask regions per axis of length L on the rolled grid: [0, L-M), [L-M, L-s),
//     [L-s, L); label = 3*region_y + region_x; a pair with different labels gets -100,
//     added to the logit.
//  R7 logit = scale*(q.k) + bias + mask, scale = hd^-0.5.
//
// The producer step in front of the attention (the LayerNorm and the qkv projection that
// the NVIDIA talk's section 2 lists among the fused operations of a Swin block) follows the
// plain definitions:
//  R15 LayerNorm over the C channels of a token: population variance, eps inside the
//      square root, then the per-channel affine gamma, beta.
//  R16 qkv = LN(x) W^T + b with W [3C, C] (row n is output channel n, in the channel order
//      of R3) and b [3C].
//
// The consumer step after the attention (the output projection followed by the bias and
// residual addition that the NVIDIA talk's section 3 "inference optimisation" fuses into one
// elementwise pass, its half2 example) also follows the plain definition:
//  R18 y = residual + O Wp^T + bp, with O the attention output [T, C] (channel order of
//      R4), Wp [C, C] (row n is output channel n), bp [C], and the residual the block
//      input at the same token.
//
// Everything here runs in double precision on whatever values it is given. Inputs are
// expected to be the bf16-rounded values the GPU path also sees, widened to double.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

inline int64_t pos_mod(int64_t a, int64_t m) {
  int64_t r = a % m;
  return r < 0 ? r + m : r;
}

// R6: region of rolled coordinate c on an axis of length L.
inline int region_of(int c, int L, int M, int s) {
  if (c < L - M) return 0;
  if (c < L - s) return 1;
  return 2;
}

}  // namespace

extern "C" {

int oracle_max_threads() {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// Cyclic shift of a [B,H,W,Ch] grid (R1): out[b,y,x,:] = in[b,(y+s)%H,(x+s)%W,:].
void oracle_roll(const double* in, int B, int H, int W, int Ch, int s, double* out) {
  for (int b = 0; b < B; ++b)
    for (int y = 0; y < H; ++y)
      for (int x = 0; x < W; ++x) {
        const int64_t ys = pos_mod(y + s, H), xs = pos_mod(x + s, W);
        const double* src = in + (((int64_t)b * H + ys) * W + xs) * Ch;
        double* dst = out + (((int64_t)b * H + y) * W + x) * Ch;
        std::memcpy(dst, src, sizeof(double) * Ch);
      }
}

// Inverse of oracle_roll: out[b,y,x,:] = in[b,(y-s)%H,(x-s)%W,:].
void oracle_unroll(const double* in, int B, int H, int W, int Ch, int s, double* out) {
  oracle_roll(in, B, H, W, Ch, -s, out);
}

// Window partition (R2): [B,H,W,Ch] -> [B, nW, M*M, Ch].
void oracle_partition(const double* in, int B, int H, int W, int Ch, int M, double* out) {
  const int nWx = W / M, nWy = H / M, N = M * M;
  for (int b = 0; b < B; ++b)
    for (int wy = 0; wy < nWy; ++wy)
      for (int wx = 0; wx < nWx; ++wx)
        for (int t = 0; t < N; ++t) {
          const int y = wy * M + t / M, x = wx * M + t % M;
          const int64_t w = (int64_t)wy * nWx + wx;
          const double* src = in + (((int64_t)b * H + y) * W + x) * Ch;
          double* dst = out + (((int64_t)b * nWy * nWx + w) * N + t) * Ch;
          std::memcpy(dst, src, sizeof(double) * Ch);
        }
}

// Window reverse: [B, nW, M*M, Ch] -> [B,H,W,Ch], the inverse of oracle_partition.
void oracle_reverse(const double* in, int B, int H, int W, int Ch, int M, double* out) {
  const int nWx = W / M, nWy = H / M, N = M * M;
  for (int b = 0; b < B; ++b)
    for (int wy = 0; wy < nWy; ++wy)
      for (int wx = 0; wx < nWx; ++wx)
        for (int t = 0; t < N; ++t) {
          const int y = wy * M + t / M, x = wx * M + t % M;
          const int64_t w = (int64_t)wy * nWx + wx;
          const double* src = in + (((int64_t)b * nWy * nWx + w) * N + t) * Ch;
          double* dst = out + (((int64_t)b * H + y) * W + x) * Ch;
          std::memcpy(dst, src, sizeof(double) * Ch);
        }
}

// R5: [N, N] relative position index.
void oracle_relidx(int M, int32_t* out) {
  const int N = M * M;
  for (int i = 0; i < N; ++i)
    for (int j = 0; j < N; ++j) {
      const int yi = i / M, xi = i % M, yj = j / M, xj = j % M;
      out[(int64_t)i * N + j] = (yi - yj + M - 1) * (2 * M - 1) + (xi - xj + M - 1);
    }
}

// Dense per-head bias [nH, N, N] from the table [(2M-1)^2, nH] (the lookup done once).
void oracle_dense_bias(const double* table, int nH, int M, double* out) {
  const int N = M * M;
  std::vector<int32_t> idx((size_t)N * N);
  oracle_relidx(M, idx.data());
  for (int h = 0; h < nH; ++h)
    for (int64_t e = 0; e < (int64_t)N * N; ++e)
      out[(int64_t)h * N * N + e] = table[(int64_t)idx[e] * nH + h];
}

// R6: shift mask [nW, N, N], values 0 or -100. Built as the pages describe the
// operation: label the rolled grid, partition the labels into windows, compare.
void oracle_mask(int H, int W, int M, int s, double* out) {
  const int nWx = W / M, nWy = H / M, N = M * M;
  std::vector<double> label((size_t)H * W);
  for (int y = 0; y < H; ++y)
    for (int x = 0; x < W; ++x)
      label[(size_t)y * W + x] = 3 * region_of(y, H, M, s) + region_of(x, W, M, s);
  std::vector<double> lw((size_t)nWy * nWx * N);
  oracle_partition(label.data(), 1, H, W, 1, M, lw.data());
  for (int w = 0; w < nWy * nWx; ++w)
    for (int i = 0; i < N; ++i)
      for (int j = 0; j < N; ++j)
        out[((int64_t)w * N + i) * N + j] =
            (lw[(size_t)w * N + i] == lw[(size_t)w * N + j]) ? 0.0 : -100.0;
}

// Gather map [nW, N]: index y*W + x (in the original grid) of the token that window w,
// slot i reads, i.e. where roll then partition take it from.
void oracle_gather(int H, int W, int M, int s, int32_t* out) {
  const int nWx = W / M, nWy = H / M, N = M * M;
  std::vector<double> ids((size_t)H * W), rolled((size_t)H * W), win((size_t)H * W);
  for (int t = 0; t < H * W; ++t) ids[t] = t;
  oracle_roll(ids.data(), 1, H, W, 1, s, rolled.data());
  oracle_partition(rolled.data(), 1, H, W, 1, M, win.data());
  for (int64_t e = 0; e < (int64_t)nWy * nWx * N; ++e) out[e] = (int32_t)win[e];
}

// Attention probabilities of one (b, w, h) on an already rolled and partitioned
// qkv window block: P[i, j], rows summing to one.
static void window_probs(const double* xw /*[N, 3C] of this window*/, const double* dense_bias_h,
                         const double* mask_w /* or null */, int N, int C, int hd, int h,
                         double scale, double* P) {
  std::vector<double> srow(N);
  for (int i = 0; i < N; ++i) {
    const double* q = xw + (int64_t)i * 3 * C + h * hd;
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
      const double* k = xw + (int64_t)j * 3 * C + C + h * hd;
      double dot = 0.0;
      for (int d = 0; d < hd; ++d) dot += q[d] * k[d];
      double v = scale * dot + dense_bias_h[(int64_t)i * N + j];
      if (mask_w) v += mask_w[(int64_t)i * N + j];
      srow[j] = v;
      if (v > mx) mx = v;
    }
    double sum = 0.0;
    for (int j = 0; j < N; ++j) {
      srow[j] = std::exp(srow[j] - mx);
      sum += srow[j];
    }
    for (int j = 0; j < N; ++j) P[(int64_t)i * N + j] = srow[j] / sum;
  }
}

// Probabilities of one (b, w, h) from the original qkv: used to check row sums.
void oracle_probs(const double* qkv, const double* table, int B, int H, int W, int C, int nH,
                  int M, int s, int b, int w, int h, double* P) {
  const int N = M * M, hd = C / nH;
  std::vector<double> xr((size_t)H * W * 3 * C), xw((size_t)H * W * 3 * C);
  oracle_roll(qkv + (int64_t)b * H * W * 3 * C, 1, H, W, 3 * C, s, xr.data());
  oracle_partition(xr.data(), 1, H, W, 3 * C, M, xw.data());
  std::vector<double> db((size_t)nH * N * N), mask;
  oracle_dense_bias(table, nH, M, db.data());
  if (s > 0) {
    mask.resize((size_t)(H / M) * (W / M) * N * N);
    oracle_mask(H, W, M, s, mask.data());
  }
  (void)B;
  window_probs(xw.data() + (int64_t)w * N * 3 * C, db.data() + (int64_t)h * N * N,
               s > 0 ? mask.data() + (int64_t)w * N * N : nullptr, N, C, hd, h,
               1.0 / std::sqrt((double)hd), P);
}

// Forward: qkv [B,H,W,3C] -> Y [B,H,W,C]. Steps in the pages' order: roll, partition,
// per-window attention with bias and mask, reverse, un-roll.
void oracle_fwd(const double* qkv, const double* table, int B, int H, int W, int C, int nH,
                int M, int s, double* Y) {
  const int N = M * M, hd = C / nH, nW = (H / M) * (W / M);
  const double scale = 1.0 / std::sqrt((double)hd);
  const size_t n3 = (size_t)B * H * W * 3 * C, n1 = (size_t)B * H * W * C;
  std::vector<double> xr(n3), xw(n3), ow(n1), yr(n1);
  oracle_roll(qkv, B, H, W, 3 * C, s, xr.data());
  oracle_partition(xr.data(), B, H, W, 3 * C, M, xw.data());
  std::vector<double> db((size_t)nH * N * N), mask;
  oracle_dense_bias(table, nH, M, db.data());
  if (s > 0) {
    mask.resize((size_t)nW * N * N);
    oracle_mask(H, W, M, s, mask.data());
  }
  const int64_t units = (int64_t)B * nW * nH;
#pragma omp parallel
  {
    std::vector<double> P((size_t)N * N);
#pragma omp for schedule(dynamic, 4)
    for (int64_t u = 0; u < units; ++u) {
      const int h = (int)(u % nH);
      const int64_t bw = u / nH;  // b * nW + w
      const int w = (int)(bw % nW);
      const double* x = xw.data() + bw * N * 3 * C;
      window_probs(x, db.data() + (int64_t)h * N * N,
                   s > 0 ? mask.data() + (int64_t)w * N * N : nullptr, N, C, hd, h, scale,
                   P.data());
      for (int i = 0; i < N; ++i) {
        double* o = ow.data() + (bw * N + i) * C + h * hd;
        for (int d = 0; d < hd; ++d) o[d] = 0.0;
        for (int j = 0; j < N; ++j) {
          const double p = P[(int64_t)i * N + j];
          const double* v = x + (int64_t)j * 3 * C + 2 * C + h * hd;
          for (int d = 0; d < hd; ++d) o[d] += p * v[d];
        }
      }
    }
  }
  oracle_reverse(ow.data(), B, H, W, C, M, yr.data());
  oracle_unroll(yr.data(), B, H, W, C, s, Y);
}

// Backward of oracle_fwd for the upstream gradient dY [B,H,W,C]:
//   dqkv [B,H,W,3C] (overwritten) and dtable [(2M-1)^2, nH] (overwritten).
// The chain per (b, w, h): P from the recomputed logits, dV = P^T dO, dP = dO V^T,
// D_i = sum_j P_ij dP_ij, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q, and
// dtable[idx(i,j), h] collects dS_ij over every b, w, i, j. The mask is constant.
void oracle_bwd(const double* qkv, const double* dY, const double* table, int B, int H, int W,
                int C, int nH, int M, int s, double* dqkv, double* dtable) {
  const int N = M * M, hd = C / nH, nW = (H / M) * (W / M), R = (2 * M - 1) * (2 * M - 1);
  const double scale = 1.0 / std::sqrt((double)hd);
  const size_t n3 = (size_t)B * H * W * 3 * C, n1 = (size_t)B * H * W * C;
  std::vector<double> xr(n3), xw(n3), dyr(n1), dyw(n1), dxw(n3, 0.0), dxr(n3);
  oracle_roll(qkv, B, H, W, 3 * C, s, xr.data());
  oracle_partition(xr.data(), B, H, W, 3 * C, M, xw.data());
  oracle_roll(dY, B, H, W, C, s, dyr.data());
  oracle_partition(dyr.data(), B, H, W, C, M, dyw.data());
  std::vector<double> db((size_t)nH * N * N), mask;
  oracle_dense_bias(table, nH, M, db.data());
  if (s > 0) {
    mask.resize((size_t)nW * N * N);
    oracle_mask(H, W, M, s, mask.data());
  }
  std::vector<int32_t> idx((size_t)N * N);
  oracle_relidx(M, idx.data());
  const int64_t units = (int64_t)B * nW * nH;
  std::vector<double> dt_unit((size_t)units * R, 0.0);
#pragma omp parallel
  {
    std::vector<double> P((size_t)N * N), dP((size_t)N * N);
#pragma omp for schedule(dynamic, 4)
    for (int64_t u = 0; u < units; ++u) {
      const int h = (int)(u % nH);
      const int64_t bw = u / nH;
      const int w = (int)(bw % nW);
      const double* x = xw.data() + bw * N * 3 * C;
      const double* dO = dyw.data() + bw * N * C;
      double* dx = dxw.data() + bw * N * 3 * C;
      window_probs(x, db.data() + (int64_t)h * N * N,
                   s > 0 ? mask.data() + (int64_t)w * N * N : nullptr, N, C, hd, h, scale,
                   P.data());
      // dP_ij = dO_i . v_j
      for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
          const double* v = x + (int64_t)j * 3 * C + 2 * C + h * hd;
          const double* g = dO + (int64_t)i * C + h * hd;
          double acc = 0.0;
          for (int d = 0; d < hd; ++d) acc += g[d] * v[d];
          dP[(int64_t)i * N + j] = acc;
        }
      // dV_j = sum_i P_ij dO_i
      for (int j = 0; j < N; ++j) {
        double* dv = dx + (int64_t)j * 3 * C + 2 * C + h * hd;
        for (int i = 0; i < N; ++i) {
          const double p = P[(int64_t)i * N + j];
          const double* g = dO + (int64_t)i * C + h * hd;
          for (int d = 0; d < hd; ++d) dv[d] += p * g[d];
        }
      }
      // dS = P o (dP - D); reuse dP's storage for dS.
      for (int i = 0; i < N; ++i) {
        double D = 0.0;
        for (int j = 0; j < N; ++j) D += P[(int64_t)i * N + j] * dP[(int64_t)i * N + j];
        for (int j = 0; j < N; ++j)
          dP[(int64_t)i * N + j] = P[(int64_t)i * N + j] * (dP[(int64_t)i * N + j] - D);
      }
      const double* dS = dP.data();
      double* dt = dt_unit.data() + u * R;
      for (int64_t e = 0; e < (int64_t)N * N; ++e) dt[idx[e]] += dS[e];
      // dQ_i = scale sum_j dS_ij k_j ; dK_j = scale sum_i dS_ij q_i
      for (int i = 0; i < N; ++i) {
        double* dq = dx + (int64_t)i * 3 * C + h * hd;
        const double* q = x + (int64_t)i * 3 * C + h * hd;
        for (int j = 0; j < N; ++j) {
          const double g = scale * dS[(int64_t)i * N + j];
          const double* k = x + (int64_t)j * 3 * C + C + h * hd;
          double* dk = dx + (int64_t)j * 3 * C + C + h * hd;
          for (int d = 0; d < hd; ++d) {
            dq[d] += g * k[d];
            dk[d] += g * q[d];
          }
        }
      }
    }
  }
  // dtable: units summed in a fixed order, independent of the thread count.
  for (int r = 0; r < R; ++r)
    for (int h = 0; h < nH; ++h) dtable[(int64_t)r * nH + h] = 0.0;
  for (int64_t u = 0; u < units; ++u) {
    const int h = (int)(u % nH);
    for (int r = 0; r < R; ++r) dtable[(int64_t)r * nH + h] += dt_unit[(size_t)u * R + r];
  }
  // Adjoint of partition then roll is reverse then un-roll.
  oracle_reverse(dxw.data(), B, H, W, 3 * C, M, dxr.data());
  oracle_unroll(dxr.data(), B, H, W, 3 * C, s, dqkv);
}

// R15, R16: qkv[t] = LN(x[t]) W^T + b for tokens t < T; x [T, C], W [3C, C], b [3C],
// gamma and beta [C].
void oracle_qkv_proj(const double* x, const double* gamma, const double* beta, const double* w,
                     const double* b, int T, int C, double eps, double* qkv) {
  const int N = 3 * C;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double* xr = x + t * C;
    double mean = 0.0;
    for (int c = 0; c < C; ++c) mean += xr[c];
    mean /= C;
    double var = 0.0;
    for (int c = 0; c < C; ++c) var += (xr[c] - mean) * (xr[c] - mean);
    var /= C;
    const double rstd = 1.0 / std::sqrt(var + eps);
    std::vector<double> xn(C);
    for (int c = 0; c < C; ++c) xn[c] = (xr[c] - mean) * rstd * gamma[c] + beta[c];
    for (int n = 0; n < N; ++n) {
      const double* wr = w + (int64_t)n * C;
      double acc = b[n];
      for (int c = 0; c < C; ++c) acc += xn[c] * wr[c];
      qkv[t * N + n] = acc;
    }
  }
}

// R18: y[t] = residual[t] + O[t] Wp^T + bp for tokens t < T; O, residual, y [T, C],
// Wp [C, C], bp [C].
void oracle_proj_residual(const double* o, const double* wp, const double* bp, const double* residual, int T,
                          int C, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double* orow = o + t * C;
    for (int n = 0; n < C; ++n) {
      const double* wr = wp + (int64_t)n * C;
      double acc = 0.0;
      for (int c = 0; c < C; ++c) acc += orow[c] * wr[c];
      y[t * C + n] = residual[t * C + n] + (acc + bp[n]);
    }
  }
}

}  // extern "C"
