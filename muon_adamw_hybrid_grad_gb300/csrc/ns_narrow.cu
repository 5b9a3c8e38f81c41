// Newton-Schulz of narrow Muon matrices in fp32 on the CUDA cores.
//
// OpenDM VLA training-stack article, 核心揭秘一 / Muon 的工作原理: the update
// G is normalised, X <- G / (||G||_F + eps), then taken through the quintic
// X <- a X + (b A + c A A) X with A = X X^T, on its short side, and applied as
// p <- p (1 - lr wd) - lr muon_lr_scale 0.2 sqrt(max(m, n)) X.
//
// With bf16 storage of X between iterations, the error of the result depends
// on where the normalised singular values start: those near 0.13-0.21 pass
// close to x = 1.2 in the third iteration, where the quintic's slope is about
// 4, and the rounding of X there is amplified to 2.3-2.7e-2 in Frobenius
// norm. A matrix whose short side s is small and whose update is noise-like
// has all its singular values near 1 / sqrt(s), which is that range for s of
// about 25 to 55. Matrices with s < 64 therefore take this kernel, which keeps
// X, A and B in fp32 throughout (an error near 1e-6). They are few and cheap:
// a 40 x 2000 matrix costs about 2e8 flops per step.
//
// One CTA (256 threads) per matrix, over the matrix list in a grid-stride
// loop. X lives in the matrix's fp32 workspace in the parameter's own layout
// (m x n, row-major): for m <= n the canonical X is that array, for m > n it
// is its transpose, which only changes the index arithmetic (A = U^T U and
// U' = U B for a tall U, since B is symmetric). A and B (s x s, padded to
// 64 x 64) are in shared memory; 64-column chunks of X pass through shared
// memory for each product, and X' = B X is written back in place chunk by
// chunk (a chunk of X' needs only the same chunk of X). Each thread holds a
// 4 x 4 block of every 64 x 64 result.
//
// The update G is recomputed from the momentum buffer that the momentum pass
// has just written and the gradient, with the same fp32 operations that pass
// uses (Nesterov: w coef g + mu buf), and the Frobenius scale r is folded in
// as the tensor-core path does: A of the first iteration is scaled by r^2 and
// its X' by r.
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ns_epilogue.cuh"

namespace ma {
namespace {

constexpr int kNarrowThreads = 256;
constexpr int SP = 64;       // padded short side
constexpr int CW = 64;       // columns of the long side per chunk
constexpr int LD = SP + 4;   // shared row pitch in floats (16-byte rows, fewer bank conflicts)

__device__ __forceinline__ float narrow_grad(const MuonMat& M, int64_t idx) {
  return M.gdtype == DT_BF16 ? __uint_as_float(((uint32_t) static_cast<const uint16_t*>(M.g)[idx]) << 16)
                             : static_cast<const float*>(M.g)[idx];
}

// Element (i, j) of the canonical X (i < s, j < l) in the parameter layout.
__device__ __forceinline__ int64_t canon_index(const MuonMat& M, int i, int j) {
  return M.transposed ? (int64_t)j * M.n + i : (int64_t)i * M.n + j;
}

// Chunk [j0, j0 + CW) of X into shared memory, zero outside the matrix.
// KMAJOR: T[jj][i] (for the Gram product); otherwise T[i][jj] (for B X).
// The global reads run along the parameter's rows in both cases.
template <bool KMAJOR>
__device__ __forceinline__ void load_chunk(const MuonMat& M, const float* X, int j0, float (*T)[LD]) {
  const int s = M.s, l = M.l;
  for (int e = threadIdx.x; e < SP * CW; e += kNarrowThreads) {
    int i, jj;
    if (M.transposed) {  // parameter row = j: consecutive threads take consecutive i
      i = e % SP;
      jj = e / SP;
    } else {  // parameter row = i: consecutive threads take consecutive j
      jj = e % CW;
      i = e / CW;
    }
    const int j = j0 + jj;
    const float v = (i < s && j < l) ? X[canon_index(M, i, j)] : 0.f;
    if (KMAJOR)
      T[jj][i] = v;
    else
      T[i][jj] = v;
  }
}

__device__ __forceinline__ double narrow_block_sum(double v, double* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double r = 0.0;
  for (int w = 0; w < kNarrowThreads / 32; ++w) r += sh[w];  // every thread, same order
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kNarrowThreads) ns_narrow_kernel(const __grid_constant__ NarrowLaunch L) {
  __shared__ __align__(16) float s0[SP][LD];  // A; the chunk of B X
  __shared__ __align__(16) float s1[SP][LD];  // the chunk of X X^T; B
  __shared__ double red[kNarrowThreads / 32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 4 x 4 block (rows 4 ty.., cols 4 tx..)
  const float coef = L.sc->coef * L.gscale;
  const float mu = L.mu;
  for (int mi = blockIdx.x; mi < L.nmat; mi += gridDim.x) {
    const MuonMat& M = L.mats[mi];
    float* const X = M.xf;
    const int s = M.s, l = M.l;
    const int64_t numel = (int64_t)M.m * M.n;
    // ---- the update G (as the momentum pass forms it) and ||G||_F ----
    double sq = 0.0;
    for (int64_t e = threadIdx.x; e < numel; e += kNarrowThreads) {
      const float gh = coef * narrow_grad(M, e);
      const float b = M.buf[e];
      const float u = L.nesterov ? fmaf(mu, b, gh) : b;
      X[e] = u;
      sq += (double)u * (double)u;
    }
    const double tot = narrow_block_sum(sq, red);  // also orders the writes of X before the reads below
    const float r = (float)(1.0 / (sqrt(tot) + (double)L.eps));
    for (int it = 0; it < L.steps; ++it) {
      const bool first = it == 0, last = it == L.steps - 1;
      const float ca = L.coef[it][0], cb = L.coef[it][1], cc = L.coef[it][2];
      // ---- A = X X^T (r^2 X X^T in the first iteration) ----
      float acc[4][4] = {};
      for (int j0 = 0; j0 < l; j0 += CW) {
        load_chunk<true>(M, X, j0, s1);
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < CW; ++jj) {
          const float4 a = *reinterpret_cast<const float4*>(&s1[jj][4 * ty]);
          const float4 b = *reinterpret_cast<const float4*>(&s1[jj][4 * tx]);
          const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
        }
        __syncthreads();
      }
      const float sa = first ? r * r : 1.f;
#pragma unroll
      for (int p = 0; p < 4; ++p)
        *reinterpret_cast<float4*>(&s0[4 * ty + p][4 * tx]) =
            make_float4(acc[p][0] * sa, acc[p][1] * sa, acc[p][2] * sa, acc[p][3] * sa);
      __syncthreads();
      // ---- B = a I + b A + c A A (A is symmetric: A[i][k] = A[k][i]) ----
      float aa[4][4] = {};
#pragma unroll 4
      for (int k = 0; k < SP; ++k) {
        const float4 a = *reinterpret_cast<const float4*>(&s0[k][4 * ty]);
        const float4 b = *reinterpret_cast<const float4*>(&s0[k][4 * tx]);
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) aa[p][q] = fmaf(av[p], bv[q], aa[p][q]);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = 4 * ty + p, k = 4 * tx + q;
          const float lin = fmaf(cb, s0[i][k], i == k ? ca : 0.f);
          o[q] = (i < s && k < s) ? fmaf(cc, aa[p][q], lin) : 0.f;
        }
        *reinterpret_cast<float4*>(&s1[4 * ty + p][4 * tx]) = make_float4(o[0], o[1], o[2], o[3]);
      }
      __syncthreads();
      // ---- X' = B X (r B X in the first iteration), chunk by chunk in place;
      // the last iteration applies it to the parameter instead ----
      const float sx = first ? r : 1.f;
      const float lrm = L.sp->ns_lr * M.lr_mult;
      const float dec = L.sp->ns_decay[M.group];
      for (int j0 = 0; j0 < l; j0 += CW) {
        load_chunk<false>(M, X, j0, s0);
        __syncthreads();
        float o[4][4] = {};
#pragma unroll 4
        for (int k = 0; k < SP; ++k) {
          const float4 b = *reinterpret_cast<const float4*>(&s1[k][4 * ty]);  // B[4 ty + p][k]
          const float4 x = *reinterpret_cast<const float4*>(&s0[k][4 * tx]);  // X[k][j0 + 4 tx + q]
          const float bv[4] = {b.x, b.y, b.z, b.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) o[p][q] = fmaf(bv[p], xv[q], o[p][q]);
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int i = 4 * ty + p;
          if (i >= s) continue;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = j0 + 4 * tx + q;
            if (j >= l) continue;
            const int64_t idx = canon_index(M, i, j);
            const float v = o[p][q] * sx;
            if (!last) {
              X[idx] = v;
            } else {
              const float pn = fmaf(M.p[idx], dec, -lrm * v);
              M.p[idx] = pn;
              if (M.shadow) M.shadow[idx] = ns_f2bf(pn);
            }
          }
        }
        __syncthreads();  // the chunk buffer is refilled next; X' is visible to the next Gram
      }
    }
  }
}

}  // namespace

cudaError_t launch_ns_narrow(const NarrowLaunch& L, int num_sms, cudaStream_t st) {
  const int grid = L.nmat < 4 * num_sms ? L.nmat : 4 * num_sms;
  if (grid <= 0) return cudaSuccess;
  ns_narrow_kernel<<<grid, kNarrowThreads, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace ma
