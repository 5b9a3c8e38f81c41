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
// loop; the host orders the list largest first. X lives in the matrix's fp32
// workspace in the parameter's own layout (m x n, row-major): for m <= n the
// canonical X is that array, for m > n it is its transpose, which only
// changes the index arithmetic (A = U^T U and U' = U B for a tall U, since B
// is symmetric). A and B (s x s, padded to 64 x 64) are in shared memory;
// 64-column chunks of X pass through shared memory for each product, and
// X' = B X is written back in place chunk by chunk (a chunk of X' needs only
// the same chunk of X).
//
// Latency: every chunk is fetched into registers (four 16-byte loads per
// thread where the layout allows) one chunk ahead, so the global loads of
// chunk c + 1 are in flight while chunk c is multiplied out of shared memory.
//
// Work split: thread (ty, tx) of the 16 x 16 grid holds rows ty + 16 p
// (p < 4) of each 64-row result. Rows interleave so that a short side s < 64
// leaves every warp with ceil((s - row) / 16) live row groups, the same count
// on all four schedulers; a warp skips the groups that lie wholly in the zero
// padding, and the Gram product also skips the column groups tx + 16 q >= s
// (the same for every thread). To read the four rows of a thread as one
// 16-byte word, the Gram chunk and B are stored with row i at position
// 4 (i mod 16) + i / 16.
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
constexpr int SP = 64;                                 // padded short side
constexpr int CW = 64;                                 // columns of the long side per chunk
constexpr int LD = SP + 4;                             // shared row pitch in floats (16-byte rows)
constexpr int QPT = SP * CW / 4 / kNarrowThreads;      // 4-float words of a chunk per thread
constexpr int UB = 8;                                  // elements in flight per thread forming G

__device__ __forceinline__ float narrow_grad(const MuonMat& M, int64_t idx) {
  return M.gdtype == DT_BF16 ? __uint_as_float(((uint32_t) static_cast<const uint16_t*>(M.g)[idx]) << 16)
                             : static_cast<const float*>(M.g)[idx];
}

// Element (i, j) of the canonical X (i < s, j < l) in the parameter layout.
__device__ __forceinline__ int64_t canon_index(const MuonMat& M, int i, int j) {
  return M.transposed ? (int64_t)j * M.n + i : (int64_t)i * M.n + j;
}

// Shared position of row i in the interleaved layouts.
__device__ __forceinline__ int perm_row(int i) { return 4 * (i & 15) + (i >> 4); }

// Word k of the thread's share of chunk [j0, j0 + CW): the 4 floats at
// (hi, lo..lo+3) of the chunk in memory order, where (hi, lo) is (i, jj) for a
// wide matrix (parameter rows are rows of X) and (jj, i) for a tall one
// (parameter rows are columns of X). Zero outside the matrix.
__device__ __forceinline__ void word_coords(int k, int& hi, int& lo) {
  const int q = threadIdx.x + k * kNarrowThreads;
  hi = q >> 4;
  lo = 4 * (q & 15);
}

__device__ __forceinline__ void fetch_chunk(const MuonMat& M, const float* X, int j0, float4 (&v)[QPT]) {
  const int s = M.s, l = M.l;
  // X starts 16-byte aligned (the host pads every slot); rows of X in memory
  // are l floats long for a wide matrix, s for a tall one
  const bool vec = M.transposed ? (s % 4 == 0) : (l % 4 == 0);
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    int hi, lo;
    word_coords(k, hi, lo);
    const int i0 = M.transposed ? lo : hi, j = M.transposed ? j0 + hi : j0 + lo;
    float f[4];
    if (M.transposed) {
      const float* src = X + (int64_t)j * s + i0;
      if (vec && j < l && i0 + 3 < s) {
        v[k] = *reinterpret_cast<const float4*>(src);
        continue;
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) f[t] = (j < l && i0 + t < s) ? src[t] : 0.f;
    } else {
      const float* src = X + (int64_t)i0 * l + j;
      if (vec && i0 < s && j + 3 < l) {
        v[k] = *reinterpret_cast<const float4*>(src);
        continue;
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) f[t] = (i0 < s && j + t < l) ? src[t] : 0.f;
    }
    v[k] = make_float4(f[0], f[1], f[2], f[3]);
  }
}

// The fetched chunk into shared memory. GRAM: T[jj][perm_row(i)] (the
// reduction index jj outer, rows interleaved); otherwise T[i][jj] (B X reduces
// over i).
template <bool GRAM>
__device__ __forceinline__ void store_chunk(const MuonMat& M, const float4 (&v)[QPT], float (*T)[LD]) {
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    int hi, lo;
    word_coords(k, hi, lo);
    const float f[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
    if (M.transposed) {  // (jj = hi, i = lo + t)
      if (GRAM) {
#pragma unroll
        for (int t = 0; t < 4; ++t) T[hi][perm_row(lo + t)] = f[t];
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) T[lo + t][hi] = f[t];
      }
    } else {  // (i = hi, jj = lo + t)
      if (GRAM) {
#pragma unroll
        for (int t = 0; t < 4; ++t) T[lo + t][perm_row(hi)] = f[t];
      } else {
        *reinterpret_cast<float4*>(&T[hi][lo]) = v[k];
      }
    }
  }
}

// acc[p][q] += sum over the chunk's columns of X[ty + 16 p][.] X[tx + 16 q][.]
// for p < NP, q < NQ.
template <int NP, int NQ>
__device__ __forceinline__ void gram_chunk(const float (*T)[LD], int ty, int tx, float (&acc)[4][4]) {
#pragma unroll 4
  for (int jj = 0; jj < CW; ++jj) {
    const float4 a = *reinterpret_cast<const float4*>(&T[jj][4 * ty]);
    const float4 b = *reinterpret_cast<const float4*>(&T[jj][4 * tx]);
    const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
  }
}

template <int NP>
__device__ __forceinline__ void gram_chunk_q(const float (*T)[LD], int nq, int ty, int tx, float (&acc)[4][4]) {
  switch (nq) {
    case 1: gram_chunk<NP, 1>(T, ty, tx, acc); break;
    case 2: gram_chunk<NP, 2>(T, ty, tx, acc); break;
    case 3: gram_chunk<NP, 3>(T, ty, tx, acc); break;
    default: gram_chunk<NP, 4>(T, ty, tx, acc); break;
  }
}

// o[p][q] += sum_{k < kmax} B[ty + 16 p][k] X[k][4 tx + q] for p < NP, with
// Bp[k][perm_row(i)] = B[i][k] and T[k][jj] the chunk of X.
template <int NP>
__device__ __forceinline__ void bx_chunk(const float (*Bp)[LD], const float (*T)[LD], int kmax, int ty, int tx,
                                         float (&o)[4][4]) {
#pragma unroll 4
  for (int k = 0; k < kmax; ++k) {
    const float4 b = *reinterpret_cast<const float4*>(&Bp[k][4 * ty]);
    const float4 x = *reinterpret_cast<const float4*>(&T[k][4 * tx]);
    const float bv[4] = {b.x, b.y, b.z, b.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) o[p][q] = fmaf(bv[p], xv[q], o[p][q]);
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

__global__ void __launch_bounds__(kNarrowThreads, 3) ns_narrow_kernel(const __grid_constant__ NarrowLaunch L) {
  __shared__ __align__(16) float s0[SP][LD];  // A; the chunk of B X
  __shared__ __align__(16) float s1[SP][LD];  // the chunk of X X^T; B (rows interleaved)
  __shared__ double red[kNarrowThreads / 32];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float coef = L.sc->coef * L.gscale;
  const float mu = L.mu;
  for (int mi = blockIdx.x; mi < L.nmat; mi += gridDim.x) {
    const MuonMat& M = L.mats[mi];
    float* const X = M.xf;
    const int s = M.s, l = M.l;
    const int64_t numel = (int64_t)M.m * M.n;
    // live row groups of this warp (rows ty + 16 p of its lower ty), column
    // groups of the Gram product, and the reduction length of A A and B X
    const int ty0 = ty & ~1;
    const int np = min(4, max(0, (s - ty0 + 15) / 16));
    const int nq = min(4, (s + 15) / 16);
    const int kmax = (s + 3) & ~3;
    const int nch = (l + CW - 1) / CW;
    // ---- the update G (as the momentum pass forms it) and ||G||_F ----
    double sq = 0.0;
    for (int64_t e0 = threadIdx.x; e0 < numel; e0 += (int64_t)UB * kNarrowThreads) {
      float gv[UB], bv[UB];
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        const int64_t e = e0 + (int64_t)k * kNarrowThreads;
        gv[k] = e < numel ? narrow_grad(M, e) : 0.f;
        bv[k] = e < numel ? M.buf[e] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        const int64_t e = e0 + (int64_t)k * kNarrowThreads;
        if (e < numel) {
          const float u = L.nesterov ? fmaf(mu, bv[k], coef * gv[k]) : bv[k];
          X[e] = u;
          sq += (double)u * (double)u;
        }
      }
    }
    const double tot = narrow_block_sum(sq, red);  // also orders the writes of X before the reads below
    const float r = (float)(1.0 / (sqrt(tot) + (double)L.eps));
    float4 stage[QPT];
    fetch_chunk(M, X, 0, stage);
    for (int it = 0; it < L.steps; ++it) {
      const bool first = it == 0, last = it == L.steps - 1;
      const float ca = L.coef[it][0], cb = L.coef[it][1], cc = L.coef[it][2];
      // ---- A = X X^T (r^2 X X^T in the first iteration) ----
      float acc[4][4] = {};
      for (int c = 0; c < nch; ++c) {
        store_chunk<true>(M, stage, s1);
        __syncthreads();
        if (c + 1 < nch) fetch_chunk(M, X, (c + 1) * CW, stage);
        switch (np) {
          case 0: break;
          case 1: gram_chunk_q<1>(s1, nq, ty, tx, acc); break;
          case 2: gram_chunk_q<2>(s1, nq, ty, tx, acc); break;
          case 3: gram_chunk_q<3>(s1, nq, ty, tx, acc); break;
          default: gram_chunk_q<4>(s1, nq, ty, tx, acc); break;
        }
        __syncthreads();  // the chunk buffer is refilled next
      }
      fetch_chunk(M, X, 0, stage);  // the first chunk of B X, in flight during A A
      const float sa = first ? r * r : 1.f;
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) s0[ty + 16 * p][tx + 16 * q] = acc[p][q] * sa;
      __syncthreads();
      // ---- B = a I + b A + c A A (A is symmetric: A[i][k] = A[k][i]); thread
      // (ty, tx) forms rows 4 ty.. and columns 4 tx.. of it ----
      float aa[4][4] = {};
      if (4 * ty < s) {
#pragma unroll 4
        for (int k = 0; k < kmax; ++k) {
          const float4 a = *reinterpret_cast<const float4*>(&s0[k][4 * ty]);
          const float4 b = *reinterpret_cast<const float4*>(&s0[k][4 * tx]);
          const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) aa[p][q] = fmaf(av[p], bv[q], aa[p][q]);
        }
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = 4 * ty + p, k = 4 * tx + q;
          const float lin = fmaf(cb, s0[i][k], i == k ? ca : 0.f);
          s1[k][perm_row(i)] = (i < s && k < s) ? fmaf(cc, aa[p][q], lin) : 0.f;
        }
      }
      __syncthreads();  // B complete; A no longer read (s0 takes the chunks of X)
      // ---- X' = B X (r B X in the first iteration), chunk by chunk in place;
      // the last iteration applies it to the parameter instead ----
      const float sx = first ? r : 1.f;
      const float lrm = L.sp->ns_lr * M.lr_mult;
      const float dec = L.sp->ns_decay[M.group];
      for (int c = 0; c < nch; ++c) {
        const int j0 = c * CW;
        store_chunk<false>(M, stage, s0);
        __syncthreads();
        if (c + 1 < nch) fetch_chunk(M, X, j0 + CW, stage);
        float pv[4][4];
        if (last) {  // the parameter's values, loaded while the product runs
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i = ty + 16 * p, j = j0 + 4 * tx + q;
              pv[p][q] = (p < np && i < s && j < l) ? M.p[canon_index(M, i, j)] : 0.f;
            }
        }
        float o[4][4] = {};
        switch (np) {
          case 0: break;
          case 1: bx_chunk<1>(s1, s0, kmax, ty, tx, o); break;
          case 2: bx_chunk<2>(s1, s0, kmax, ty, tx, o); break;
          case 3: bx_chunk<3>(s1, s0, kmax, ty, tx, o); break;
          default: bx_chunk<4>(s1, s0, kmax, ty, tx, o); break;
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int i = ty + 16 * p;
          if (p >= np || i >= s) continue;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = j0 + 4 * tx + q;
            if (j >= l) continue;
            const int64_t idx = canon_index(M, i, j);
            const float v = o[p][q] * sx;
            if (!last) {
              X[idx] = v;
            } else {
              const float pn = fmaf(pv[p][q], dec, -lrm * v);
              M.p[idx] = pn;
              if (M.shadow) M.shadow[idx] = ns_f2bf(pn);
            }
          }
        }
        __syncthreads();  // the chunk buffer is refilled next; X' is visible to the next Gram
      }
      if (!last) fetch_chunk(M, X, 0, stage);  // the next iteration's first Gram chunk
    }
  }
}

}  // namespace

cudaError_t launch_ns_narrow(const NarrowLaunch& L, int num_sms, cudaStream_t st) {
  const int grid = L.nmat < 3 * num_sms ? L.nmat : 3 * num_sms;
  if (grid <= 0) return cudaSuccess;
  ns_narrow_kernel<<<grid, kNarrowThreads, 0, st>>>(L);
  return cudaGetLastError();
}

}  // namespace ma
