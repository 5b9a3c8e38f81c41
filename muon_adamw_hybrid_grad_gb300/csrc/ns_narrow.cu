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
// about 25 to 55. Matrices with s < 64 therefore take this path, which keeps
// X, A and B in fp32 throughout (an error near 1e-6). They are few and cheap:
// a 40 x 2000 matrix costs about 2e8 flops per step.
//
// Two kernels, both of 256-thread CTAs:
//   ns_narrow_resident_kernel (below, after the shared helpers): a cluster of
//     1 to 8 CTAs per matrix, each holding a slice of X's long side in shared
//     memory for the whole chain; the partial Gram matrices are summed through
//     distributed shared memory.
//   ns_narrow_stream_kernel: one CTA per matrix, for matrices whose slices
//     would not fit in 8 CTAs' shared memory. X lives in the matrix's fp32
//     workspace in the parameter's own layout (m x n, row-major; for a wide
//     matrix, m <= n, the canonical s x l X is that array, for a tall one its
//     transpose). A and B (s x s, padded to 64 x 64) are in shared memory;
//     64-column chunks of X pass through shared memory for each product, and
//     X' = B X is written back in place chunk by chunk (a chunk of X' needs
//     only the same chunk of X). Every chunk is fetched into registers one
//     chunk ahead (four 16-byte words per thread), so the global loads of
//     chunk c + 1 are in flight while chunk c is multiplied out of shared
//     memory; each word goes to shared memory as one 16-byte store, in a
//     layout chosen per orientation:
//       wide:  the chunk as T[i][jj] for both products (rows of X);
//       tall:  T[jj][4 (i mod 16) + i / 16] for X X^T (rows of the parameter,
//              entries interleaved by the fetch), T[jj][i] for B X, which is
//              computed as (B X)^T = X^T B and staged through a third tile
//              so that it leaves along the parameter's rows.
//
// Work split (both kernels): thread (ty, tx) of the 16 x 16 grid holds rows
// ty + 16 p (p < 4) of each 64-row result. Rows interleave so that a short
// side s < 64 leaves every warp with ceil((s - row) / 16) live row groups, the
// same count on all four schedulers; a warp skips the groups that lie wholly
// in the zero padding, the Gram product skips the column groups tx + 16 q >= s
// (the same for every thread), and A A and B X stop their reductions at s
// rounded up to 4.
//
// The update G is recomputed from the momentum buffer that the momentum pass
// has just written and the gradient, with the same fp32 operations that pass
// uses (Nesterov: w coef g + mu buf), and the Frobenius scale r is folded in
// as the tensor-core path does: A of the first iteration is scaled by r^2 and
// its X' by r.
#include <cooperative_groups.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ns_epilogue.cuh"

namespace ma {
namespace {

constexpr int kNarrowThreads = 256;
constexpr int SP = 64;                             // padded short side
constexpr int CW = 64;                             // columns of the long side per chunk
constexpr int LD = SP + 4;                         // shared row pitch in floats (16-byte rows)
constexpr int QPT = SP * CW / 4 / kNarrowThreads;  // 4-float words of a chunk per thread
constexpr int UB = 8;                              // elements in flight per thread forming G
constexpr int UBV = 4;                             // 16-byte words of them, where aligned
constexpr int kTile = SP * LD;                     // floats per shared tile
constexpr size_t kNarrowSmem = 3 * kTile * sizeof(float) + (kNarrowThreads / 32) * sizeof(double);

typedef float Tile[LD];

// The fields of one matrix that the kernel uses, held in registers.
struct Narrow {
  float* X;            // fp32 X in the parameter layout
  float* p;            // fp32 master
  uint16_t* shadow;    // bf16 copy of p, or null
  int s, l;            // short and long side
  bool xvec, pvec;     // rows of X (of p and shadow) allow 4-float words
};

// Word k of this thread: 16 words per row of 64 floats.
__device__ __forceinline__ void word_coords(int k, int& hi, int& lo) {
  const int q = threadIdx.x + k * kNarrowThreads;
  hi = q >> 4;
  lo = 4 * (q & 15);
}

// Chunk [j0, j0 + CW) of X into registers (zero outside the matrix).
//   wide:           word (hi, lo) = X[hi][j0 + lo .. + 3]
//   tall, !INTERL:  word (hi, lo) = X[lo .. + 3][j0 + hi]
//   tall, INTERL:   word (hi, lo) = X[lo / 4 + 16 t][j0 + hi], t = 0..3
template <bool TALL, bool INTERL>
__device__ __forceinline__ void fetch_chunk(const Narrow& N, int j0, float4 (&v)[QPT]) {
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    int hi, lo;
    word_coords(k, hi, lo);
    float f[4] = {0.f, 0.f, 0.f, 0.f};
    if (!TALL) {
      const int j = j0 + lo;
      if (hi < N.s) {
        const float* src = N.X + (int64_t)hi * N.l + j;
        if (N.xvec && j + 3 < N.l) {
          v[k] = *reinterpret_cast<const float4*>(src);
          continue;
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (j + t < N.l) f[t] = src[t];
      }
    } else {
      const int j = j0 + hi;
      if (j < N.l) {
        const float* row = N.X + (int64_t)j * N.s;
        if (INTERL) {
          const int a = lo >> 2;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (a + 16 * t < N.s) f[t] = row[a + 16 * t];
        } else {
          if (N.xvec && lo + 3 < N.s) {
            v[k] = *reinterpret_cast<const float4*>(row + lo);
            continue;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (lo + t < N.s) f[t] = row[lo + t];
        }
      }
    }
    v[k] = make_float4(f[0], f[1], f[2], f[3]);
  }
}

__device__ __forceinline__ void store_chunk(const float4 (&v)[QPT], Tile* T) {
#pragma unroll
  for (int k = 0; k < QPT; ++k) {
    int hi, lo;
    word_coords(k, hi, lo);
    *reinterpret_cast<float4*>(&T[hi][lo]) = v[k];
  }
}

__device__ __forceinline__ float4 ld4(const float* T, int pitch, int r, int c) {
  return *reinterpret_cast<const float4*>(T + r * pitch + c);
}

// acc[p][q] += sum over columns jj < ncols (a multiple of 4) of
// X[ty + 16 p][jj] X[tx + 16 q][jj], p < NP, q < NQ. Wide: T[i][jj].
template <int NP, int NQ>
__device__ __forceinline__ void gram_wide(const float* T, int pitch, int ncols, int ty, int tx, float (&acc)[4][4]) {
#pragma unroll 2
  for (int jj = 0; jj < ncols; jj += 4) {
    float4 a[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) a[p] = ld4(T, pitch, ty + 16 * p, jj);
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const float4 b = ld4(T, pitch, tx + 16 * q, jj);
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        float c = acc[p][q];
        c = fmaf(a[p].x, b.x, c);
        c = fmaf(a[p].y, b.y, c);
        c = fmaf(a[p].z, b.z, c);
        c = fmaf(a[p].w, b.w, c);
        acc[p][q] = c;
      }
    }
  }
}

// Tall: T[jj][4 (i mod 16) + i / 16].
template <int NP, int NQ>
__device__ __forceinline__ void gram_tall(const float* T, int pitch, int ncols, int ty, int tx, float (&acc)[4][4]) {
#pragma unroll 4
  for (int jj = 0; jj < ncols; ++jj) {
    const float4 a = ld4(T, pitch, jj, 4 * ty), b = ld4(T, pitch, jj, 4 * tx);
    const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int q = 0; q < NQ; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
  }
}

template <bool TALL, int NP>
__device__ __forceinline__ void gram_q(const float* T, int pitch, int ncols, int nq, int ty, int tx,
                                       float (&acc)[4][4]) {
  switch (nq) {
    case 1: TALL ? gram_tall<NP, 1>(T, pitch, ncols, ty, tx, acc) : gram_wide<NP, 1>(T, pitch, ncols, ty, tx, acc); break;
    case 2: TALL ? gram_tall<NP, 2>(T, pitch, ncols, ty, tx, acc) : gram_wide<NP, 2>(T, pitch, ncols, ty, tx, acc); break;
    case 3: TALL ? gram_tall<NP, 3>(T, pitch, ncols, ty, tx, acc) : gram_wide<NP, 3>(T, pitch, ncols, ty, tx, acc); break;
    default: TALL ? gram_tall<NP, 4>(T, pitch, ncols, ty, tx, acc) : gram_wide<NP, 4>(T, pitch, ncols, ty, tx, acc); break;
  }
}

template <bool TALL>
__device__ __forceinline__ void gram_chunk(const float* T, int pitch, int ncols, int np, int nq, int ty, int tx,
                                           float (&acc)[4][4]) {
  switch (np) {
    case 0: break;
    case 1: gram_q<TALL, 1>(T, pitch, ncols, nq, ty, tx, acc); break;
    case 2: gram_q<TALL, 2>(T, pitch, ncols, nq, ty, tx, acc); break;
    case 3: gram_q<TALL, 3>(T, pitch, ncols, nq, ty, tx, acc); break;
    default: gram_q<TALL, 4>(T, pitch, ncols, nq, ty, tx, acc); break;
  }
}

// Bp[k][4 (i mod 16) + i / 16] = B[i][k].
// Wide: o[p][q] += sum_{k < kmax} B[ty + 16 p][k] X[k][4 tx + q], T[k][jj] the chunk.
template <int NP>
__device__ __forceinline__ void bx_wide(const float* Bp, const float* T, int pitch, int kmax, int ty, int tx,
                                        float (&o)[4][4]) {
#pragma unroll 4
  for (int k = 0; k < kmax; ++k) {
    const float4 b = ld4(Bp, LD, k, 4 * ty), x = ld4(T, pitch, k, 4 * tx);
    const float bv[4] = {b.x, b.y, b.z, b.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) o[p][q] = fmaf(bv[p], xv[q], o[p][q]);
  }
}

// Tall: o[p][q] += sum_{k < kmax} B[ty + 16 p][k] X[k][tx + 16 q], T[jj][k] the chunk.
template <int NP>
__device__ __forceinline__ void bx_tall(const float* Bp, const float* T, int pitch, int kmax, int ty, int tx,
                                        float (&o)[4][4]) {
#pragma unroll 1
  for (int k = 0; k < kmax; k += 4) {
    float4 x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q] = ld4(T, pitch, tx + 16 * q, k);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float4 b = ld4(Bp, LD, k + t, 4 * ty);
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float xv = t == 0 ? x[q].x : t == 1 ? x[q].y : t == 2 ? x[q].z : x[q].w;
#pragma unroll
        for (int p = 0; p < NP; ++p) o[p][q] = fmaf(bv[p], xv, o[p][q]);
      }
    }
  }
}

template <bool TALL>
__device__ __forceinline__ void bx_chunk(const float* Bp, const float* T, int pitch, int np, int kmax, int ty, int tx,
                                         float (&o)[4][4]) {
  switch (np) {
    case 0: break;
    case 1: TALL ? bx_tall<1>(Bp, T, pitch, kmax, ty, tx, o) : bx_wide<1>(Bp, T, pitch, kmax, ty, tx, o); break;
    case 2: TALL ? bx_tall<2>(Bp, T, pitch, kmax, ty, tx, o) : bx_wide<2>(Bp, T, pitch, kmax, ty, tx, o); break;
    case 3: TALL ? bx_tall<3>(Bp, T, pitch, kmax, ty, tx, o) : bx_wide<3>(Bp, T, pitch, kmax, ty, tx, o); break;
    default: TALL ? bx_tall<4>(Bp, T, pitch, kmax, ty, tx, o) : bx_wide<4>(Bp, T, pitch, kmax, ty, tx, o); break;
  }
}

// The last iteration: p <- p dec - lrm v for 4 consecutive elements at idx
// (one 16-byte word where `vec`), and the bf16 shadow.
__device__ __forceinline__ void apply4(const Narrow& N, int64_t idx, int cnt, bool vec, const float (&v)[4],
                                       float dec, float lrm) {
  if (vec && cnt == 4) {
    const float4 pv = *reinterpret_cast<const float4*>(N.p + idx);
    const float4 pn = make_float4(fmaf(pv.x, dec, -lrm * v[0]), fmaf(pv.y, dec, -lrm * v[1]),
                                  fmaf(pv.z, dec, -lrm * v[2]), fmaf(pv.w, dec, -lrm * v[3]));
    *reinterpret_cast<float4*>(N.p + idx) = pn;
    if (N.shadow) {
      uint2 h;
      h.x = (uint32_t)ns_f2bf(pn.x) | ((uint32_t)ns_f2bf(pn.y) << 16);
      h.y = (uint32_t)ns_f2bf(pn.z) | ((uint32_t)ns_f2bf(pn.w) << 16);
      *reinterpret_cast<uint2*>(N.shadow + idx) = h;
    }
    return;
  }
  float pv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) pv[t] = t < cnt ? N.p[idx + t] : 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if (t >= cnt) break;
    const float pn = fmaf(pv[t], dec, -lrm * v[t]);
    N.p[idx + t] = pn;
    if (N.shadow) N.shadow[idx + t] = ns_f2bf(pn);
  }
}

// X' = v for 4 consecutive elements at idx.
__device__ __forceinline__ void store4(float* X, int64_t idx, int cnt, bool vec, const float (&v)[4]) {
  if (vec && cnt == 4) {
    *reinterpret_cast<float4*>(X + idx) = make_float4(v[0], v[1], v[2], v[3]);
    return;
  }
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (t < cnt) X[idx + t] = v[t];
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

template <bool TALL>
__device__ void narrow_matrix(const NarrowLaunch& L, const MuonMat& M, float* smem, double* red) {
  Tile* const s0 = reinterpret_cast<Tile*>(smem);              // A; the chunk of B X
  Tile* const s1 = reinterpret_cast<Tile*>(smem + kTile);      // the Gram chunk; B (rows interleaved)
  Tile* const s2 = reinterpret_cast<Tile*>(smem + 2 * kTile);  // tall: the chunk of X' = B X, staged
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  Narrow N;
  N.X = M.xf;
  N.p = M.p;
  N.shadow = M.shadow;
  N.s = M.s;
  N.l = M.l;
  // X starts 16-byte aligned (the host pads every slot); its rows in memory
  // are l floats long for a wide matrix, s for a tall one
  N.xvec = TALL ? (N.s % 4 == 0) : (N.l % 4 == 0);
  N.pvec = M.pvec != 0;
  const int s = N.s, l = N.l;
  const int64_t numel = (int64_t)M.m * M.n;
  // live row groups of this warp (rows ty + 16 p of its lower ty), column
  // groups of the Gram product, and the reduction length of A A and B X
  const int np = min(4, max(0, (s - (ty & ~1) + 15) / 16));
  const int nq = min(4, (s + 15) / 16);
  const int kmax = (s + 3) & ~3;
  const int nch = (l + CW - 1) / CW;
  const float lrm = L.sp->ns_lr * M.lr_mult;
  const float dec = L.sp->ns_decay[M.group];
  // ---- the update G (as the momentum pass forms it) and ||G||_F ----
  float r;
  {
    const float coef = L.sc->coef * L.gscale, mu = L.mu;
    const bool gbf = M.gdtype == DT_BF16;
    const void* const g = M.g;
    const float* const buf = M.buf;
    double sq = 0.0;
    for (int64_t e0 = threadIdx.x; e0 < numel; e0 += (int64_t)UB * kNarrowThreads) {
      float gv[UB], bv[UB];
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        const int64_t e = e0 + (int64_t)k * kNarrowThreads;
        gv[k] = 0.f;
        bv[k] = 0.f;
        if (e < numel) {
          gv[k] = gbf ? __uint_as_float(((uint32_t) static_cast<const uint16_t*>(g)[e]) << 16)
                      : static_cast<const float*>(g)[e];
          bv[k] = buf[e];
        }
      }
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        const int64_t e = e0 + (int64_t)k * kNarrowThreads;
        if (e < numel) {
          const float u = L.nesterov ? fmaf(mu, bv[k], coef * gv[k]) : bv[k];
          N.X[e] = u;
          sq += (double)u * (double)u;
        }
      }
    }
    const double tot = narrow_block_sum(sq, red);  // also orders the writes of X before the reads below
    r = (float)(1.0 / (sqrt(tot) + (double)L.eps));
  }
  {
    float4 stage[QPT];
    for (int it = 0; it < L.steps; ++it) {
      const bool first = it == 0, last = it == L.steps - 1;
      const float ca = L.coef[it][0], cb = L.coef[it][1], cc = L.coef[it][2];
      // ---- A = X X^T (r^2 X X^T in the first iteration) ----
      fetch_chunk<TALL, true>(N, 0, stage);
      float acc[4][4] = {};
      for (int c = 0; c < nch; ++c) {
        store_chunk(stage, s1);
        __syncthreads();
        if (c + 1 < nch) fetch_chunk<TALL, true>(N, (c + 1) * CW, stage);
        gram_chunk<TALL>(&s1[0][0], LD, CW, np, nq, ty, tx, acc);
        __syncthreads();  // the chunk buffer is refilled next
      }
      fetch_chunk<TALL, false>(N, 0, stage);  // the first chunk of B X, in flight during A A
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
          const float4 a = ld4(&s0[0][0], LD, k, 4 * ty), b = ld4(&s0[0][0], LD, k, 4 * tx);
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
          s1[k][4 * (i & 15) + (i >> 4)] = (i < s && k < s) ? fmaf(cc, aa[p][q], lin) : 0.f;
        }
      }
      __syncthreads();  // B complete; A no longer read (s0 takes the chunks of X)
      // ---- X' = B X (r B X in the first iteration), chunk by chunk in place;
      // the last iteration applies it to the parameter instead ----
      const float sx = first ? r : 1.f;
      for (int c = 0; c < nch; ++c) {
        const int j0 = c * CW;
        store_chunk(stage, s0);
        __syncthreads();
        if (c + 1 < nch) fetch_chunk<TALL, false>(N, j0 + CW, stage);
        float o[4][4] = {};
        bx_chunk<TALL>(&s1[0][0], &s0[0][0], LD, np, kmax, ty, tx, o);
        if (!TALL) {
          // o[p][q] = X'[ty + 16 p][j0 + 4 tx + q]: along the parameter's rows
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int i = ty + 16 * p, j = j0 + 4 * tx;
            if (p >= np || i >= s || j >= l) continue;
            const float v[4] = {o[p][0] * sx, o[p][1] * sx, o[p][2] * sx, o[p][3] * sx};
            const int cnt = min(4, l - j);
            const int64_t idx = (int64_t)i * l + j;
            if (!last)
              store4(N.X, idx, cnt, N.xvec, v);
            else
              apply4(N, idx, cnt, N.pvec, v, dec, lrm);
          }
        } else {
          // o[p][q] = X'[ty + 16 p][j0 + tx + 16 q]: staged as s2[jj][i], then
          // out along the parameter's rows (each s floats long)
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) s2[tx + 16 * q][ty + 16 * p] = o[p][q] * sx;
        }
        __syncthreads();  // the chunk buffer is refilled next; tall: X' staged
        if (TALL) {
#pragma unroll
          for (int k = 0; k < QPT; ++k) {
            int hi, lo;
            word_coords(k, hi, lo);
            const int j = j0 + hi;
            if (j >= l || lo >= s) continue;
            const float4 w = ld4(&s2[0][0], LD, hi, lo);
            const float v[4] = {w.x, w.y, w.z, w.w};
            const int cnt = min(4, s - lo);
            const int64_t idx = (int64_t)j * s + lo;
            if (!last)
              store4(N.X, idx, cnt, N.xvec, v);
            else
              apply4(N, idx, cnt, N.pvec, v, dec, lrm);
          }
        }
      }
      __syncthreads();  // X' complete before the next Gram reads it; s2 free
    }
  }
}

__global__ void __launch_bounds__(kNarrowThreads, 2) ns_narrow_stream_kernel(const __grid_constant__ NarrowLaunch L) {
  extern __shared__ __align__(16) float narrow_smem[];
  double* const red = reinterpret_cast<double*>(narrow_smem + 3 * kTile);
  for (int mi = blockIdx.x; mi < L.nmat; mi += gridDim.x) {
    const MuonMat& M = L.mats[L.idx[mi]];
    if (M.transposed)
      narrow_matrix<true>(L, M, narrow_smem, red);
    else
      narrow_matrix<false>(L, M, narrow_smem, red);
  }
}

// ---------------------------------------------------------------------------
// Resident kernel: a cluster of C CTAs per matrix. CTA `rank` holds columns
// [rank lc, rank lc + ncol) of the canonical X in shared memory as XS[i][j]
// (row pitch P floats, rows s.. R-1 and columns ncol.. zero) from the update
// through the parameter update; nothing of X goes back to global memory in
// between. Two 64 x 68 tiles T0, T1 alternate. Iteration it:
//   X X^T over the CTA's columns (no barriers: XS is only read) into
//   T[it mod 2], thread-major (thread t's 16 values as 4 words at t + 256 k);
//   a cluster barrier; every CTA adds the C partial tiles in rank order
//   (through distributed shared memory, 16-byte words), so all of them hold
//   the same A, written as A[i][k] into the other tile; then B = a I + b A +
//   c A A over it, and X' = B X over the CTA's columns in 64-column chunks,
//   each written back in place once every thread has read it.
// A partial tile is overwritten two iterations later, after the next
// iteration's cluster barrier, which every CTA reaches only once it has read
// all partials of this one; the other tile is free locally from this
// iteration's barrier on (its partials were read before it). The Frobenius
// norm's sum of squares is exchanged the same way, its barrier split around
// the first Gram product. All CTAs of a cluster take
// the same path (the same matrix and iteration count), so each cluster
// barrier is reached by all of them; a final cluster barrier keeps every CTA's
// shared memory alive until the last remote read of it.
// ---------------------------------------------------------------------------

// The two halves of a cluster barrier (every thread of every CTA of the
// cluster executes both, in this order, between two full barriers).
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory offset and global index of element e of this CTA's slice, in
// the order of the parameter's rows (e < s ncol < 2^31).
template <bool TALL>
__device__ __forceinline__ void slice_coords(int e, int s, int l, int c0, int ncol, int P, int& xo, int64_t& gidx) {
  if (!TALL) {  // parameter [s][l]: row i, columns c0 + j
    const int i = e / ncol, j = e - i * ncol;
    xo = i * P + j;
    gidx = (int64_t)i * l + c0 + j;
  } else {  // parameter [l][s]: rows c0 + j, column i
    const int j = e / s, i = e - j * s;
    xo = i * P + j;
    gidx = (int64_t)c0 * s + e;
  }
}

template <bool TALL>
__device__ void resident_matrix(const NarrowLaunch& L, const MuonMat& M, int C, int rank, float* smem) {
  namespace cg = cooperative_groups;
  float* const T0 = smem;                                             // partial A, or A then B
  float* const T1 = smem + SP * LD;                                   // the same, alternating
  double* const xch = reinterpret_cast<double*>(smem + 2 * SP * LD);  // [0]: this CTA's sum of squares
  double* const red = xch + 8;
  float* const XS = smem + kNarrowFixedFloats;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int s = M.s, l = M.l;
  const int R = narrow_rows(s), lc = narrow_cols(l, C), P = narrow_pitch(lc);
  const int c0 = rank * lc;
  const int ncol = max(0, min(lc, l - c0));
  const int np = min(4, max(0, (s - (ty & ~1) + 15) / 16));
  const int nq = min(4, (s + 15) / 16);
  const int kmax = (s + 3) & ~3;
  const float lrm = L.sp->ns_lr * M.lr_mult;
  const float dec = L.sp->ns_decay[M.group];
  // ---- the slice of G (as the momentum pass forms it) and ||G||_F ----
  for (int e = threadIdx.x; e < R * P / 4; e += kNarrowThreads)
    reinterpret_cast<float4*>(XS)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  float r;
  {
    const float coef = L.sc->coef * L.gscale, mu = L.mu;
    const bool gbf = M.gdtype == DT_BF16;
    const void* const g = M.g;
    const float* const buf = M.buf;
    const int cnt = s * ncol;
    double sq = 0.0;
    // 16-byte words of 4 consecutive elements of a parameter row where the
    // rows hold whole words (then every CTA's slice starts on one)
    const bool uvec = (TALL ? (s % 4 == 0) : (l % 4 == 0)) &&
                      reinterpret_cast<uintptr_t>(g) % (gbf ? 8 : 16) == 0 && reinterpret_cast<uintptr_t>(buf) % 16 == 0;
    const int words = uvec ? cnt / 4 : 0;
    for (int w0 = threadIdx.x; w0 < words; w0 += UBV * kNarrowThreads) {
      float4 gv[UBV], bv[UBV];
      int xo[UBV];
#pragma unroll
      for (int k = 0; k < UBV; ++k) {
        const int w = w0 + k * kNarrowThreads;
        xo[k] = -1;
        if (w < words) {
          int64_t gi;
          slice_coords<TALL>(4 * w, s, l, c0, ncol, P, xo[k], gi);
          bv[k] = *reinterpret_cast<const float4*>(buf + gi);
          if (gbf) {
            const uint2 h = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(g) + gi);
            gv[k] = make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u),
                                __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xffff0000u));
          } else {
            gv[k] = *reinterpret_cast<const float4*>(static_cast<const float*>(g) + gi);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < UBV; ++k) {
        if (xo[k] < 0) continue;
        float4 u = bv[k];
        if (L.nesterov)
          u = make_float4(fmaf(mu, bv[k].x, coef * gv[k].x), fmaf(mu, bv[k].y, coef * gv[k].y),
                          fmaf(mu, bv[k].z, coef * gv[k].z), fmaf(mu, bv[k].w, coef * gv[k].w));
        if (!TALL) {
          *reinterpret_cast<float4*>(XS + xo[k]) = u;  // X[i][j..j+3]
        } else {
          XS[xo[k]] = u.x;  // X[i..i+3][j]
          XS[xo[k] + P] = u.y;
          XS[xo[k] + 2 * P] = u.z;
          XS[xo[k] + 3 * P] = u.w;
        }
        sq += (double)u.x * u.x + (double)u.y * u.y + (double)u.z * u.z + (double)u.w * u.w;
      }
    }
    for (int e0 = 4 * words + threadIdx.x; e0 < cnt; e0 += UB * kNarrowThreads) {
      float gv[UB], bv[UB];
      int xo[UB];
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        const int e = e0 + k * kNarrowThreads;
        gv[k] = 0.f;
        bv[k] = 0.f;
        xo[k] = -1;
        if (e < cnt) {
          int64_t gi;
          slice_coords<TALL>(e, s, l, c0, ncol, P, xo[k], gi);
          gv[k] = gbf ? __uint_as_float(((uint32_t) static_cast<const uint16_t*>(g)[gi]) << 16)
                      : static_cast<const float*>(g)[gi];
          bv[k] = buf[gi];
        }
      }
#pragma unroll
      for (int k = 0; k < UB; ++k) {
        if (xo[k] >= 0) {
          const float u = L.nesterov ? fmaf(mu, bv[k], coef * gv[k]) : bv[k];
          XS[xo[k]] = u;
          sq += (double)u * (double)u;
        }
      }
    }
    const double tot = narrow_block_sum(sq, red);  // also orders the writes of XS before the reads below
    if (C > 1) {
      // every CTA's sum of squares is read after the first Gram product, which
      // does not need it (r enters as the factor r^2 of that A)
      if (threadIdx.x == 0) xch[0] = tot;
      cluster_arrive();
      r = 0.f;
    } else {
      r = (float)(1.0 / (sqrt(tot) + (double)L.eps));
    }
  }
  for (int it = 0; it < L.steps; ++it) {
    const bool first = it == 0;
    const float ca = L.coef[it][0], cb = L.coef[it][1], cc = L.coef[it][2];
    float* const PT = (it & 1) ? T1 : T0;  // this iteration's partial
    float* const AB = (it & 1) ? T0 : T1;  // A, then B
    // ---- A = X X^T (r^2 X X^T in the first iteration) ----
    {
      float acc[4][4] = {};
      gram_chunk<false>(XS, P, lc, np, nq, ty, tx, acc);
      if (first && C > 1) {
        cluster_wait();
        double tot = 0.0;
        for (int q = 0; q < C; ++q) tot += *cg::this_cluster().map_shared_rank(xch, q);  // rank order everywhere
        r = (float)(1.0 / (sqrt(tot) + (double)L.eps));
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
        reinterpret_cast<float4*>(PT)[p * kNarrowThreads + threadIdx.x] =
            make_float4(acc[p][0], acc[p][1], acc[p][2], acc[p][3]);
    }
    float sum[4][4] = {};
    if (C > 1) {
      cg::cluster_group cl = cg::this_cluster();
      cl.sync();  // every partial written; the other tile's partials all read
      // row groups p >= np are zero in every partial: not read
#pragma unroll 4
      for (int rk = 0; rk < C; ++rk) {
        const float4* rp = reinterpret_cast<const float4*>(cl.map_shared_rank(PT, rk));
        float4 w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
          w[p] = p < np ? rp[p * kNarrowThreads + threadIdx.x] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          sum[p][0] += w[p].x;
          sum[p][1] += w[p].y;
          sum[p][2] += w[p].z;
          sum[p][3] += w[p].w;
        }
      }
    } else {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float4 w = reinterpret_cast<const float4*>(PT)[p * kNarrowThreads + threadIdx.x];
        sum[p][0] = w.x;
        sum[p][1] = w.y;
        sum[p][2] = w.z;
        sum[p][3] = w.w;
      }
    }
    {
      const float sa = first ? r * r : 1.f;
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) AB[(ty + 16 * p) * LD + tx + 16 * q] = sum[p][q] * sa;
    }
    __syncthreads();
    // ---- B = a I + b A + c A A; thread (ty, tx) forms rows 4 ty.. and
    // columns 4 tx.. of it, then writes it over A ----
    float bv[4][4];
    {
      float aa[4][4] = {};
      if (4 * ty < s) {
#pragma unroll 4
        for (int k = 0; k < kmax; ++k) {
          const float4 a = ld4(AB, LD, k, 4 * ty), b = ld4(AB, LD, k, 4 * tx);
          const float av[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) aa[p][q] = fmaf(av[p], bw[q], aa[p][q]);
        }
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = 4 * ty + p, k = 4 * tx + q;
          const float lin = fmaf(cb, AB[i * LD + k], i == k ? ca : 0.f);
          bv[p][q] = (i < s && k < s) ? fmaf(cc, aa[p][q], lin) : 0.f;
        }
    }
    __syncthreads();  // A fully read
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = 4 * ty + p, k = 4 * tx + q;
        AB[k * LD + 4 * (i & 15) + (i >> 4)] = bv[p][q];
      }
    __syncthreads();
    // ---- X' = B X (r B X in the first iteration), 64 columns at a time ----
    const float sx = first ? r : 1.f;
    for (int j0 = 0; j0 < lc; j0 += CW) {
      float o[4][4] = {};
      bx_chunk<false>(AB, XS + j0, P, np, kmax, ty, tx, o);
      __syncthreads();  // every thread has read these columns
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        if (p >= np) continue;
        *reinterpret_cast<float4*>(XS + (ty + 16 * p) * P + j0 + 4 * tx) =
            make_float4(o[p][0] * sx, o[p][1] * sx, o[p][2] * sx, o[p][3] * sx);
      }
    }
    __syncthreads();  // X' complete
  }
  // ---- p <- p dec - lrm X' over the slice, along the parameter's rows ----
  float* const pp = M.p;
  uint16_t* const sh = M.shadow;
  const bool vec = M.pvec != 0;  // rows of p a multiple of 8 floats, p and shadow 16-byte aligned
  if (vec) {
    const int words = s * ncol / 4;  // 4 consecutive elements of a parameter row
    for (int w0 = threadIdx.x; w0 < words; w0 += 4 * kNarrowThreads) {
      float4 pv[4];
      int64_t gi[4];
      int xo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int w = w0 + k * kNarrowThreads;
        xo[k] = -1;
        if (w < words) {
          slice_coords<TALL>(4 * w, s, l, c0, ncol, P, xo[k], gi[k]);
          pv[k] = *reinterpret_cast<const float4*>(pp + gi[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (xo[k] < 0) continue;
        // the 4 elements: X'[i][j..j+3] (wide) or X'[i..i+3][j] (tall)
        const int st = TALL ? P : 1;
        const float4 pn = make_float4(fmaf(pv[k].x, dec, -lrm * XS[xo[k]]), fmaf(pv[k].y, dec, -lrm * XS[xo[k] + st]),
                                      fmaf(pv[k].z, dec, -lrm * XS[xo[k] + 2 * st]),
                                      fmaf(pv[k].w, dec, -lrm * XS[xo[k] + 3 * st]));
        *reinterpret_cast<float4*>(pp + gi[k]) = pn;
        if (sh) {
          uint2 hb;
          hb.x = (uint32_t)ns_f2bf(pn.x) | ((uint32_t)ns_f2bf(pn.y) << 16);
          hb.y = (uint32_t)ns_f2bf(pn.z) | ((uint32_t)ns_f2bf(pn.w) << 16);
          *reinterpret_cast<uint2*>(sh + gi[k]) = hb;
        }
      }
    }
  } else {
    const int cnt = s * ncol;
    for (int e0 = threadIdx.x; e0 < cnt; e0 += 4 * kNarrowThreads) {
      float pv[4];
      int64_t gi[4];
      int xo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = e0 + k * kNarrowThreads;
        xo[k] = -1;
        if (e < cnt) {
          slice_coords<TALL>(e, s, l, c0, ncol, P, xo[k], gi[k]);
          pv[k] = pp[gi[k]];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (xo[k] < 0) continue;
        const float pn = fmaf(pv[k], dec, -lrm * XS[xo[k]]);
        pp[gi[k]] = pn;
        if (sh) sh[gi[k]] = ns_f2bf(pn);
      }
    }
  }
  if (C > 1) cg::this_cluster().sync();  // no CTA leaves while another may still read its tiles
}

__global__ void __launch_bounds__(kNarrowThreads, 2) ns_narrow_resident_kernel(const __grid_constant__ NarrowLaunch L) {
  extern __shared__ __align__(16) float narrow_smem[];
  const int C = L.cluster;
  const int rank = C > 1 ? (int)cooperative_groups::this_cluster().block_rank() : 0;
  const MuonMat& M = L.mats[L.idx[blockIdx.x / C]];
  if (M.transposed)
    resident_matrix<true>(L, M, C, rank, narrow_smem);
  else
    resident_matrix<false>(L, M, C, rank, narrow_smem);
}

}  // namespace

cudaError_t ns_narrow_prepare(size_t resident_smem, int* stream_blocks_per_sm) {
  cudaError_t e =
      cudaFuncSetAttribute(ns_narrow_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNarrowSmem);
  if (e != cudaSuccess) return e;
  if (resident_smem > 0 &&
      (e = cudaFuncSetAttribute(ns_narrow_resident_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)resident_smem)) != cudaSuccess)
    return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(stream_blocks_per_sm, ns_narrow_stream_kernel, kNarrowThreads,
                                                    kNarrowSmem);
  if (e == cudaSuccess && *stream_blocks_per_sm < 1) *stream_blocks_per_sm = 1;
  return e;
}

cudaError_t launch_ns_narrow(const NarrowLaunch& L, size_t smem, int num_sms, int blocks_per_sm, cudaStream_t st) {
  if (L.nmat <= 0) return cudaSuccess;
  if (L.cluster == 0) {
    const int resident = blocks_per_sm * num_sms;
    const int grid = L.nmat < resident ? L.nmat : resident;
    ns_narrow_stream_kernel<<<grid, kNarrowThreads, kNarrowSmem, st>>>(L);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)(L.nmat * L.cluster), 1, 1);
  cfg.blockDim = dim3(kNarrowThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (L.cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)L.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, ns_narrow_resident_kernel, L);
}

}  // namespace ma
