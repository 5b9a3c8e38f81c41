// CUDA-core grouped GEMM for the Newton-Schulz iterations: a slow, simple
// kernel with the same inputs, outputs and epilogue as the tensor-core
// kernel, used to cross-check it on the GPU (config ns_kernel = MA_NS_SIMT).
//
// One 64x64 output tile per block, bf16 operands widened to fp32 in shared
// memory, fp32 accumulation. For the symmetric products (X X^T and A A) only
// tiles on or below the diagonal are computed; the epilogue mirrors them.
#include "internal.h"
#include "ns_epilogue.cuh"

namespace ma {
namespace {

constexpr int TM = 64, TN = 64, TK = 32;

__global__ void __launch_bounds__(256) ns_simt_kernel(NsProblem pb, NsEpiArgs ep, int tiles_per_mat) {
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int mat = blockIdx.x / tiles_per_mat;
  int t = blockIdx.x % tiles_per_mat;
  int ti = 0, tj = 0;
  const bool sym = pb.kind != NS_UPDATE;
  if (sym) {
    // lower-triangle enumeration: row block ti holds ti + 1 tiles
    while (t > ti) {
      t -= ti + 1;
      ++ti;
    }
    tj = t;
  } else {
    const int tn = pb.N / TN;
    ti = t / tn;
    tj = t % tn;
  }
  const int i0 = ti * TM, j0 = tj * TN;
  const size_t pstride = (size_t)pb.M * pb.K;
  const uint16_t* P = pb.P + (size_t)mat * pstride;
  const uint16_t* Q = pb.Q + (size_t)mat * (sym ? pstride : (size_t)pb.K * pb.N);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < pb.K; k0 += TK) {
    // P tile: rows i0..i0+63, cols k0..k0+31 (row-major, ld K)
    for (int e = threadIdx.x; e < TM * TK; e += 256) {
      const int r = e / TK, k = e % TK;
      As[k][r] = ns_bf2f(P[(size_t)(i0 + r) * pb.K + k0 + k]);
    }
    if (sym) {
      for (int e = threadIdx.x; e < TN * TK; e += 256) {
        const int r = e / TK, k = e % TK;
        Bs[k][r] = ns_bf2f(Q[(size_t)(j0 + r) * pb.K + k0 + k]);
      }
    } else {
      for (int e = threadIdx.x; e < TN * TK; e += 256) {
        const int k = e / TN, c = e % TN;
        Bs[k][c] = ns_bf2f(Q[(size_t)(k0 + k) * pb.N + j0 + c]);
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < TK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = As[k][ty * 4 + u];
        b[u] = Bs[k][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int w = 0; w < 4; ++w) acc[u][w] = fmaf(a[u], b[w], acc[u][w]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) ns_epilogue_element(pb, ep, mat, i0 + ty * 4 + u, j0 + tx * 4 + w, acc[u][w]);
}

}  // namespace

void launch_ns_simt(const NsProblem& prob, NsEpiArgs epi, cudaStream_t st) {
  int tiles;
  if (prob.kind == NS_UPDATE) {
    tiles = (prob.M / TM) * (prob.N / TN);
  } else {
    const int nt = prob.M / TM;
    tiles = nt * (nt + 1) / 2;
  }
  const int grid = tiles * prob.nmat;
  if (grid > 0) ns_simt_kernel<<<grid, 256, 0, st>>>(prob, epi, tiles);
}

}  // namespace ma
