// HBM-bound kernels of the hybrid Muon + AdamW step.
//
// OpenDM VLA training-stack article, 核心揭秘一 (MuonAdamW hybrid optimizer) and
// the defaults table 训练栈默认参数速查表:
//   grad_sumsq / clip_finalize : global gradient norm, clip at max_grad_norm 1.0
//   muon_momentum              : Nesterov momentum (muon_momentum 0.95) and the
//                                bf16 canonical (short-side-first) copy that the
//                                Newton-Schulz GEMMs read
//   ns_prep                    : 1 / (||update||_F + eps), the Frobenius
//                                normalisation folded into iteration 1
//   adamw                      : fused multi-tensor AdamW for all other params
//
// All loads and stores are 16-byte vectors where alignment allows; every
// reduction runs in a fixed order, so results are bitwise reproducible.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace ma {
namespace {

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

__device__ __forceinline__ void unpack8(const uint4& w, float* x) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Kahan-compensated fp32 accumulator (per thread).
struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    float y = x - c;
    float t = s + y;
    if (__builtin_expect(isinf(t), 0)) {  // inf - inf in the compensation would turn it into NaN
      s = t;
      c = 0.f;
      return;
    }
    c = (t - s) - y;
    s = t;
  }
};

// Fixed-order block reduction of one double per thread; result valid in thread 0.
template <int NT>
__device__ __forceinline__ double block_sum_double(double v, double* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = lane < NT / 32 ? sh[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  }
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// Global gradient norm: per-block partial sums of squares.
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 512;

__global__ void __launch_bounds__(kNormThreads) grad_sumsq_kernel(const GradChunk* __restrict__ chunks,
                                                                  int nchunks, float* __restrict__ partials) {
  __shared__ double sh[kNormThreads / 32];
  Kahan acc;
  for (int c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const GradChunk ch = chunks[c];
    if (ch.dtype == DT_BF16) {
      const uint16_t* g = static_cast<const uint16_t*>(ch.g);
      int64_t nv = ch.vec ? ch.n / 8 : 0;
      const uint4* gv = reinterpret_cast<const uint4*>(g);
      int64_t i = threadIdx.x;
      for (; i + 3 * kNormThreads < nv; i += 4 * kNormThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = __ldg(gv + i + u * kNormThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float x[8];
          unpack8(w[u], x);
          float s8 = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) s8 = fmaf(x[e], x[e], s8);
          acc.add(s8);
        }
      }
      for (; i < nv; i += kNormThreads) {
        float x[8];
        unpack8(__ldg(gv + i), x);
        float s8 = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s8 = fmaf(x[e], x[e], s8);
        acc.add(s8);
      }
      for (int64_t j = nv * 8 + threadIdx.x; j < ch.n; j += kNormThreads) {
        float x = bf2f(g[j]);
        acc.add(x * x);
      }
    } else {
      const float* g = static_cast<const float*>(ch.g);
      int64_t nv = ch.vec ? ch.n / 4 : 0;
      const float4* gv = reinterpret_cast<const float4*>(g);
      int64_t i = threadIdx.x;
      for (; i + 3 * kNormThreads < nv; i += 4 * kNormThreads) {
        float4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = __ldg(gv + i + u * kNormThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float s4 = w[u].x * w[u].x;
          s4 = fmaf(w[u].y, w[u].y, s4);
          s4 = fmaf(w[u].z, w[u].z, s4);
          s4 = fmaf(w[u].w, w[u].w, s4);
          acc.add(s4);
        }
      }
      for (; i < nv; i += kNormThreads) {
        float4 w = __ldg(gv + i);
        float s4 = w.x * w.x;
        s4 = fmaf(w.y, w.y, s4);
        s4 = fmaf(w.z, w.z, s4);
        s4 = fmaf(w.w, w.w, s4);
        acc.add(s4);
      }
      for (int64_t j = nv * 4 + threadIdx.x; j < ch.n; j += kNormThreads) {
        float x = g[j];
        acc.add(x * x);
      }
    }
  }
  double tot = block_sum_double<kNormThreads>((double)acc.s - (double)acc.c, sh);
  if (threadIdx.x == 0) partials[blockIdx.x] = (float)tot;
}

// ---------------------------------------------------------------------------
// Norm finalise and clip coefficient (one block).
// ---------------------------------------------------------------------------
constexpr int kClipThreads = 256;

__global__ void __launch_bounds__(kClipThreads) clip_finalize_kernel(const float* __restrict__ partials, int n,
                                                                     float max_norm, float clip_eps,
                                                                     StepScalars* __restrict__ out) {
  __shared__ double sh[kClipThreads / 32];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += kClipThreads) s += (double)partials[i];
  double tot = block_sum_double<kClipThreads>(s, sh);
  if (threadIdx.x == 0) {
    double total = sqrt(tot);
    double coef;
    if (isnan(total)) {
      coef = total;  // a NaN norm poisons every update, as multiplying by a NaN factor does
    } else if (max_norm > 0.f) {
      coef = (double)max_norm / (total + (double)clip_eps);
      if (coef > 1.0) coef = 1.0;
    } else {
      coef = 1.0;
    }
    out->total = (float)total;
    out->coef = (float)coef;
  }
}

// ---------------------------------------------------------------------------
// Sharded step: this rank's sum of squares (fp64) from its partials, and the
// norm and clip coefficient from the sum over all ranks.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kClipThreads) sumsq_partials_kernel(const float* __restrict__ partials, int n,
                                                                      double* __restrict__ out) {
  __shared__ double sh[kClipThreads / 32];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += kClipThreads) s += (double)partials[i];
  const double tot = block_sum_double<kClipThreads>(s, sh);
  if (threadIdx.x == 0) *out = tot;
}

__global__ void clip_from_sumsq_kernel(const double* __restrict__ sumsq, float max_norm, float clip_eps,
                                       StepScalars* __restrict__ out) {
  const double total = sqrt(*sumsq);
  double coef;
  if (isnan(total)) {
    coef = total;
  } else if (max_norm > 0.f) {
    coef = (double)max_norm / (total + (double)clip_eps);
    if (coef > 1.0) coef = 1.0;
  } else {
    coef = 1.0;
  }
  out->total = (float)total;
  out->coef = (float)coef;
}

// ---------------------------------------------------------------------------
// Muon momentum + canonical bf16 pack.
// One tile of one parameter per iteration (64 x 64 for tall matrices, 16
// rows x 256 columns otherwise, so that a warp streams 1 KB row segments);
// 256 threads, each owns an 8-wide column group of two rows. buf <- mu*buf +
// w*coef*g; the update
// (Nesterov: w*coef*g + mu*buf) goes to X in bf16; w = 1, or 1 - mu for the
// exponential-average form of the momentum. Wide matrices (X = update)
// are written straight from registers, 16 bytes per thread, with no block
// barrier. Tall matrices (X = update^T) go through a shared-memory tile,
// double-buffered so that one barrier per tile suffices. Sum of squares of
// the update: one fp32 partial per warp and tile (fixed order).
// ---------------------------------------------------------------------------
constexpr int kMomThreads = 256;
constexpr int kMomWarps = kMomThreads / 32;

__global__ void __launch_bounds__(kMomThreads) muon_momentum_kernel(const MomTile* __restrict__ tiles, int ntiles,
                                                                    const MuonMat* __restrict__ mats,
                                                                    const StepScalars* __restrict__ sc, MomArgs args,
                                                                    float* __restrict__ tile_partials) {
  // transpose tiles of tall matrices: 16-byte chunk c of row r sits at chunk
  // c ^ ((r >> 3) & 7), so that a thread writes its 8 values as one chunk and
  // the column reads of the write-out hit 8 different chunks (banks)
  __shared__ __align__(16) uint16_t su[2][kMomTile][kMomTile];
  const float coef = sc->coef * args.gscale;
  const float mu = args.mu;
  // tall matrices: 64 x 64 tiles, 8 column groups x 32 rows of threads (rows r, r + 32)
  const int cg = threadIdx.x & 7;
  const int rr = threadIdx.x >> 3;
  // other matrices: 16 x 256 tiles, a warp per row pair (rows w, w + 8) over 32 column groups
  const int cgw = threadIdx.x & 31;
  const int rrw = threadIdx.x >> 5;
  int ntrans = 0;                   // transposed tiles seen: selects the shared buffer
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const MomTile tl = tiles[t];
    const MuonMat M = mats[tl.mat];
    uint16_t(*sbuf)[kMomTile] = su[ntrans & 1];
    float acc = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = M.transposed ? rr + 32 * half : rrw + 8 * half;
      const int64_t gr = tl.r0 + r;
      const int gc = tl.c0 + (M.transposed ? cg : cgw) * 8;
      float u[8];
      const bool vec = gr < M.m && gc + 8 <= M.n && M.vec;
      if (vec) {
        const int64_t off = gr * (int64_t)M.n + gc;
        float g[8];
        if (M.gdtype == DT_BF16) {
          unpack8(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(M.g) + off)), g);
        } else {
          const float4* gp = reinterpret_cast<const float4*>(static_cast<const float*>(M.g) + off);
          float4 a = __ldg(gp), b = __ldg(gp + 1);
          g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w; g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
        }
        float4* bp = reinterpret_cast<float4*>(M.buf + off);
        float4 b0 = bp[0], b1 = bp[1];
        float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float gh = coef * g[e];
          bb[e] = fmaf(mu, bb[e], gh);
          u[e] = args.nesterov ? fmaf(mu, bb[e], gh) : bb[e];
        }
        bp[0] = make_float4(bb[0], bb[1], bb[2], bb[3]);
        bp[1] = make_float4(bb[4], bb[5], bb[6], bb[7]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          u[e] = 0.f;
          if (gr < M.m && gc + e < M.n) {
            const int64_t off = gr * (int64_t)M.n + gc + e;
            const float g = M.gdtype == DT_BF16 ? bf2f(static_cast<const uint16_t*>(M.g)[off])
                                                 : static_cast<const float*>(M.g)[off];
            const float gh = coef * g;
            const float b = fmaf(mu, M.buf[off], gh);
            M.buf[off] = b;
            u[e] = args.nesterov ? fmaf(mu, b, gh) : b;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(u[e], u[e], acc);
      if (!M.transposed) {
        // X[row][col] = update[row][col], straight from registers
        if (gr < M.m) {
          uint16_t* dst = M.x0 + gr * (int64_t)M.L + gc;
          if (gc + 8 <= M.n) {
            uint4 w;
            w.x = pack2(u[0], u[1]);
            w.y = pack2(u[2], u[3]);
            w.z = pack2(u[4], u[5]);
            w.w = pack2(u[6], u[7]);
            *reinterpret_cast<uint4*>(dst) = w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (gc + e < M.n) dst[e] = f2bf(u[e]);
          }
        }
      } else {
        *reinterpret_cast<uint4*>(&sbuf[r][(cg ^ ((r >> 3) & 7)) * 8]) =
            make_uint4(pack2(u[0], u[1]), pack2(u[2], u[3]), pack2(u[4], u[5]), pack2(u[6], u[7]));
      }
    }
    if (M.transposed) {
      __syncthreads();
      // X[col][row] = update[row][col]: canonical row = parameter column
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cc = rr + 32 * half;
        const int64_t pc = tl.c0 + cc;
        const int pr = tl.r0 + cg * 8;
        if (pc < M.n) {
          uint16_t v[8];
          // rows cg*8 .. cg*8+7 all have (row >> 3) & 7 == cg
          const int col = (((cc >> 3) ^ cg) << 3) | (cc & 7);
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = sbuf[cg * 8 + e][col];
          uint16_t* dst = M.x0 + pc * (int64_t)M.L + pr;
          if (pr + 8 <= M.m) {
            uint4 w;
            w.x = (uint32_t)v[0] | ((uint32_t)v[1] << 16);
            w.y = (uint32_t)v[2] | ((uint32_t)v[3] << 16);
            w.z = (uint32_t)v[4] | ((uint32_t)v[5] << 16);
            w.w = (uint32_t)v[6] | ((uint32_t)v[7] << 16);
            *reinterpret_cast<uint4*>(dst) = w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (pr + e < M.m) dst[e] = v[e];
          }
        }
      }
      ++ntrans;  // the next transposed tile writes the other buffer
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) tile_partials[(size_t)t * kMomWarps + (threadIdx.x >> 5)] = acc;
  }
}

// ---------------------------------------------------------------------------
// Per-matrix Frobenius scale: one 256-thread block per matrix sums the
// matrix's per-warp partials in a fixed order (double precision).
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) ns_prep_kernel(const MuonMat* __restrict__ mats, int nmat,
                                                               const float* __restrict__ part, float eps,
                                                               float* __restrict__ rscale) {
  __shared__ double sh[kPrepThreads / 32];
  const int w = blockIdx.x;
  if (w >= nmat) return;
  const int64_t b = (int64_t)mats[w].tile_begin * kMomWarps, e = (int64_t)mats[w].tile_end * kMomWarps;
  double s = 0.0;
  for (int64_t i = b + threadIdx.x; i < e; i += kPrepThreads) s += (double)part[i];
  const double tot = block_sum_double<kPrepThreads>(s, sh);
  if (threadIdx.x == 0) rscale[w] = (float)(1.0 / (sqrt(tot) + (double)eps));
}

// ---------------------------------------------------------------------------
// Multi-tensor AdamW (decoupled weight decay first, eps outside the sqrt).
// ---------------------------------------------------------------------------
constexpr int kAdamThreads = 256;

__device__ __forceinline__ void adam_one(float& p, float& m, float& v, float g, float coef, const AdamArgs& a,
                                         float decay, float step_size, float inv_sqrt_bc2) {
  const float gh = coef * g;
  m = fmaf(a.beta1, m, a.omb1 * gh);
  v = fmaf(a.beta2, v, a.omb2 * gh * gh);
  const float denom = fmaf(sqrtf(v), inv_sqrt_bc2, a.eps);
  p = fmaf(p, decay, -step_size * (m / denom));
}

__global__ void __launch_bounds__(kAdamThreads) adamw_kernel(const AdamChunk* __restrict__ chunks, int nchunks,
                                                             const StepScalars* __restrict__ sc,
                                                             const __grid_constant__ AdamArgs a) {
  const float coef = sc->coef;
  for (int c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const AdamChunk ch = chunks[c];
    const float decay = a.sp->adam_decay[ch.group], step_size = a.sp->adam_step[ch.group];
    const float inv_sqrt_bc2 = a.sp->adam_inv_sqrt_bc2;
    const int64_t nv = ch.vec ? ch.n / 4 : 0;
    float4* pv = reinterpret_cast<float4*>(ch.p);
    float4* mv = reinterpret_cast<float4*>(ch.m);
    float4* vv = reinterpret_cast<float4*>(ch.v);
    for (int64_t i = threadIdx.x; i < nv; i += kAdamThreads) {
      float4 p = pv[i], m = mv[i], v = vv[i];
      float g[4];
      if (ch.gdtype == DT_BF16) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(ch.g) + i);
        g[0] = __uint_as_float(w.x << 16);
        g[1] = __uint_as_float(w.x & 0xFFFF0000u);
        g[2] = __uint_as_float(w.y << 16);
        g[3] = __uint_as_float(w.y & 0xFFFF0000u);
      } else {
        const float4 w = __ldg(reinterpret_cast<const float4*>(ch.g) + i);
        g[0] = w.x; g[1] = w.y; g[2] = w.z; g[3] = w.w;
      }
      adam_one(p.x, m.x, v.x, g[0], coef, a, decay, step_size, inv_sqrt_bc2);
      adam_one(p.y, m.y, v.y, g[1], coef, a, decay, step_size, inv_sqrt_bc2);
      adam_one(p.z, m.z, v.z, g[2], coef, a, decay, step_size, inv_sqrt_bc2);
      adam_one(p.w, m.w, v.w, g[3], coef, a, decay, step_size, inv_sqrt_bc2);
      pv[i] = p;
      mv[i] = m;
      vv[i] = v;
      if (ch.shadow) {
        uint2 s;
        s.x = pack2(p.x, p.y);
        s.y = pack2(p.z, p.w);
        reinterpret_cast<uint2*>(ch.shadow)[i] = s;
      }
    }
    for (int64_t j = nv * 4 + threadIdx.x; j < ch.n; j += kAdamThreads) {
      float p = ch.p[j], m = ch.m[j], v = ch.v[j];
      const float g = ch.gdtype == DT_BF16 ? bf2f(static_cast<const uint16_t*>(ch.g)[j])
                                            : static_cast<const float*>(ch.g)[j];
      adam_one(p, m, v, g, coef, a, decay, step_size, inv_sqrt_bc2);
      ch.p[j] = p;
      ch.m[j] = m;
      ch.v[j] = v;
      if (ch.shadow) ch.shadow[j] = f2bf(p);
    }
  }
}

}  // namespace

void launch_grad_sumsq(const GradChunk* chunks, int nchunks, float* partials, int grid, cudaStream_t st) {
  grad_sumsq_kernel<<<grid, kNormThreads, 0, st>>>(chunks, nchunks, partials);
}

void launch_clip_finalize(const float* partials, int n, float max_norm, float clip_eps, StepScalars* out,
                          cudaStream_t st) {
  clip_finalize_kernel<<<1, kClipThreads, 0, st>>>(partials, n, max_norm, clip_eps, out);
}

void launch_sumsq_partials(const float* partials, int n, double* out, cudaStream_t st) {
  sumsq_partials_kernel<<<1, kClipThreads, 0, st>>>(partials, n, out);
}

void launch_clip_from_sumsq(const double* sumsq, float max_norm, float clip_eps, StepScalars* out, cudaStream_t st) {
  clip_from_sumsq_kernel<<<1, 1, 0, st>>>(sumsq, max_norm, clip_eps, out);
}

void launch_muon_momentum(const MomTile* tiles, int ntiles, const MuonMat* mats, const StepScalars* sc,
                          MomArgs args, float* tile_partials, int grid, cudaStream_t st) {
  muon_momentum_kernel<<<grid, kMomThreads, 0, st>>>(tiles, ntiles, mats, sc, args, tile_partials);
}

void launch_ns_prep(const MuonMat* mats, int nmat, const float* tile_partials, float eps, float* rscale,
                    cudaStream_t st) {
  if (nmat > 0) ns_prep_kernel<<<nmat, kPrepThreads, 0, st>>>(mats, nmat, tile_partials, eps, rscale);
}

void launch_adamw(const AdamChunk* chunks, int nchunks, const StepScalars* sc, AdamArgs args, int grid,
                  cudaStream_t st) {
  adamw_kernel<<<grid, kAdamThreads, 0, st>>>(chunks, nchunks, sc, args);
}

}  // namespace ma
