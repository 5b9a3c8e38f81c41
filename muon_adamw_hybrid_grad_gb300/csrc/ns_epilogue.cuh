// Element-level epilogue of the three Newton-Schulz GEMMs (device code).
//
// Newton-Schulz as described in the OpenDM article (核心揭秘一 / Muon 的工作原理):
// five iterations of  A = X X^T,  B = b A + c A A,  X <- a X + B X,  on the
// short side of the update, starting from X0 = update / (||update||_F + eps).
// The factor a is folded into B (B = a I + b A + c A A), so the update is
// the plain product X' = B X and its epilogue reads nothing back; the bf16
// rounding points stay those of the textbook order (X, A and B stored in
// bf16), which keeps the error of the original evaluation. The
// normalisation is folded in too: X0 is stored unscaled (U) and
// r = 1/(||U||+eps) is applied as r^2 to the first Gram matrix and r to the
// first X update. The last update does not store X: it applies the Muon
// step to the fp32 master weights (transposing back for tall matrices):
//   p <- p * (1 - lr * wd) - lr * muon_lr_scale * 0.2 * sqrt(max(m, n)) * O.
// Padding rows/cols of the workspaces are never written, so they stay zero.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace ma {

__device__ __forceinline__ float ns_bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t ns_f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Store one output element (i, j) of matrix `mat` (index within the bucket).
__device__ __forceinline__ void ns_epilogue_element(const NsProblem& pb, const NsEpiArgs& ep, int mat, int i, int j,
                                                    float acc) {
  const MuonMat& M = pb.mats[mat];
  if (pb.kind == NS_GRAM || pb.kind == NS_POLY) {
    if (i >= M.s || j >= M.s || j > i) return;
    const size_t base = (size_t)mat * pb.S * pb.S;
    float v;
    if (pb.kind == NS_GRAM) {
      const float r = pb.first ? pb.rscale[mat] : 1.f;
      v = acc * (r * r);
    } else {
      v = fmaf(ep.c, acc, fmaf(ep.b, ns_bf2f(pb.aux[base + (size_t)i * pb.S + j]), i == j ? ep.a : 0.f));
    }
    const uint16_t h = ns_f2bf(v);
    pb.out[base + (size_t)i * pb.S + j] = h;
    if (i != j) pb.out[base + (size_t)j * pb.S + i] = h;
    return;
  }
  // NS_UPDATE
  if (i >= M.s || j >= M.l) return;
  const size_t idx = (size_t)mat * pb.S * pb.L + (size_t)i * pb.L + j;
  const float v = pb.first ? acc * pb.rscale[mat] : acc;
  if (!pb.last) {
    pb.out[idx] = ns_f2bf(v);
    return;
  }
  const int pi = M.transposed ? j : i;
  const int pj = M.transposed ? i : j;
  const size_t po = (size_t)pi * M.n + pj;
  const float p = fmaf(M.p[po], ep.sp->ns_decay[M.group], -(ep.sp->ns_lr * M.lr_mult) * v);
  M.p[po] = p;
  if (M.shadow) M.shadow[po] = ns_f2bf(p);
}

}  // namespace ma
