// Newton-Schulz grouped GEMMs on the 5th-generation tensor cores (sm_103a).
//
// Newton-Schulz orthogonalisation as described in the OpenDM article
// (核心揭秘一 / Muon 的工作原理): A = X X^T, B = b A + c A A, X <- a X + B X,
// five times, on the short side, evaluated as A = X X^T, B = a I + b A + c A A,
// X' = B X so that the largest product's epilogue reads nothing back. Each
// ns_tc_kernel launch covers one of the three products for every Muon matrix
// of up to four shape buckets; the last iteration's B X updates the
// parameters in its epilogue instead of storing X'.
//
// ns_tc_kernel (one persistent CTA per SM, 320 threads):
//   warp 0     TMA producer: 128x64 tiles of the left operand and the CTA's
//              part of the right-hand tile into a shared-memory ring
//              (128-byte swizzle; 6 stages of 32 KiB for CTA pairs, 4 of
//              48 KiB otherwise, fewer for the last iteration), completion
//              tracked by mbarrier transaction counts;
//   warp 1     allocates 512 TMEM columns; one lane issues tcgen05.mma
//              kind::f16 (bf16 x bf16 -> fp32), either cta_group::2 with
//              M = 256 over a CTA pair (X X^T, A A, last iteration) or
//              cta_group::1 with M = 128 in a CTA of its own (B X), and
//              commits stage releases and accumulator-ready signals to
//              mbarriers; every operand copy is a plain TMA load into the
//              shared memory of the CTA that reads it;
//   warps 2-9  epilogue: tcgen05.ld of the fp32 accumulator (a warp may only
//              read its TMEM lane quarter, warp % 4; two warps share each
//              quarter and take alternate 32-column blocks), the fused
//              polynomial, bf16 staging tiles leaving through TMA stores
//              (the last iteration: fp32 parameter blocks in and out by TMA).
// Two accumulators (2 x 256 columns) let the epilogue of one tile overlap
// the main loop of the next. X X^T and A A are symmetric: only output tiles
// that touch the lower triangle are computed and the epilogue mirrors them;
// on a diagonal unit the left tile also serves as the right-hand operand.
// Units reach clusters in a longest-first order fixed at planning time, and
// consecutive launches overlap their set-up with the previous launch's tail
// (programmatic dependent launch).
//
// ns_small_kernel takes buckets of small matrices (canonical S = 128,
// L <= 512) through every iteration and the update in one launch, one CTA
// per matrix with X, A and B resident in shared memory.
//
// Every mbarrier wait is bounded (kWaitLimitNs of wall time). On expiry the
// CTA records an error code in the device flag, the other roles stop at
// their next wait, in-flight copies and MMAs are drained (again bounded)
// and TMEM is released before the CTA exits.
#include <cuda.h>
#include <stdio.h>
#include <string.h>

#include <queue>
#include <utility>

#include "internal.h"
#include "ns_epilogue.cuh"

namespace ma {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int A_STAGE = BM * BK * 2;      // 16 KB
constexpr int B_STAGE = BN_MAX * BK * 2;  // 32 KB
constexpr int EPI_WARPS = 8;  // two warps per TMEM lane quarter, splitting the columns
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int PBLOCK_BYTES = 32 * 32 * 4;  // one 32x32 fp32 parameter block
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Shared-memory layout (offsets from the 1024-byte aligned base). A stage
// holds one 64-wide k-block of both operands: for a CTA that runs its own
// MMAs, its 128 rows of the left operand and the whole right-hand tile; for a
// CTA pair running one M = 256 MMA (PAIR), each CTA's own 128 rows and its
// half of the right-hand tile, so a stage is two thirds of the bytes and the
// ring deepens from 4 to 6 stages (the main loop is bound by TMA latency,
// not by bandwidth). The
// last iteration's variant (APPLY) trades operand stages for two parameter
// blocks per epilogue warp, into which p is fetched by TMA ahead of use.
//   [stages][APPLY: 2 fp32 blocks per epilogue warp][bf16 tiles per epilogue warp][mbarriers, TMEM slot, flag]
// Without bf16 shadows (SHADOW false) the last iteration's variant needs no
// shadow tiles, and its paired ring gets a fifth stage in their place.
template <bool PAIR, bool APPLY, bool SHADOW = true>
struct Smem {
  static constexpr int STAGE = A_STAGE + (PAIR ? B_STAGE / 2 : B_STAGE);
  static constexpr int STAGES = PAIR ? (APPLY ? (SHADOW ? 4 : 5) : 6) : (APPLY ? 3 : 4);
  static constexpr size_t PBUF = (size_t)STAGES * STAGE;
  static constexpr size_t SB = PBUF + (APPLY ? (size_t)EPI_WARPS * 2 * PBLOCK_BYTES : 0);
  // bf16 tiles per epilogue warp: APPLY the shadow tile (none without shadows); otherwise a row
  // tile and a column tile
  static constexpr size_t SB_PER_WARP = APPLY ? (SHADOW ? 2048 : 0) : 4096;
  static constexpr size_t BARS = SB + (size_t)EPI_WARPS * SB_PER_WARP;
  // full[S], empty[S], tmem full[2], tmem empty[2], drain, APPLY: parameter blocks [2 per epilogue warp]
  static constexpr int NBARS = 2 * STAGES + 5 + (APPLY ? 2 * EPI_WARPS : 0);
  static constexpr size_t BYTES = 1024 + BARS + 256;
  static_assert(NBARS * 8 + 8 <= 256, "barrier area");
  static_assert(BYTES <= 232448, "shared memory per CTA");
};

// error codes written to the device flag
constexpr int kErrWaitProducer = 0x101;
constexpr int kErrWaitMma = 0x102;
constexpr int kErrWaitEpilogue = 0x103;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// CLUSTER: acquire at cluster scope (arrivals from the other CTA of a pair).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (CLUSTER)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  return ok != 0;
}

// Wait until the phase of parity `parity` of `bar` has completed. Returns
// false if the CTA is aborting or the wait ran past the limit (then the
// abort flag and the device error code are set).
template <bool CLUSTER = false>
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                            int code) {
  const uint64_t t0 = global_timer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicCAS(err, 0, code);
        return false;
      }
    }
  }
}

// The common case (the phase has already completed, or completes within the
// instruction's own suspend window) stays inline on the issuing warps' paths.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, int code) {
  if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
  return mbar_wait_slow<CLUSTER>(bar, parity, abort_flag, err, code);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Bulk tensor store of a shared-memory box (elements outside the tensor are
// not written), tracked in this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Until every bulk store this thread committed has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Generic-proxy writes to shared memory become visible to the TMA (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// tcgen05 operations of one CTA (CL = 1) or of a CTA pair (CL = 2: one MMA of
// M = 256 issued by the even CTA covers both CTAs' operands and accumulators).
template <int CL>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (CL == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` (this CTA) once this thread's prior MMAs have completed.
template <int CL>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if constexpr (CL == 1)
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

template <int CL>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  if constexpr (CL == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    // one warp of each CTA of the pair, collectively: the same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int CL>
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  if constexpr (CL == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

// Address of this CTA's shared-memory location `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// The MMAs of a CTA pair (issued by the even CTA) have completed: one
// arrival on the mbarrier at offset `bar` in each CTA of the pair, as two
// commits (the executing CTA's own barrier, then the odd CTA's, addressed
// through the cluster window).
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  umma_commit<2>(bar);
  umma_commit<2>(mapa_shared(bar, 1));
}

// Arrive on an mbarrier of any CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of the pair's other CTA (cluster address `bar`).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1.
//   K-major: rows of 64 bf16 (128 B); 8-row groups 1024 B apart (SBO).
//   MN-major: rows = K index, 64 MN-elements per 128 B row; 8-row groups
//   1024 B apart (SBO); 64-element MN panels `panel_bytes` apart (LBO).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B,
// A K-major, B K-major or MN-major, M = m (128, or 256 for a CTA pair), N = n.
__device__ __forceinline__ uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;   // D format: f32
  d |= 1u << 7;   // A format: bf16
  d |= 1u << 10;  // B format: bf16
  if (b_mn_major) d |= 1u << 16;
  d |= (uint32_t)(n >> 3) << 17;
  d |= (uint32_t)(m >> 4) << 24;
  return d;
}

struct TileCoord {
  int prob, mat, ti, tj;
};

// Work unit g -> (problem, matrix, row unit, column block). A row unit is
// L.cl consecutive 128-row blocks (one per CTA of the cluster).
// The work unit at position `pos` of the launch's order (no table: the
// plain round-robin order, position = unit).
__device__ __forceinline__ int unit_at(const TcLaunch& L, int pos) {
  return L.order != nullptr ? __ldg(L.order + pos) : pos;
}

__device__ __forceinline__ TileCoord decode_tile(const TcLaunch& L, int g) {
  TileCoord c{0, 0, 0, 0};
  int pi = 0;
  while (pi + 1 < L.nprob && g >= L.prob[pi + 1].tile_begin) ++pi;
  const TcProblem& P = L.prob[pi];
  const int local = g - P.tile_begin;
  c.prob = pi;
  c.mat = local / P.tiles_per_mat;
  int t = local - c.mat * P.tiles_per_mat;
  if (P.p.kind == NS_UPDATE) {
    c.ti = t / P.tiles_n;
    c.tj = t - c.ti * P.tiles_n;
  } else {
    // row unit ti holds the tiles whose columns start at or before its last row
    const int bmu = BM * L.cl;
    int ti = 0;
    for (;;) {
      const int cnt = (ti * bmu + bmu - 1) / P.bn + 1;
      if (t < cnt) break;
      t -= cnt;
      ++ti;
    }
    c.ti = ti;
    c.tj = t;
  }
  return c;
}


// A symmetric product's unit whose right-hand rows (this CTA's part of the
// column block) are this CTA's own left-hand rows: the stage's left tile then
// serves as the right-hand operand too and the second copy is not loaded.
__device__ __forceinline__ bool rhs_is_lhs(const TcProblem& P, const TileCoord& c, int cl, uint32_t crank) {
  const int nown = P.bn / cl;
  return P.p.kind != NS_UPDATE && nown == BM && c.tj * P.bn + (int)crank * nown == (c.ti * cl + (int)crank) * BM;
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Two floats rounded to nearest-even bf16 in one conversion: lo in the low
// half, hi in the high half (the same rounding as two scalar conversions).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Epilogue of one 32x32 block of the accumulator for A = X X^T,
// B = a I + b A + c A A and the iterations' X' = B X (the last iteration has
// its own epilogue): rows row0..row0+31 (this warp's TMEM lane quarter; lane
// l holds row row0 + l), columns col0..col0+31 of matrix `mat`. Values are
// computed in registers, written as bf16 into the warp's 2 KiB row tile `rt`
// in the 64-byte swizzle layout (the 16-byte chunk q of row r at
// q ^ ((r >> 1) & 3)) and leave with one TMA store, so that no global store
// passes through the load/store units the operand feed shares. The
// symmetric products store only blocks on or below the diagonal: a block
// below it also leaves transposed, from the column tile that follows `rt`,
// at the mirrored position; a block on it is completed to a symmetric block
// in `rt` (upper half taken from the lower one) before its store, so every
// element is written exactly once. Elements outside the matrix are stored as
// zero (the workspaces' padding stays zero). Only the b A term of B is read
// from memory, issued before TMEM is read so that its latency overlaps it.
__device__ __forceinline__ void epilogue_block(const NsProblem& pb, const CUtensorMap* tmo, const NsEpiArgs& ep,
                                               int mat, int row0, int col0, uint32_t taddr, uint8_t* rt, int lane) {
  const MuonMat& M = pb.mats[mat];
  const int s = M.s;
  const bool update = pb.kind == NS_UPDATE;
  const int lim = update ? M.l : s;          // valid columns
  if (row0 >= s || col0 >= lim) return;      // padding only: never written
  if (!update && col0 >= row0 + 32) return;  // above the diagonal: the mirror of a lower block
  const int gi = row0 + lane;
  // warp-uniform: the block lies inside the matrix (no element to zero)
  const bool inside = row0 + 32 <= s && col0 + 32 <= lim;
  uint4 preA[4];
  if (pb.kind == NS_POLY) {
#pragma unroll
    for (int q = 0; q < 4; ++q) preA[q] = make_uint4(0u, 0u, 0u, 0u);
    if (gi < s) {  // A is stored in full (mirrored); padding is zero
      const uint4* ap = reinterpret_cast<const uint4*>(pb.aux + (size_t)mat * pb.S * pb.S + (size_t)gi * pb.S + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) preA[q] = __ldg(ap + q);
    }
  }
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
  float o[32];
  if (pb.kind == NS_POLY) {
    // c (A A) + (b A + a I); the a I term only in blocks on the diagonal
    const bool on_diag = col0 == row0;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const uint32_t u = u4_get(preA[e >> 3], (e >> 1) & 3);
      const float a = __uint_as_float((e & 1) ? (u & 0xFFFF0000u) : (u << 16));
      const float lin = on_diag ? fmaf(ep.b, a, e == lane ? ep.a : 0.f) : ep.b * a;
      o[e] = fmaf(ep.c, __uint_as_float(r[e]), lin);
    }
  } else if (pb.first) {
    // first iteration: the Frobenius scale r (r^2 for A = X X^T)
    const float rs = pb.rscale[mat];
    const float sc = update ? rs : rs * rs;
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]) * sc;
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]);
  }
  if (!inside) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (gi >= s || col0 + e >= lim) o[e] = 0.f;
  }

  uint8_t* const ct = rt + 2048;
  if (lane == 0) bulk_wait_read_all();  // the previous block's stores have read both tiles
  __syncwarp();
  uint32_t pk[16];  // this lane's row as bf16 pairs (columns 2j, 2j + 1)
#pragma unroll
  for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
  uint4* const rrow = reinterpret_cast<uint4*>(rt + lane * 64);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    rrow[q ^ ((lane >> 1) & 3)] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  // blocks are 32-aligned: one meets the diagonal iff col0 == row0
  const bool diag = !update && col0 == row0;
  const bool below = !update && col0 + 32 <= row0;
  if (below) {
    // transposed tile T[c][r] = block[r][c], written as bf16 pairs: lanes 2k
    // and 2k + 1 swap their packed rows; the even lane writes T[2j][2k..2k+1]
    // (both low halves), the odd lane T[2j+1][2k..2k+1] (both high halves)
    const uint32_t sel = (lane & 1) ? 0x3276u : 0x5410u;
    uint8_t* const tb = ct + (lane & 1) * 64 + ((lane >> 1) & 3) * 4;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t oth = __shfl_xor_sync(0xffffffffu, pk[j], 1);
      *reinterpret_cast<uint32_t*>(tb + 2 * j * 64 + (((lane >> 3) ^ (j & 3)) << 4)) = __byte_perm(pk[j], oth, sel);
    }
  } else if (diag) {
    __syncwarp();
    // (row e, column lane) for e < lane <- (row lane, column e)
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < lane)
        *reinterpret_cast<uint16_t*>(rt + e * 64 + (((lane >> 3) ^ ((e >> 1) & 3)) << 4) + (lane & 7) * 2) =
            ns_f2bf(o[e]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const int y = mat * pb.S;
    tma_store_2d(tmo, smem_u32(rt), col0, y + row0);
    if (below) tma_store_2d(tmo, smem_u32(ct), row0, y + col0);
    bulk_commit();
  }
}

// An epilogue warp is done reading an accumulator from TMEM: one arrival per
// warp on the MMA issuer's barrier (the leader's, for a CTA pair).
template <bool PAIR>
__device__ __forceinline__ void release_accumulator(uint32_t tempty, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (PAIR)
      mbar_arrive_cluster(mapa_shared(tempty, 0));
    else
      mbar_arrive(tempty);
  }
}

// Last-iteration update of one 32x32 block straight from registers, for
// parameters without TMA maps (unaligned rows or fewer than 32 of either
// side): lane l holds canonical row row0 + l, columns col0..col0+31. Tall
// parameters are read and written along their rows, so that the lanes'
// addresses are contiguous; the others one element per lane-row.
__device__ __forceinline__ void apply_block_direct(const MuonMat& M, const NsEpiArgs& ep, float rs, int row0,
                                                   int col0, uint32_t taddr, int lane) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait();
  // the descriptor's fields in registers (the stores below could otherwise
  // alias it), and every load issued before the first store
  float* const P = M.p;
  uint16_t* const SH = M.shadow;
  const size_t n = (size_t)M.n;
  const bool tr = M.transposed != 0;
  const int gi = row0 + lane;
  const int cnt = M.l - col0 < 32 ? M.l - col0 : 32;
  if (gi >= M.s || cnt <= 0) return;
  const float lrm = ep.sp->ns_lr * M.lr_mult;
  const float dec = ep.sp->ns_decay[M.group];
  float pv[32];
#pragma unroll
  for (int e = 0; e < 32; ++e)
    pv[e] = e < cnt ? P[tr ? (size_t)(col0 + e) * n + gi : (size_t)gi * n + col0 + e] : 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    if (e < cnt) {
      const size_t po = tr ? (size_t)(col0 + e) * n + gi : (size_t)gi * n + col0 + e;
      const float q = fmaf(pv[e], dec, -lrm * (__uint_as_float(r[e]) * rs));
      P[po] = q;
      if (SH) SH[po] = ns_f2bf(q);
    }
  }
}

// Epilogue of the last Newton-Schulz iteration:
//   p <- p (1 - lr wd) - lr_eff O,  O = B X read from TMEM and never stored.
// For a matrix with TMA maps, each epilogue warp owns two 4 KiB fp32 block
// buffers and its 2 KiB bf16 tile. When a tile starts (while its main loop
// still runs) the warp fetches the parameter blocks of its first two 32x32
// blocks by TMA; block k+1 is fetched as block k starts, into the buffer that
// block k-1's stores have left. A block is updated in place in shared memory
// and leaves through TMA stores of p and of its bf16 shadow. Elements outside
// the parameter read as zero and are not written (the store clips them).
// Blocks sit in shared memory in the 128-byte (fp32) and 64-byte (bf16)
// swizzle layouts: the 16-byte chunk q of row r is at q ^ (r & 7), resp.
// q ^ ((r >> 1) & 3), which keeps both the row-per-lane accesses (parameter
// row = TMEM lane) and the column-per-lane ones (tall parameters, parameter
// column = TMEM lane) free of bank conflicts. Matrices without maps take
// apply_block_direct.
template <int CL, bool PAIR, bool SHADOW>
__device__ __forceinline__ void apply_epilogue(const TcLaunch& L, uint8_t* smem, size_t pbuf_off, size_t sb_off,
                                               uint32_t pbar_base, uint32_t tmem_base, uint32_t tfull0,
                                               uint32_t tempty0, volatile int* abort_flag, int warp, int lane,
                                               uint32_t crank, int unit0, int nunits) {
  const int w8 = warp - 2;
  const int quarter = warp & 3;
  const int half = w8 >> 2;
  uint8_t* const pb = smem + pbuf_off + (size_t)w8 * 2 * PBLOCK_BYTES;
  const uint32_t pb_s = smem_u32(pb);
  uint8_t* const shb = smem + sb_off + (size_t)w8 * Smem<PAIR, true, SHADOW>::SB_PER_WARP;
  const uint32_t shb_s = smem_u32(shb);
  const uint32_t bar0 = pbar_base + 16u * (uint32_t)w8;
  const NsEpiArgs& ep = L.epi;
  uint32_t ph = 0;    // bit b: parity of the next completion of buffer b
  uint32_t pend = 0;  // bit b: a load into buffer b is in flight
  int acc = 0;
  uint32_t acc_phase = 0;
  int g_next = unit0 < L.npos ? unit_at(L, unit0) : -1;
  for (int pos = unit0; pos < L.npos; pos += nunits) {
    const int g = g_next;  // read one unit ahead, off this unit's critical path
    g_next = pos + nunits < L.npos ? unit_at(L, pos + nunits) : -1;
    if (g < 0) continue;
    const TileCoord c = decode_tile(L, g);
    const TcProblem& P = L.prob[c.prob];
    const MuonMat& M = P.p.mats[c.mat];
    const int row0 = (c.ti * CL + (int)crank) * BM + quarter * 32;
    const int nb = P.bn / 64;                       // blocks of this warp in the tile
    const int colw = c.tj * P.bn + 32 * half;       // canonical column of block 0; block k at +64k
    const bool tma = M.tma != 0;
    const bool tr = M.transposed != 0;
    const bool has_shadow = SHADOW && M.shadow != nullptr;
    const int s = M.s, l = M.l;
    const CUtensorMap* maps = P.p.pmaps + 2 * c.mat;
    if (tma) {
      if (lane == 0) {
        bulk_wait_read_all();  // the previous tile's stores have left both buffers
        for (int k = 0; k < 2 && k < nb; ++k) {
          const int cc = colw + 64 * k;
          if (row0 < s && cc < l) {
            mbar_expect_tx(bar0 + 8 * k, PBLOCK_BYTES);
            tma_load_2d(pb_s + k * PBLOCK_BYTES, maps, tr ? row0 : cc, tr ? cc : row0, bar0 + 8 * k);
          }
        }
      }
      for (int k = 0; k < 2 && k < nb; ++k)
        if (row0 < s && colw + 64 * k < l) pend |= 1u << k;
      __syncwarp();
    }
    const bool got = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, L.err, kErrWaitEpilogue);
    if (!__all_sync(0xffffffffu, got)) break;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN_MAX);
    bool ok = true;
    for (int k = 0; k < nb; ++k) {
      const int c0 = 32 * half + 64 * k;
      const int cc = c.tj * P.bn + c0;
      if (!tma) {
        apply_block_direct(M, ep, P.p.first ? P.p.rscale[c.mat] : 1.f, row0, cc, tbase + (uint32_t)c0, lane);
        continue;
      }
      if (k >= 1) {
        const int cn = cc + 64;
        const bool next = k + 1 < nb && row0 < s && cn < l;
        if (lane == 0) {
          bulk_wait_read_all();  // block k-1's stores have read its buffer and the bf16 tile
          if (next) {
            const int b = (k + 1) & 1;
            mbar_expect_tx(bar0 + 8 * b, PBLOCK_BYTES);
            tma_load_2d(pb_s + b * PBLOCK_BYTES, maps, tr ? row0 : cn, tr ? cn : row0, bar0 + 8 * b);
          }
        }
        if (next) pend |= 1u << ((k + 1) & 1);
        __syncwarp();
      }
      if (!(row0 < s && cc < l)) continue;
      uint32_t r[32];
      tmem_ld_32x32b_x32(tbase + (uint32_t)c0, r);
      tmem_ld_wait();
      const int b = k & 1;
      const bool in = mbar_wait(bar0 + 8 * b, (ph >> b) & 1u, abort_flag, L.err, kErrWaitEpilogue);
      if (!__all_sync(0xffffffffu, in)) {
        ok = false;
        break;
      }
      ph ^= 1u << b;
      pend &= ~(1u << b);
      const float rs = P.p.first ? P.p.rscale[c.mat] : 1.f;
      const float lrm = ep.sp->ns_lr * M.lr_mult;
      const float dec = ep.sp->ns_decay[M.group];
      float o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]) * rs;
      uint8_t* const buf = pb + b * PBLOCK_BYTES;
      if (!tr) {
        // lane = parameter row row0 + lane; TMEM column e = parameter column cc + e
        float4* const prow = reinterpret_cast<float4*>(buf + lane * 128);
        uint4* const srow = reinterpret_cast<uint4*>(shb + lane * 64);
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          float4 v0 = prow[q ^ (lane & 7)];
          float4 v1 = prow[(q + 1) ^ (lane & 7)];
          v0.x = fmaf(v0.x, dec, -lrm * o[4 * q + 0]);
          v0.y = fmaf(v0.y, dec, -lrm * o[4 * q + 1]);
          v0.z = fmaf(v0.z, dec, -lrm * o[4 * q + 2]);
          v0.w = fmaf(v0.w, dec, -lrm * o[4 * q + 3]);
          v1.x = fmaf(v1.x, dec, -lrm * o[4 * q + 4]);
          v1.y = fmaf(v1.y, dec, -lrm * o[4 * q + 5]);
          v1.z = fmaf(v1.z, dec, -lrm * o[4 * q + 6]);
          v1.w = fmaf(v1.w, dec, -lrm * o[4 * q + 7]);
          prow[q ^ (lane & 7)] = v0;
          prow[(q + 1) ^ (lane & 7)] = v1;
          if (has_shadow)
            srow[(q >> 1) ^ ((lane >> 1) & 3)] = make_uint4(pack_bf16x2(v0.x, v0.y), pack_bf16x2(v0.z, v0.w),
                                                            pack_bf16x2(v1.x, v1.y), pack_bf16x2(v1.z, v1.w));
        }
      } else {
        // lane = parameter column row0 + lane; TMEM column e = parameter row cc + e
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float* const a = reinterpret_cast<float*>(buf + e * 128 + ((((lane >> 2) ^ (e & 7))) << 4) + (lane & 3) * 4);
          const float q = fmaf(*a, dec, -lrm * o[e]);
          *a = q;
          if (has_shadow)
            *reinterpret_cast<uint16_t*>(shb + e * 64 + ((((lane >> 3) ^ ((e >> 1) & 3))) << 4) + (lane & 7) * 2) =
                ns_f2bf(q);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int x = tr ? row0 : cc, y = tr ? cc : row0;
        tma_store_2d(maps, pb_s + b * PBLOCK_BYTES, x, y);
        if (has_shadow) tma_store_2d(maps + 1, shb_s, x, y);
        bulk_commit();
      }
    }
    if (!ok) break;
    release_accumulator<PAIR>(tempty0 + 8 * acc, lane);
    if (++acc == 2) {
      acc = 0;
      acc_phase ^= 1u;
    }
  }
  // Drain: the stores have read shared memory and loads still in flight
  // (after an abort) have landed before the CTA may leave.
  if (lane == 0) bulk_wait_read_all();
  for (int b = 0; b < 2; ++b) {
    if ((pend >> b) & 1u) {
      const uint64_t t0 = global_timer();
      while (!mbar_try_wait(bar0 + 8 * b, (ph >> b) & 1u)) {
        if (global_timer() - t0 > kWaitLimitNs) {
          atomicCAS(L.err, 0, kErrWaitEpilogue);
          break;
        }
      }
    }
  }
  __syncwarp();
}

// CL = 1: one CTA per work unit, running its own M = 128 MMAs (X' = B X of
// iterations 1 .. n-1, and every product when pairs are switched off).
// CL = 2 (PAIR): a cluster of two CTAs per unit of two adjacent 128-row
// blocks that share the right-hand operand tile, running
// tcgen05.mma.cta_group::2 with M = 256. The even CTA (leader) issues every
// MMA, which reads each CTA's own 128 rows of the left operand and each CTA's
// half of the right-hand tile from that CTA's shared memory and accumulates
// into each CTA's own TMEM. Both CTAs load their parts by TMA; the odd CTA's
// copies complete on the leader's full barrier, whose expected byte count
// covers both. The leader's commits release each stage and each accumulator
// in both CTAs; both CTAs' epilogue warps release the accumulator on the
// leader's barrier. Used where the right-hand operand is K-major (X X^T, A A)
// and for the last iteration. No operand tile is ever multicast: each CTA
// loads exactly the bytes its own shared memory holds.
template <int CL, bool APPLY, bool PAIR, bool SHADOW = true>
__global__ void __launch_bounds__(THREADS, 1) ns_tc_kernel(const __grid_constant__ TcLaunch L) {
  static_assert(PAIR == (CL == 2), "a cluster of two CTAs runs the paired MMA");
  constexpr int G = PAIR ? 2 : 1;  // tcgen05 cta_group
  using SM = Smem<PAIR, APPLY, SHADOW>;
  static_assert((SM::BYTES >> 4) < 0x4000, "operand descriptors: 14-bit address field");
  constexpr int STAGES = SM::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::BARS);
  // bars[0..S): full, [S..2S): empty, [2S..2S+2): tmem full, [2S+2..2S+4): tmem empty, [2S+4]: drain,
  // APPLY: [2S+5 + 2w + b): parameter block b of epilogue warp w
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + SM::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t crank = CL == 2 ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const bool issues_mma = !PAIR || leader;
  const int unit0 = blockIdx.x / CL;  // this cluster's first position in the work order
  const int nunits = gridDim.x / CL;  // clusters in the grid

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);  // one producer arrival + the bytes of every copy
      // one commit from the CTA that issues the MMAs (both CTAs' parts, PAIR)
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      // one arrival per epilogue warp of each CTA whose TMEM the MMAs write
      mbar_init(tempty0 + 8 * a, (PAIR ? 2 : 1) * EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int i = 2 * STAGES + 5; i < SM::NBARS; ++i) mbar_init(smem_u32(bars + i), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) tmem_alloc<G>(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  if (CL == 2) cluster_sync();  // the peer's barriers exist before any copy or commit reaches them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched with programmatic stream serialization: the set-up above may
  // overlap the previous launch's last CTAs; every global access below comes
  // after that launch has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next launch may start its own set-up as this launch's CTAs leave
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (every CTA) ----------------
      for (int p = 0; p < L.nprob; ++p) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L.prob[p].tmP)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L.prob[p].tmQ)) : "memory");
      }
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      // test hook: with stall_test, CTA 0 issues nothing, so its MMA warp's
      // bounded wait for the first stage runs out and reports the error
      bool ok = !(L.stall_test && blockIdx.x == 0);
      int g_next = unit0 < L.npos ? unit_at(L, unit0) : -1;
      for (int pos = unit0; pos < L.npos && ok; pos += nunits) {
        const int g = g_next;  // read one unit ahead, off this unit's critical path
        g_next = pos + nunits < L.npos ? unit_at(L, pos + nunits) : -1;
        if (g < 0) continue;
        const TileCoord c = decode_tile(L, g);
        const TcProblem& P = L.prob[c.prob];
        const int kblocks = P.p.K / BK;
        const int rowP = c.mat * P.p.M + (c.ti * CL + (int)crank) * BM;
        const bool sym = P.p.kind != NS_UPDATE;
        // this CTA's part of the right-hand tile: columns [n0, n0 + bn / CL) of the
        // column block (the whole block for CL = 1, half of it for a pair), in
        // boxes of 128 rows (K-major) or 64 columns (MN-major)
        const int nown = P.bn / CL;
        const int n0 = c.tj * P.bn + (int)crank * nown;
        const int nbox = sym ? nown / BM : nown / 64;
        const bool same = rhs_is_lhs(P, c, CL, crank);
        // bytes landing in this CTA per stage: its left rows + its part of the right tile
        const uint32_t tx = (uint32_t)(A_STAGE + (same ? 0 : nown * BK * 2));
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, L.err, kErrWaitProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = smem_u32(smem + (size_t)stage * SM::STAGE);
          const uint32_t sb = sa + A_STAGE;
          if (issues_mma) {
            mbar_expect_tx(fb, (PAIR ? 2u : 1u) * tx);  // PAIR: both CTAs' copies complete here
            tma_load_2d(sa, &P.tmP, kb * BK, rowP, fb);
          } else {
            tma_load_2d_pair(sa, &P.tmP, kb * BK, rowP, mapa_shared(fb, 0));
          }
          for (int q = 0; q < (same ? 0 : nbox); ++q) {
            // sym: rows (column block) of the same matrix, K-major; update: X, MN-major
            const uint32_t dst = sb + q * (sym ? BM * BK * 2 : 64 * BK * 2);
            const int x = sym ? kb * BK : n0 + q * 64;
            const int y = sym ? c.mat * P.p.N + n0 + q * BM : c.mat * P.p.K + kb * BK;
            if (PAIR && !leader)
              tma_load_2d_pair(dst, &P.tmQ, x, y, mapa_shared(fb, 0));
            else
              tma_load_2d(dst, &P.tmQ, x, y, fb);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: wait for the copies of the most recent ring lap to land. With
      // PAIR the leader's full barriers count both CTAs' copies; the odd CTA's
      // own copies are also covered by the leader's MMA drain (they are read
      // by its MMAs) and by the closing cluster barrier.
      const int pending = issues_mma ? (issued < STAGES ? issued : STAGES) : 0;
      int s = stage;
      uint32_t ph = phase;
      for (int i = 0; i < pending; ++i) {
        if (--s < 0) {
          s = STAGES - 1;
          ph ^= 1u;
        }
        // full[s] completes phase `ph` when those copies land; a dedicated
        // bound keeps this loop finite even when the CTA is aborting.
        const uint64_t t0 = global_timer();
        while (!mbar_try_wait(full0 + 8 * s, ph)) {
          if (global_timer() - t0 > kWaitLimitNs) {
            atomicCAS(L.err, 0, kErrWaitProducer);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && issues_mma) {
      // ---------------- MMA issuer (PAIR: the leader only) ----------------
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      // Descriptors of stage 0's operands; a stage is STAGE bytes further
      // (the address field counts 16-byte units, so stage and K16 steps are
      // plain additions). K-major: the K16 step is 32 bytes. MN-major
      // right-hand operand: 64-element panels 8 KB apart (LBO), 8-row groups
      // 1 KB apart (SBO), the K16 step is 16 rows of 128 bytes.
      const uint32_t s0 = smem_u32(smem);
      const uint64_t a_desc0 = sdesc(s0, 16, 1024);
      const uint64_t bk_desc0 = sdesc(s0 + A_STAGE, 16, 1024);
      const uint64_t bmn_desc0 = sdesc(s0 + A_STAGE, 64u * BK * 2u, 1024u);
      int g_next = unit0 < L.npos ? unit_at(L, unit0) : -1;
      for (int pos = unit0; pos < L.npos && ok; pos += nunits) {
        const int g = g_next;  // read one unit ahead, off this unit's critical path
        g_next = pos + nunits < L.npos ? unit_at(L, pos + nunits) : -1;
        if (g < 0) continue;
        const TileCoord c = decode_tile(L, g);
        const TcProblem& P = L.prob[c.prob];
        const int kblocks = P.p.K / BK;
        const bool sym = P.p.kind != NS_UPDATE;
        const uint32_t idesc = idesc_bf16(G * BM, P.bn, !sym);
        // the right-hand operand: the stage's right tile, or its left tile when the rows coincide
        const uint64_t b_desc0 = rhs_is_lhs(P, c, CL, crank) ? a_desc0 : sym ? bk_desc0 : bmn_desc0;
        const uint32_t b_kstep = sym ? 2u : 128u;
        // the epilogues (PAIR: of both CTAs) have released this accumulator
        if (!mbar_wait<PAIR>(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag, L.err, kErrWaitMma)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN_MAX);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, L.err, kErrWaitMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t soff = (uint32_t)stage * (uint32_t)(SM::STAGE >> 4);
          const uint64_t ad = a_desc0 + soff;
          const uint64_t bd = b_desc0 + soff;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16<G>(d_tmem, ad + 2u * kk, bd + b_kstep * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          if (PAIR)
            umma_commit_pair(empty0 + 8 * stage);  // both CTAs' parts of this stage are free
          else
            umma_commit<1>(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR)
          umma_commit_pair(tfull0 + 8 * acc);
        else
          umma_commit<1>(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit<G>(drain);
      const uint64_t t0 = global_timer();
      while (!mbar_try_wait(drain, 0)) {
        if (global_timer() - t0 > kWaitLimitNs) {
          atomicCAS(L.err, 0, kErrWaitMma);
          break;
        }
      }
    }
  } else if (APPLY) {
    // ---------------- epilogue of the last iteration ----------------
    apply_epilogue<CL, PAIR, SHADOW>(L, smem, SM::PBUF, SM::SB, smem_u32(bars + 2 * STAGES + 5), tmem_base, tfull0, tempty0,
                       abort_flag, warp, lane, crank, unit0, nunits);
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. 32*quarter+31
    const int half = (warp - 2) >> 2;  // which alternate 32-column blocks
    uint8_t* const rt = smem + SM::SB + (size_t)(warp - 2) * SM::SB_PER_WARP;
    int acc = 0;
    uint32_t acc_phase = 0;
    int g_next = unit0 < L.npos ? unit_at(L, unit0) : -1;
    for (int pos = unit0; pos < L.npos; pos += nunits) {
      const int g = g_next;  // read one unit ahead, off this unit's critical path
      g_next = pos + nunits < L.npos ? unit_at(L, pos + nunits) : -1;
      if (g < 0) continue;
      const TileCoord c = decode_tile(L, g);
      const TcProblem& P = L.prob[c.prob];
      // every lane waits; the vote keeps the warp converged for tcgen05.ld
      const bool got = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, L.err, kErrWaitEpilogue);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN_MAX);
      const int row0 = (c.ti * CL + (int)crank) * BM + quarter * 32;
      for (int c0 = 32 * half; c0 < P.bn; c0 += 64)
        epilogue_block(P.p, &P.tmO, L.epi, c.mat, row0, c.tj * P.bn + c0, tbase + (uint32_t)c0, rt, lane);
      release_accumulator<PAIR>(tempty0 + 8 * acc, lane);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_read_all();  // the stores have read shared memory before the CTA may leave
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA of a pair leaves while the other may still read its shared
  // memory or TMEM, or arrive on its barriers.
  if (CL == 2) cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<G>(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Newton-Schulz of small matrices (canonical s <= 128 rows, padded to S = 128,
// l <= 512 columns) in one launch: one CTA takes a whole matrix through every
// iteration and the parameter update. X (128 x L bf16), A and B (128 x 128
// bf16) stay in shared memory as 128-row panels of 64 columns in the 128-byte
// swizzle layout, which serves as the K-major operand of X X^T and A A (both
// operands: the rows coincide) and of B in B X, and as the MN-major right-hand
// operand of B X (panels 16 KiB apart). Products accumulate in TMEM: A at
// columns 0..127, A A at 128..255, X' = B X over columns 0..L-1 once those are
// read. The CTA's 8 warps all run the epilogues (two warps per TMEM lane
// quarter), which round to bf16 into the panels; the last one updates the
// parameters from registers. Thread 0 also issues the copies and the MMAs:
// the phases follow each other, every thread waiting at each product's
// barrier, so no warp is set aside for issuing and a thread may hold up to
// 255 registers. The next matrix's X is loaded by TMA as soon as the last
// B X has read X.
// ---------------------------------------------------------------------------
constexpr int SMALL_EPI_WARPS = 8;
constexpr int SMALL_THREADS = 32 * SMALL_EPI_WARPS;
constexpr int SMALL_PANEL = 128 * 64 * 2;  // 16 KiB

struct SmallSmem {
  static constexpr size_t X = 0;
  static constexpr size_t A = X + (size_t)(kSmallMaxL / 64) * SMALL_PANEL;
  static constexpr size_t B = A + 2 * (size_t)SMALL_PANEL;
  static constexpr size_t BARS = B + 2 * (size_t)SMALL_PANEL;
  static constexpr size_t BYTES = 1024 + BARS + 64;
  static_assert(BYTES <= 232448, "shared memory per CTA");
  static_assert((BYTES >> 4) < 0x4000, "operand descriptors: 14-bit address field");
};

// Bring `bytes` (a multiple of 16, 16-byte aligned start) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// bf16 pairs of 32 consecutive columns c0.. (c0 % 32 == 0) into row r of the
// panel layout: chunk q of the row sits at q ^ (r & 7).
__device__ __forceinline__ void small_put_row(uint8_t* panels, int r, int c0, const uint32_t (&pk)[16]) {
  uint8_t* const row = panels + (size_t)(c0 >> 6) * SMALL_PANEL + (size_t)r * 128;
  const int q0 = (c0 & 63) >> 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(row + (((q0 + j) ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

__device__ __forceinline__ void small_get_row(const uint8_t* panels, int r, int c0, uint4 (&v)[4]) {
  const uint8_t* const row = panels + (size_t)(c0 >> 6) * SMALL_PANEL + (size_t)r * 128;
  const int q0 = (c0 & 63) >> 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4*>(row + (((q0 + j) ^ (r & 7)) << 4));
}

// Last-iteration update of a small matrix's parameter in 32 x 32 blocks, with
// the lanes along parameter rows (coalesced). Wide parameters (canonical row =
// parameter row) pass a block through the warp's padded fp32 tile `t` to get
// there; for tall ones (canonical row = parameter column) lane l already holds
// parameter column row0 + l. A lane's part of a block: `nr` parameter rows
// from offset `base` (one element per row, a row apart).
struct SmallBlk {
  int base, nr;
};

__device__ __forceinline__ SmallBlk small_block_at(int n, int s, int l, bool tr, int row0, int col0, int lane) {
  SmallBlk b;
  if (!tr) {
    const int gc = col0 + lane;
    b.base = row0 * n + gc;
    b.nr = gc < l ? s - row0 : 0;
  } else {
    const int gc = row0 + lane;
    b.base = col0 * n + gc;
    b.nr = gc < s ? l - col0 : 0;
  }
  if (b.nr > 32) b.nr = 32;
  return b;
}

__device__ __forceinline__ void small_load_block(const float* P, int n, SmallBlk b, float (&pv)[32]) {
#pragma unroll
  for (int r = 0; r < 32; ++r) pv[r] = r < b.nr ? P[b.base + r * n] : 0.f;
}

// The block's update direction for this lane's parameter column, from TMEM.
__device__ __forceinline__ void small_block_dir(uint32_t taddr, float rs, bool tr, float (*t)[33], int lane,
                                                float (&o)[32]) {
  uint32_t v[32];
  tmem_ld_32x32b_x32(taddr, v);
  tmem_ld_wait();
  if (!tr) {
#pragma unroll
    for (int e = 0; e < 32; ++e) t[lane][e] = __uint_as_float(v[e]) * rs;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) o[r] = t[r][lane];
    __syncwarp();
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(v[e]) * rs;
  }
}

__device__ __forceinline__ void small_store_block(float* P, uint16_t* SH, int n, SmallBlk b, float dec, float lrm,
                                                  const float (&pv)[32], const float (&o)[32]) {
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    if (r < b.nr) {
      const float q = fmaf(pv[r], dec, -lrm * o[r]);
      P[b.base + r * n] = q;
      if (SH) SH[b.base + r * n] = ns_f2bf(q);
    }
  }
}

// L1 prefetch of a 32 x 32 parameter block of a small matrix (the layout of
// small_block_at): lane r takes the 128 bytes of the block's r-th
// parameter row, so the block's loads find it close when they come.
__device__ __forceinline__ void small_prefetch_block(const MuonMat& M, int row0, int col0, int lane) {
  const bool tr = M.transposed != 0;
  const int pr = tr ? col0 + lane : row0 + lane;  // parameter row of this lane
  const int pc = tr ? row0 : col0;                // first parameter column of the block
  if (pr < M.m && pc < M.n)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(M.p + (size_t)pr * M.n + pc) : "memory");
}

// Every thread waits for phase `parity` of `bar`; false on the CTA when any
// thread's bounded wait ran out (the error is recorded), so all leave together.
__device__ __forceinline__ bool small_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  const bool ok = mbar_wait(bar, parity, abort_flag, err, kErrWaitEpilogue);
  return __syncthreads_and(ok) != 0;
}

__global__ void __launch_bounds__(SMALL_THREADS, 1) ns_small_kernel(const __grid_constant__ SmallLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* const Xp = smem + SmallSmem::X;
  uint8_t* const Ap = smem + SmallSmem::A;
  uint8_t* const Bp = smem + SmallSmem::B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SmallSmem::BARS);
  const uint32_t load_bar = smem_u32(bars), mma_bar = smem_u32(bars + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int npan = L.L / 64;

  if (threadIdx.x == 0) {
    mbar_init(load_bar, 1);
    mbar_init(mma_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&L.tmX)) : "memory");
  }
  if (warp == 0) tmem_alloc<1>(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t xs = smem_u32(Xp), as = smem_u32(Ap), bs = smem_u32(Bp);
  auto load_x = [&](int mat) {  // thread 0
    mbar_expect_tx(load_bar, (uint32_t)(npan * SMALL_PANEL));
    for (int q = 0; q < npan; ++q) tma_load_2d(xs + q * SMALL_PANEL, &L.tmX, 64 * q, mat * 128, load_bar);
  };
  // epilogue geometry: TMEM lane quarter (rows) and alternate 32-column blocks
  const int quarter = warp & 3;
  const int half = warp >> 2;
  const int row = 32 * quarter + lane;  // this lane's canonical row
  const uint32_t tq = tmem + ((uint32_t)(32 * quarter) << 16);

  uint32_t load_ph = 0, mma_ph = 0;
  bool ok = true;
  bool pending = false;  // thread 0: an X load is in flight
  bool mma_out = false;  // thread 0: MMAs committed and not yet waited for
  // test hook: CTA 0 loads nothing, so its first bounded wait runs out
  if (threadIdx.x == 0 && (int)blockIdx.x < L.nmat && !(L.stall_test && blockIdx.x == 0)) {
    load_x(blockIdx.x);
    pending = true;
  }
  for (int mat = blockIdx.x; mat < L.nmat && ok; mat += gridDim.x) {
    const MuonMat& M = L.mats[mat];
    const int s = M.s, l = M.l;
    const float r = L.rscale[mat];
    if (!(ok = small_wait(load_bar, load_ph, abort_flag, L.err))) break;
    load_ph ^= 1u;
    pending = false;
    if (threadIdx.x == 0) {
      // the parameters the update reads at the end, into L2 while the iterations run
      const size_t pbytes = (size_t)M.m * M.n * 4;
      if ((reinterpret_cast<uintptr_t>(M.p) & 15) == 0)
        for (size_t o = 0; o + 16 <= pbytes; o += (size_t)1 << 20) {
          const size_t n = pbytes - o < ((size_t)1 << 20) ? pbytes - o : ((size_t)1 << 20);
          bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(M.p) + o, (uint32_t)(n & ~(size_t)15));
        }
    }
    for (int it = 0; it < L.steps && ok; ++it) {
      const bool first = it == 0, last = it == L.steps - 1;
      const float ca = L.coef[it][0], cb = L.coef[it][1], cc = L.coef[it][2];
      // ---- A = X X^T (columns 0..127) ----
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 128, false);
        for (int q = 0; q < npan; ++q) {
          const uint64_t d0 = sdesc(xs + q * SMALL_PANEL, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) umma_bf16<1>(tmem, d0 + 2u * kk, d0 + 2u * kk, id, (q | kk) != 0 ? 1u : 0u);
        }
        umma_commit<1>(mma_bar);
        mma_out = true;
      }
      if (!(ok = small_wait(mma_bar, mma_ph, abort_flag, L.err))) break;
      mma_ph ^= 1u;
      mma_out = false;
      tc_fence_after();
      {
        const float sc = first ? r * r : 1.f;
        for (int c0 = 32 * half; c0 < 128; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tq + (uint32_t)c0, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float x0 = __uint_as_float(v[2 * j]) * sc, x1 = __uint_as_float(v[2 * j + 1]) * sc;
            if (row >= s || c0 + 2 * j >= s) x0 = 0.f;
            if (row >= s || c0 + 2 * j + 1 >= s) x1 = 0.f;
            pk[j] = pack_bf16x2(x0, x1);
          }
          small_put_row(Ap, row, c0, pk);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      // ---- A A (columns 128..255); B = c A A + b A + a I ----
      if (threadIdx.x == 0) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 128, false);
        for (int q = 0; q < 2; ++q) {
          const uint64_t d0 = sdesc(as + q * SMALL_PANEL, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16<1>(tmem + 128u, d0 + 2u * kk, d0 + 2u * kk, id, (q | kk) != 0 ? 1u : 0u);
        }
        umma_commit<1>(mma_bar);
        mma_out = true;
      }
      if (!(ok = small_wait(mma_bar, mma_ph, abort_flag, L.err))) break;
      mma_ph ^= 1u;
      mma_out = false;
      tc_fence_after();
      {
        for (int c0 = 32 * half; c0 < 128; c0 += 64) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tq + 128u + (uint32_t)c0, v);
          uint4 a4[4];
          small_get_row(Ap, row, c0, a4);
          tmem_ld_wait();
          const bool on_diag = c0 == 32 * quarter;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t u = u4_get(a4[j >> 2], j & 3);
            float o[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int col = 2 * j + e;
              const float av = __uint_as_float(e ? (u & 0xFFFF0000u) : (u << 16));
              const float lin = on_diag ? fmaf(cb, av, col == lane ? ca : 0.f) : cb * av;
              o[e] = fmaf(cc, __uint_as_float(v[col]), lin);
              if (row >= s || c0 + col >= s) o[e] = 0.f;
            }
            pk[j] = pack_bf16x2(o[0], o[1]);
          }
          small_put_row(Bp, row, c0, pk);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      // the last iteration's update starts with this warp's first parameter block
      if (last) {
        small_prefetch_block(M, 32 * quarter, 32 * half, lane);
        small_prefetch_block(M, 32 * quarter, 32 * half + 64, lane);
      }
      // ---- X' = B X (columns 0..L-1) ----
      if (threadIdx.x == 0) {
        tc_fence_after();
        for (int n0 = 0; n0 < L.L; n0 += 256) {
          const int nn = L.L - n0 < 256 ? L.L - n0 : 256;
          const uint32_t id = idesc_bf16(128, nn, true);
          const uint64_t b0 = sdesc(xs + (n0 / 64) * SMALL_PANEL, SMALL_PANEL, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t a = sdesc(bs + (ks >> 2) * SMALL_PANEL, 16, 1024) + 2u * (ks & 3);
            umma_bf16<1>(tmem + (uint32_t)n0, a, b0 + 128u * ks, id, ks != 0 ? 1u : 0u);
          }
        }
        umma_commit<1>(mma_bar);
        mma_out = true;
      }
      if (!(ok = small_wait(mma_bar, mma_ph, abort_flag, L.err))) break;
      mma_ph ^= 1u;
      mma_out = false;
      tc_fence_after();
      if (!last) {
        {
          const float sc = first ? r : 1.f;
          // two blocks per TMEM wait (L is a multiple of 128: blocks c0 and c0 + 64 both exist)
          for (int c0 = 32 * half; c0 < L.L; c0 += 128) {
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(tq + (uint32_t)c0, v[0]);
            tmem_ld_32x32b_x32(tq + (uint32_t)(c0 + 64), v[1]);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int cb0 = c0 + 64 * h;
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float x0 = __uint_as_float(v[h][2 * j]) * sc, x1 = __uint_as_float(v[h][2 * j + 1]) * sc;
                if (row >= s || cb0 + 2 * j >= l) x0 = 0.f;
                if (row >= s || cb0 + 2 * j + 1 >= l) x1 = 0.f;
                pk[j] = pack_bf16x2(x0, x1);
              }
              small_put_row(Xp, row, cb0, pk);
            }
          }
        }
        fence_proxy_async_smem();
      } else {
        // X has been read for the last time: the next matrix's comes in meanwhile
        if (threadIdx.x == 0 && mat + (int)gridDim.x < L.nmat) {
          load_x(mat + gridDim.x);
          pending = true;
        }
        {
          // A and B are free now: a padded 32 x 33 fp32 tile per epilogue warp
          float(*t)[33] = reinterpret_cast<float(*)[33]>(Ap + (size_t)warp * 32 * 33 * 4);
          const float rs = first ? r : 1.f;
          const float lrm = L.sp->ns_lr * M.lr_mult;
          const float dec = L.sp->ns_decay[M.group];
          // the matrix's fields in registers: the stores below go through
          // generic pointers that could otherwise alias the descriptor
          float* const P = M.p;
          uint16_t* const SH = M.shadow;
          const int n = M.n, row0 = 32 * quarter;
          const bool tr = M.transposed != 0;
          // each block's loads are issued before the previous block's stores
          int c0 = 32 * half;
          SmallBlk b = small_block_at(n, s, l, tr, row0, c0, lane);
          float pv[32];
          small_load_block(P, n, b, pv);
          for (; c0 < l; c0 += 64) {
            if (c0 + 128 < l) small_prefetch_block(M, row0, c0 + 128, lane);
            const SmallBlk bn = c0 + 64 < l ? small_block_at(n, s, l, tr, row0, c0 + 64, lane) : SmallBlk{0, 0};
            float pn[32];
            small_load_block(P, n, bn, pn);
            float o[32];
            small_block_dir(tq + (uint32_t)c0, rs, tr, t, lane, o);
            small_store_block(P, SH, n, b, dec, lrm, pv, o);
#pragma unroll
            for (int r = 0; r < 32; ++r) pv[r] = pn[r];
            b = bn;
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
  }
  // A load issued for a matrix this CTA no longer reaches (after an abort)
  // lands before the CTA leaves; the MMAs have all been waited for.
  if (!ok && pending) {
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(load_bar, load_ph) && global_timer() - t0 < kWaitLimitNs) {
    }
  }
  // ... and MMAs still running finish before TMEM is released
  if (!ok && mma_out) {
    const uint64_t t0 = global_timer();
    while (!mbar_try_wait(mma_bar, mma_ph) && global_timer() - t0 < kWaitLimitNs) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(tmem, 512);
}

// ---- host side ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// cuTensorMapEncodeTiled of a row-major 2-D tensor.
CUresult encode_rowmajor(CUtensorMap* tm, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t cols,
                         uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool encode_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
               char* errbuf, size_t errlen) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled entry point not available");
    return false;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled failed (%d) for %llux%llu box %ux%u", (int)r,
             (unsigned long long)rows, (unsigned long long)cols, box_rows, box_cols);
    return false;
  }
  return true;
}

}  // namespace

int ns_tc_num_tiles_sym(int units_m, int bmu, int bn) {
  int n = 0;
  for (int ti = 0; ti < units_m; ++ti) n += (ti * bmu + bmu - 1) / bn + 1;
  return n;
}

bool ns_tc_pairable(const NsProblem& p) { return p.M % (2 * BM) == 0; }

bool tc_encode_problem(TcProblem& tp, int cl, char* errbuf, size_t errlen) {
  const NsProblem& p = tp.p;
  if (p.M % BM || p.K % BK || p.N % 128) {
    snprintf(errbuf, errlen, "tcgen05 GEMM needs M%%128 == 0, K%%64 == 0, N%%128 == 0 (M=%d N=%d K=%d)", p.M, p.N,
             p.K);
    return false;
  }
  if (cl == 2 && !ns_tc_pairable(p)) {
    snprintf(errbuf, errlen, "paired launch needs M %% 256 == 0 (M=%d)", p.M);
    return false;
  }
  tp.bn = (p.N % 256 == 0) ? 256 : 128;
  tp.tiles_m = p.M / BM;
  tp.tiles_n = p.N / tp.bn;
  const int units_m = tp.tiles_m / cl;
  tp.tiles_per_mat =
      p.kind == NS_UPDATE ? units_m * tp.tiles_n : ns_tc_num_tiles_sym(units_m, BM * cl, tp.bn);
  const uint64_t nm = (uint64_t)p.nmat;
  // Output: [nmat * S] rows x (UPDATE: L, else S) cols, 32 x 32 bf16 blocks, 64-byte swizzle.
  if (encode_rowmajor(&tp.tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, (uint64_t)(p.kind == NS_UPDATE ? p.L : p.S),
                      nm * p.S, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS) {
    snprintf(errbuf, errlen, "cuTensorMapEncodeTiled failed for the output of a %dx%d bucket", p.S, p.L);
    return false;
  }
  // Left operand: [nmat * M] rows x K cols, K-major tiles of 128 x 64.
  if (!encode_2d(&tp.tmP, p.P, (uint64_t)p.K, nm * p.M, BK, BM, errbuf, errlen)) return false;
  if (p.kind == NS_UPDATE) {
    // Right operand X: [nmat * K] rows x N cols, MN-major tiles of 64 (K) x 64 (N).
    if (!encode_2d(&tp.tmQ, p.Q, (uint64_t)p.N, nm * p.K, 64, BK, errbuf, errlen)) return false;
  } else {
    // Right operand = rows of the same matrix: [nmat * N] rows x K cols.
    if (!encode_2d(&tp.tmQ, p.Q, (uint64_t)p.K, nm * p.N, BK, BM, errbuf, errlen)) return false;
  }
  return true;
}

void tc_unit_order(const TcLaunch& L, int ncl, std::vector<int32_t>& order) {
  std::vector<std::vector<int32_t>> lists((size_t)ncl);
  using Entry = std::pair<double, int>;  // (work so far, cluster)
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> least;
  for (int c = 0; c < ncl; ++c) least.push({0.0, c});
  for (int q = 0; q < L.nprob; ++q) {
    const TcProblem& P = L.prob[q];
    const double cost = (double)(P.p.K / BK) + 6.0;
    const int n = P.tiles_per_mat * P.p.nmat;
    for (int u = 0; u < n; ++u) {
      const Entry e = least.top();
      least.pop();
      lists[(size_t)e.second].push_back(P.tile_begin + u);
      least.push({e.first + cost, e.second});
    }
  }
  size_t rounds = 0;
  for (const auto& l : lists) rounds = l.size() > rounds ? l.size() : rounds;
  order.assign(rounds * (size_t)ncl, -1);
  for (int c = 0; c < ncl; ++c)
    for (size_t r = 0; r < lists[(size_t)c].size(); ++r) order[r * (size_t)ncl + (size_t)c] = lists[(size_t)c][r];
}

bool tc_encode_param_maps(CUtensorMap* maps, const MuonMat& M) {
  memset(maps, 0, 2 * sizeof(CUtensorMap));
  const bool shadow = M.shadow != nullptr;
  // row strides and base addresses on 16-byte boundaries; at least one full box per dimension
  if (M.m < 32 || M.n < 32 || M.n % (shadow ? 8 : 4) != 0) return false;
  if (reinterpret_cast<uintptr_t>(M.p) % 16 != 0 || (shadow && reinterpret_cast<uintptr_t>(M.shadow) % 16 != 0))
    return false;
  if (encode_rowmajor(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, M.p, (uint64_t)M.n, (uint64_t)M.m, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return false;
  if (shadow && encode_rowmajor(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M.shadow, (uint64_t)M.n,
                                (uint64_t)M.m, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
    return false;
  return true;
}

namespace {
template <int CL, bool APPLY, bool PAIR, bool SHADOW = true>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(ns_tc_kernel<CL, APPLY, PAIR, SHADOW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)Smem<PAIR, APPLY, SHADOW>::BYTES);
}

template <bool APPLY, bool PAIR, bool SHADOW = true>
cudaError_t max_pairs_of(int* n) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Smem<PAIR, APPLY, SHADOW>::BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, ns_tc_kernel<2, APPLY, PAIR, SHADOW>, &cfg);
}

template <bool APPLY, bool PAIR, bool SHADOW = true>
cudaError_t launch_pair(const TcLaunch& L, int grid_units, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * grid_units, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Smem<PAIR, APPLY, SHADOW>::BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ns_tc_kernel<2, APPLY, PAIR, SHADOW>, L);
}
}  // namespace

cudaError_t ns_tc_prepare(int* max_pairs) {
  cudaError_t e;
  if ((e = set_smem_attr<1, false, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<1, true, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<2, false, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<2, true, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<2, true, true, false>()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)SmallSmem::BYTES)) != cudaSuccess)
    return e;
  int a = 0, c = 0, d = 0;
  if ((e = max_pairs_of<false, true>(&a)) != cudaSuccess) return e;
  if ((e = max_pairs_of<true, true>(&c)) != cudaSuccess) return e;
  if ((e = max_pairs_of<true, true, false>(&d)) != cudaSuccess) return e;
  const int m = a < c ? a : c;
  *max_pairs = m < d ? m : d;
  return cudaSuccess;
}

bool tc_encode_small(SmallLaunch& sl, const uint16_t* X, int nmat, int L, char* errbuf, size_t errlen) {
  // X of every matrix of the bucket: [nmat * 128] rows x L cols, panels of 128 x 64
  return encode_2d(&sl.tmX, X, (uint64_t)L, (uint64_t)nmat * 128u, 64, 128, errbuf, errlen);
}

cudaError_t launch_ns_small(const SmallLaunch& L, int num_sms, cudaStream_t st) {
  const int grid = L.nmat < num_sms ? L.nmat : num_sms;
  if (grid <= 0) return cudaSuccess;
  ns_small_kernel<<<grid, SMALL_THREADS, SmallSmem::BYTES, st>>>(L);
  return cudaGetLastError();
}

cudaError_t launch_ns_tc(const TcLaunch& L, cudaStream_t st) {
  // the work order was laid out for exactly this many clusters
  const int grid_units = L.nclusters;
  if (grid_units <= 0) return cudaSuccess;
  // every problem of a launch is the same product of the same iteration
  const bool update = L.prob[0].p.kind == NS_UPDATE;
  const bool apply = update && L.prob[0].p.last;
  if (L.cl == 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid_units, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = apply ? Smem<false, true>::BYTES : Smem<false, false>::BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return apply ? cudaLaunchKernelEx(&cfg, ns_tc_kernel<1, true, false>, L)
                 : cudaLaunchKernelEx(&cfg, ns_tc_kernel<1, false, false>, L);
  }
  if (apply) return L.shadow ? launch_pair<true, true>(L, grid_units, st) : launch_pair<true, true, false>(L, grid_units, st);
  return launch_pair<false, true>(L, grid_units, st);
}

}  // namespace ma
