// Internal types shared by the host runtime (capi.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace ma {

// Elements per multi-tensor chunk of the gradient-norm and AdamW streams.
constexpr int64_t kChunk = 1 << 16;
// Tiles of 4096 elements the Muon momentum kernel walks: 64 x 64 for tall
// matrices (their X is written transposed through a shared tile), 16 rows x
// 256 columns for the others (longer contiguous row segments); and the
// partial sums of squares it writes per tile (one per warp).
constexpr int kMomTile = 64;
constexpr int kMomWideRows = 16;
constexpr int kMomWideCols = 256;
constexpr int kMomPartialsPerTile = 8;
// Padding granule of the canonical Newton-Schulz workspaces (rows and cols).
constexpr int kPad = 128;
// Muon matrices whose short side is below this run Newton-Schulz in fp32 on
// the CUDA cores (ns_narrow.cu) instead of through the bf16 tensor-core path.
constexpr int kNarrowMinS = 64;

enum GradDtype : int32_t { DT_F32 = 0, DT_BF16 = 1 };

struct GradChunk {      // one slice of one gradient
  const void* g;
  int64_t n;
  int32_t dtype;
  int32_t vec;          // 1 if g is 16-byte aligned (vector loads allowed)
};

struct AdamChunk {      // one slice of one AdamW parameter
  float* p;
  const void* g;
  float* m;
  float* v;
  uint16_t* shadow;     // bf16 copy or nullptr
  int64_t n;
  int32_t gdtype;
  int32_t vec;          // 1 if every pointer allows 4-wide vector access
  int32_t group;        // option group: index into AdamArgs' per-group decay and step size
  int32_t pad;
};

struct MuonMat {        // one Muon matrix (device-visible metadata)
  float* p;             // fp32 master [m][n]
  const void* g;        // gradient [m][n]
  float* buf;           // momentum [m][n]
  uint16_t* shadow;     // bf16 [m][n] or nullptr
  uint16_t* x0;         // canonical bf16 X of this matrix, [S][L], row stride L
  int32_t m, n;         // parameter shape
  int32_t s, l;         // canonical shape: s = min(m,n), l = max(m,n)
  int32_t S, L;         // padded canonical shape (multiples of kPad)
  int32_t transposed;   // 1 if m > n (X = update^T)
  int32_t gdtype;
  int32_t vec;          // rows of g/buf allow 16-byte vector access
  int32_t pvec;         // rows of p (and shadow) allow 8-element vector access
  int32_t tile_begin;   // momentum tiles [tile_begin, tile_end) in the tile list
  int32_t tile_end;
  float lr_mult;        // muon_lr_scale * moonlight * sqrt(max(m, n))
  int32_t tma;          // 1 if p (and shadow) have TMA maps: the last iteration moves them by TMA
  int32_t group;        // option group: index into NsEpiArgs::decay
  float* xf;            // narrow matrices (s < kNarrowMinS): fp32 X in the parameter's layout; else nullptr
};

struct MomTile {
  int32_t mat;
  int32_t r0, c0;       // tile origin in the parameter (row, col)
  int32_t pad;
};

struct StepScalars {    // written on the device each step
  float total;          // global gradient norm
  float coef;           // clip coefficient
  float pad0, pad1;
};

// Distinct (lr_scale, weight_decay_scale) pairs of the parameters, group 0
// being (1, 1); each chunk or matrix names its group.
constexpr int kMaxOptionGroups = 8;

// Scalars that change every step (they depend on lr and the step count t):
// one host-to-device copy writes them to HBM at the start of each step and
// the kernels that need them read them there, so that a captured step graph
// stays valid from step to step.
struct StepParams {
  float adam_decay[kMaxOptionGroups];  // 1 - lr * lr_scale * wd * wd_scale
  float adam_step[kMaxOptionGroups];   // lr * lr_scale / (1 - beta1^t)
  float adam_inv_sqrt_bc2;             // 1 / sqrt(1 - beta2^t)
  float ns_lr;                         // lr
  float ns_decay[kMaxOptionGroups];    // 1 - lr * lr_scale * muon_wd * wd_scale
  float pad[2];
};

struct AdamArgs {
  float beta1, beta2, omb1, omb2, eps;
  const StepParams* sp;
};

struct MomArgs {
  float mu;
  int32_t nesterov;
  float gscale;         // weight of the clipped gradient: 1, or 1 - mu for the exponential-average form
};

enum NsKind : int32_t { NS_GRAM = 0, NS_POLY = 1, NS_UPDATE = 2 };

struct NsEpiArgs {
  float a, b, c;         // this iteration's coefficients
  const StepParams* sp;  // the last iteration's lr and decays
};

// One grouped GEMM problem: all same-shape matrices of one bucket. The
// quintic step X <- a X + (b A + c A A) X is evaluated as
//   GRAM:   A = X X^T                     (P = Q = X, K = L)         symmetric
//   POLY:   B = a I + b A + c A A         (P = Q = A, K = S)         symmetric
//   UPDATE: X' = B X                      (P = B, Q = X MN-major, K = S)
// so that the largest product's epilogue reads nothing back; only POLY
// reads A for its b A term. Iteration 1 scales A by r^2 and X' by r, with
// r = 1 / (||update||_F + eps).
struct NsProblem {
  const uint16_t* P;
  const uint16_t* Q;
  const uint16_t* aux;  // POLY: A; otherwise unused
  uint16_t* out;        // GRAM: A; POLY: B; UPDATE: X'
  const MuonMat* mats;  // this bucket's matrices
  const float* rscale;  // per matrix 1 / (||update||_F + eps), same indexing
  const CUtensorMap* pmaps;  // per matrix [2]: p (fp32) and shadow (bf16) maps, same indexing
  int32_t kind;
  int32_t S, L;
  int32_t M, N, K;
  int32_t nmat;
  int32_t first, last;  // first / last Newton-Schulz iteration
  int32_t shadow;       // some matrix of the bucket has a bf16 shadow
};

// ---- the thread-local message behind muon_adamw_last_error() (capi.cu) ----
void set_last_error(const char* msg);
void clear_last_error();

// ---- launchers (stream_kernels.cu) ----
void launch_grad_sumsq(const GradChunk* chunks, int nchunks, float* partials, int grid, cudaStream_t st);
void launch_clip_finalize(const float* partials, int n, float max_norm, float clip_eps, StepScalars* out,
                          cudaStream_t st);
// The sum of the norm pass's partials, in fp64, to *out (one block): this
// rank's share of the global sum of squares in a sharded step.
void launch_sumsq_partials(const float* partials, int n, double* out, cudaStream_t st);
// Norm and clip coefficient from a global sum of squares (one thread), with
// the same rules as clip_finalize.
void launch_clip_from_sumsq(const double* sumsq, float max_norm, float clip_eps, StepScalars* out, cudaStream_t st);
void launch_muon_momentum(const MomTile* tiles, int ntiles, const MuonMat* mats, const StepScalars* sc,
                          MomArgs args, float* tile_partials, int grid, cudaStream_t st);
void launch_ns_prep(const MuonMat* mats, int nmat, const float* tile_partials, float eps, float* rscale,
                    cudaStream_t st);
void launch_adamw(const AdamChunk* chunks, int nchunks, const StepScalars* sc, AdamArgs args, int grid,
                  cudaStream_t st);

// ---- Newton-Schulz GEMMs ----
// CUDA-core cross-check kernel (ns_simt.cu)
void launch_ns_simt(const NsProblem& prob, NsEpiArgs epi, cudaStream_t st);

// tcgen05 / TMEM / TMA kernel (ns_tc.cu)
constexpr int kTcMaxProblems = 4;
struct TcProblem {
  CUtensorMap tmP;      // K-major loads of P, box {64, 128}
  CUtensorMap tmQ;      // GRAM/POLY: K-major box {64, 128}; UPDATE: MN-major box {64, 64}
  CUtensorMap tmO;      // stores of the output, box {32, 32}
  NsProblem p;
  int32_t bn;           // N tile: 128 or 256
  int32_t tiles_m;      // M / 128
  int32_t tiles_n;      // N / bn
  int32_t tiles_per_mat;  // work units per matrix (a unit = cl row blocks x one column block)
  int32_t tile_begin;   // first global work unit of this problem
  int32_t pad[3];
};
struct TcLaunch {
  TcProblem prob[kTcMaxProblems];
  int32_t nprob;
  int32_t total_tiles;  // work units in the launch
  NsEpiArgs epi;
  int* err;             // device error flag
  // Work assignment: cluster c takes the units order[c], order[c + nclusters],
  // ... (npos entries, -1 = nothing), from tc_unit_order; no table (nullptr)
  // when that is the plain round-robin order (position = unit).
  const int32_t* order;
  int32_t npos;
  int32_t nclusters;    // clusters in the grid
  int32_t cl;           // CTAs per cluster: 1, or 2 (a CTA pair running cta_group::2 MMAs)
  int32_t stall_test;   // test hook: CTA 0's producer issues no loads (its waits then run out)
  int32_t shadow;       // some matrix of the launch writes a bf16 shadow (the last iteration keeps shadow tiles)
};
// TMA maps of one parameter for the last iteration's write-back: maps[0] the
// fp32 master, maps[1] the bf16 shadow (unused without one); 32 x 32 boxes.
// False (and M.tma stays 0) when the layout does not allow TMA.
bool tc_encode_param_maps(CUtensorMap* maps, const MuonMat& M);
// Whether a problem can run in CTA pairs (its row blocks pair up).
bool ns_tc_pairable(const NsProblem& p);
// Encode the tensor maps of `tp` and count its work units for cluster size cl (host).
bool tc_encode_problem(TcProblem& tp, int cl, char* errbuf, size_t errlen);
// Newton-Schulz of a bucket of small matrices (S = 128, L <= kSmallMaxL) in
// one launch, a CTA per matrix (ns_tc.cu): every iteration and the update.
constexpr int kSmallMaxL = 512;
struct SmallLaunch {
  CUtensorMap tmX;           // X of the bucket: [nmat * 128] rows x L cols, boxes of 64 x 128
  const MuonMat* mats;       // the bucket's matrices
  const float* rscale;       // per matrix 1 / (||update||_F + eps)
  const StepParams* sp;      // lr and decays of the update
  int* err;                  // device error flag
  int32_t nmat, L, steps;
  int32_t stall_test;        // test hook: CTA 0 loads no X (its bounded wait runs out)
  float coef[64][3];         // (a, b, c) of each iteration
};
bool tc_encode_small(SmallLaunch& sl, const uint16_t* X, int nmat, int L, char* errbuf, size_t errlen);
cudaError_t launch_ns_small(const SmallLaunch& L, int num_sms, cudaStream_t st);  // grid: min(nmat, num_sms)

// Newton-Schulz of narrow matrices (short side < kNarrowMinS) in fp32 on the
// CUDA cores (ns_narrow.cu), from the update (recomputed from the momentum
// buffer and the gradient) through the parameter update, in one launch per
// group of matrices:
//   resident (cluster >= 1): a cluster of `cluster` CTAs per matrix, each CTA
//     holding a slice of the long side of X in shared memory for the whole
//     chain; the partial Gram matrices are summed through distributed shared
//     memory;
//   streaming (cluster == 0): one CTA per matrix, X in the matrix's fp32
//     workspace (xf), streamed through shared memory in 64-column chunks (for
//     matrices whose slices would not fit in 8 CTAs' shared memory).
struct NarrowLaunch {
  const MuonMat* mats;
  const int32_t* idx;        // the launch's matrices (indices into mats), largest first
  const StepScalars* sc;     // clip coefficient
  const StepParams* sp;      // lr and decays of the update
  int32_t nmat, steps;
  int32_t nesterov;
  int32_t cluster;           // CTAs per matrix (resident), 0 = streaming
  float mu, gscale;          // momentum coefficient, weight of the clipped gradient
  float eps;                 // of the Frobenius normalisation
  float coef[64][3];         // (a, b, c) of each iteration
};

// Shape plan of the resident kernel, shared by the host planner and the
// kernel: target columns of the long side per CTA, rows of the X slice held
// in shared memory (row s, read by some warps of the last live row group, is
// zero), columns per CTA (a multiple of 4; the last CTA may have fewer or
// none), and the row pitch in floats (a multiple of 64, plus 4).
constexpr int kNarrowColsPerCta = 256;
constexpr int kNarrowMaxCluster = 8;
constexpr size_t kNarrowMaxSmem = 227 * 1024;
constexpr int kNarrowFixedFloats = 2 * 64 * 68 + 32;  // two A / B tiles and 16 doubles
__host__ __device__ inline int narrow_rows(int s) {
  const int r = (s + 16) / 16 * 16;
  return r > 64 ? 64 : r;
}
__host__ __device__ inline int narrow_cols(int l, int cluster) { return ((l + cluster - 1) / cluster + 3) & ~3; }
__host__ __device__ inline int narrow_pitch(int lc) { return (lc + 63) / 64 * 64 + 4; }
inline size_t narrow_resident_smem(int s, int l, int cluster) {
  return ((size_t)kNarrowFixedFloats + (size_t)narrow_rows(s) * narrow_pitch(narrow_cols(l, cluster))) * 4;
}
// Cluster size for a narrow s x l matrix (canonical s <= l): the smallest
// power of two giving at most kNarrowColsPerCta columns per CTA, capped at
// kNarrowMaxCluster; 0 if its slices then exceed kNarrowMaxSmem (streaming).
inline int narrow_cluster_for(int s, int l) {
  int c = 1;
  while (c < kNarrowMaxCluster && (l + c - 1) / c > kNarrowColsPerCta) c *= 2;
  return narrow_resident_smem(s, l, c) <= kNarrowMaxSmem ? c : 0;
}

// Sets the kernels' shared-memory attributes (the resident kernel's to
// resident_smem bytes); returns the streaming kernel's resident CTAs per SM.
cudaError_t ns_narrow_prepare(size_t resident_smem, int* stream_blocks_per_sm);
// Resident: grid nmat x cluster CTAs, `smem` bytes each. Streaming: grid
// min(nmat, blocks_per_sm x num_sms), a grid-stride loop over the matrices.
cudaError_t launch_ns_narrow(const NarrowLaunch& L, size_t smem, int num_sms, int blocks_per_sm, cudaStream_t st);

// Partition of the trainable parameters over `world` ranks (host; shard.cu).
// group/numel/rows/cols per parameter (rows, cols used for Muon matrices).
// owner[i]: the rank that updates Muon matrix i (-1 otherwise); begin/end
// [i * world + r]: the elements [begin, end) of parameter i that rank r
// updates (the whole matrix at its owner, a contiguous range for AdamW,
// empty otherwise).
void shard_partition(const std::vector<int>& group, const std::vector<int64_t>& numel,
                     const std::vector<int64_t>& rows, const std::vector<int64_t>& cols, int world,
                     std::vector<int>& owner, std::vector<int64_t>& begin, std::vector<int64_t>& end);

// Static assignment of a launch's work units to `ncl` clusters (host): each
// unit, in the launch's order (longest first), goes to the cluster with the
// least work so far (a unit costs its K / 64 k-steps plus a fixed 6), ties to
// the lowest index; laid out round by round, -1 where a cluster has no unit.
// Units of equal cost give the plain round-robin order.
void tc_unit_order(const TcLaunch& L, int ncl, std::vector<int32_t>& order);
// Sets the kernels' dynamic shared-memory limit (current device) and returns
// how many CTA pairs can be resident at once.
cudaError_t ns_tc_prepare(int* max_pairs);
// grid_units: clusters to launch (CTAs = grid_units * cl), capped at the work units.
cudaError_t launch_ns_tc(const TcLaunch& L, cudaStream_t st);  // grid: L.nclusters clusters
int ns_tc_num_tiles_sym(int units_m, int bmu, int bn);  // lower-triangle work units per matrix

}  // namespace ma
