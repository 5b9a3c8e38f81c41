// Host runtime of the hybrid Muon + AdamW optimizer and its C ABI.
//
// OpenDM VLA training-stack article (gsyq.cn/news/451971), 核心揭秘一:
//   - 参数如何分流: routing of parameters to Muon or AdamW (is_muon_param);
//     the parameter list is frozen before the first step (the article records
//     shapes before wrapping, which this library mirrors by freezing the plan
//     at the first step);
//   - 关键超参默认值: momentum 0.95 (Nesterov), 5 Newton-Schulz steps, lr scale
//     0.2 * sqrt(max(shape));
//   - 训练栈默认参数速查表: max_grad_norm 1.0, cosine_with_min_lr (min 0.1).
// Everything on the device runs in the kernels of stream_kernels.cu, ns_tc.cu
// (and the ns_simt.cu cross-check); this file plans, allocates and launches.
#include <cuda_runtime.h>
#include <ctype.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <string>
#include <type_traits>
#include <utility>
#include <vector>

#include "muon_adamw.h"
#include "internal.h"

using namespace ma;

namespace {

thread_local std::string g_last_error;

ma_status fail(ma_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

ma_status ok() {
  g_last_error.clear();
  return MA_OK;
}

#define CUDA_TRY(expr)                                                                        \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess) {                                                                  \
      return fail(e_ == cudaErrorMemoryAllocation ? MA_ERR_OOM : MA_ERR_CUDA, "%s: %s (%s:%d)", \
                  #expr, cudaGetErrorString(e_), __FILE__, __LINE__);                         \
    }                                                                                         \
  } while (0)

bool contains(const std::string& s, const char* sub) { return s.find(sub) != std::string::npos; }

bool route_is_muon(const char* name, int ndim) {
  if (!name || ndim != 2) return false;
  const std::string n(name);
  if (!contains(n, "action_expert")) return false;
  bool under_layers = false;
  size_t start = 0;
  while (start <= n.size()) {
    size_t dot = n.find('.', start);
    if (dot == std::string::npos) dot = n.size();
    if (n.compare(start, dot - start, "layers") == 0 && dot - start == 6) under_layers = true;
    start = dot + 1;
  }
  if (!under_layers) return false;
  static const char kSuffix[] = ".weight";
  if (n.size() < sizeof(kSuffix) - 1 || n.compare(n.size() - (sizeof(kSuffix) - 1), std::string::npos, kSuffix) != 0)
    return false;
  std::string low(n);
  for (char& ch : low)
    if (ch >= 'A' && ch <= 'Z') ch = (char)(ch - 'A' + 'a');
  if (contains(low, "embed") || contains(low, "lm_head") || contains(low, "norm")) return false;
  return true;
}

int64_t pad_up(int64_t x, int64_t g) { return (x + g - 1) / g * g; }

struct Param {
  std::string name;
  std::vector<int64_t> shape;
  int64_t numel = 0;
  float* p = nullptr;
  const void* g = nullptr;
  int gdtype = MA_DT_BF16;
  uint16_t* shadow = nullptr;
  int group = MA_GROUP_ADAMW;
  float* st0 = nullptr;  // Muon buf or AdamW m
  float* st1 = nullptr;  // AdamW v
  double lr_scale = 1.0, wd_scale = 1.0;  // per-parameter multipliers
  bool options_set = false;               // set explicitly (wins over the exemption rule)
  int og = 0;                             // option group (index into the per-step tables)
  int64_t own_b = 0, own_e = 0;           // the elements this rank updates (all of them unless sharded)
};

struct Bucket {
  int S = 0, L = 0;
  std::vector<int> params;  // param indices in slot order
  int mat0 = 0;             // first index in the MuonMat table
  uint16_t *X0 = nullptr, *X1 = nullptr, *A = nullptr, *B = nullptr;
  bool fused = false;   // small matrices: the whole Newton-Schulz in one launch (ns_small_kernel)
  bool narrow = false;  // short side < kNarrowMinS: fp32 Newton-Schulz (ns_narrow_kernel)
  float* XF = nullptr;  // narrow, streamed: fp32 X of each slot (xf_stride floats per slot)
  size_t xf_stride = 0;  // narrow: the bucket's largest m n, rounded up to 64 floats
  bool narrow_stream = false;  // narrow: some matrix too long for a resident cluster (needs XF)
};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
  double units;
};

}  // namespace

namespace ma {
void set_last_error(const char* msg) { g_last_error = msg; }
void clear_last_error() { g_last_error.clear(); }
}  // namespace ma

struct muon_adamw {
  muon_adamw_config cfg{};
  int device = 0;
  int num_sms = 0;
  int max_pairs = 1;          // co-resident CTA pairs of the tensor-core kernel
  bool stall_test = false;    // one-shot test hook armed by muon_adamw_test_arm_stall
  cudaStream_t s0 = nullptr;  // caller's stream
  cudaStream_t s1 = nullptr;  // AdamW stream (library-owned)
  cudaStream_t s2 = nullptr;  // joins the gradient readers for muon_adamw_record_grads_consumed
  cudaEvent_t ev_fork = nullptr;
  cudaEvent_t ev_g0 = nullptr, ev_g1 = nullptr;  // last gradient reader of the latest step on s0 / s1
  bool g1_valid = false;                          // the latest step read gradients on s1
  StepParams* d_step = nullptr;                   // this step's scalars (arena)
  StepParams* h_step = nullptr;                   // two pinned host slots, alternating per step
  cudaEvent_t ev_slot[2] = {nullptr, nullptr};    // a slot's copy has been read
  bool graph_mode = true;                         // run steps as captured CUDA graphs
  bool graph_broken = false;                      // capture failed: direct launches from now on
  cudaGraphExec_t gexec = nullptr;                // the captured Newton-Schulz chain
  std::vector<Param> params;
  bool planned = false;
  int shard_rank = 0, shard_world = 1;  // sharded step: this rank's part of the parameters
  bool begun = false;                   // sharded step: step_begin queued, step_end not yet
  std::vector<std::pair<double, double>> option_groups;  // (lr_scale, wd_scale); [0] = (1, 1)
  int64_t t = 0;

  // arena
  void* arena = nullptr;
  size_t arena_bytes = 0;
  size_t state_bytes = 0, workspace_bytes = 0;

  // device tables
  GradChunk* d_norm_chunks = nullptr;
  int n_norm_chunks = 0;
  int norm_grid = 0;
  float* d_norm_partials = nullptr;
  AdamChunk* d_adam_chunks = nullptr;
  int n_adam_chunks = 0;
  int adam_grid = 0;
  MuonMat* d_mats = nullptr;
  CUtensorMap* d_pmaps = nullptr;  // per Muon matrix: TMA maps of p and shadow
  int32_t* d_orders = nullptr;     // work orders of the tensor-core launches
  int n_mats = 0;
  MomTile* d_tiles = nullptr;
  int n_tiles = 0;
  int mom_grid = 0;
  float* d_tile_partials = nullptr;
  float* d_rscale = nullptr;
  StepScalars* d_scalars = nullptr;
  int* d_err = nullptr;

  std::vector<Bucket> buckets;
  std::vector<int> muon_params, adam_params;
  // per iteration, per kind: launches (tcgen05) or problems (SIMT)
  std::vector<std::vector<TcLaunch>> tc[3];
  std::vector<SmallLaunch> small;      // one per fused bucket
  std::vector<double> small_units;     // their symmetric flops per step
  double unit_fused = 0;               // symmetric flops per step of all fused buckets
  std::vector<NarrowLaunch> narrow;    // narrow matrices: one launch per cluster size, then the streamed ones
  std::vector<size_t> narrow_smem;     // their dynamic shared memory
  std::vector<double> narrow_units;    // their symmetric flops per step
  int narrow_per_sm = 1;               // resident CTAs per SM of the streaming kernel
  int32_t* d_narrow_idx = nullptr;     // the launches' matrix indices
  double unit_narrow = 0;              // symmetric flops per step of all narrow buckets
  std::vector<std::vector<NsProblem>> simt[3];
  double unit_gram = 0, unit_poly = 0, unit_update = 0;  // symmetric flops per iteration (all buckets)
  double dense_flops = 0;
  double bytes_norm = 0, bytes_mom = 0, bytes_adam = 0;
  int64_t muon_elems = 0, adam_elems = 0, grad_elems = 0;

  // profiling
  bool profiling = false;
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> ev_pool;
  ma_profile prof{};
};

namespace {

cudaEvent_t take_event(muon_adamw* h) {
  if (!h->ev_pool.empty()) {
    cudaEvent_t e = h->ev_pool.back();
    h->ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launch helper: records a profiling event pair around `fn` when enabled, and
// returns the launch status `fn` returns (cudaSuccess for launchers that leave
// a failure to the step's final cudaGetLastError).
template <class F>
cudaError_t timed(muon_adamw* h, int kind, cudaStream_t st, double units, F&& fn) {
  auto call = [&]() -> cudaError_t {
    if constexpr (std::is_same_v<decltype(fn()), void>) {
      fn();
      return cudaSuccess;
    } else {
      return fn();
    }
  };
  if (!h->profiling) return call();
  ProfRec r{kind, take_event(h), take_event(h), units};
  if (r.a) cudaEventRecord(r.a, st);
  const cudaError_t e = call();
  if (r.b) cudaEventRecord(r.b, st);
  if (r.a && r.b) h->prof_pending.push_back(r);
  return e;
}

ma_status fold_profile(muon_adamw* h) {
  for (const ProfRec& r : h->prof_pending) {
    float ms = 0.f;
    cudaError_t e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) return fail(MA_ERR_CUDA, "cudaEventElapsedTime: %s", cudaGetErrorString(e));
    h->prof.launches[r.kind] += 1;
    h->prof.ms[r.kind] += ms;
    h->prof.units[r.kind] += r.units;
    h->ev_pool.push_back(r.a);
    h->ev_pool.push_back(r.b);
  }
  h->prof_pending.clear();
  return MA_OK;
}

// Biases and normalisation weights (HF Trainer's decay-exemption convention).
bool decay_exempt_name(const std::string& name) {
  std::string low(name);
  for (char& ch : low) ch = (char)tolower((unsigned char)ch);
  const bool bias = low.size() >= 4 && low.compare(low.size() - 4, 4, "bias") == 0;
  return bias || low.find("norm") != std::string::npos;
}

ma_status check_device_flag(muon_adamw* h) {
  if (!h->d_err) return MA_OK;
  int err = 0;
  CUDA_TRY(cudaMemcpy(&err, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (err != 0) {
    cudaMemset(h->d_err, 0, sizeof(int));
    return fail(MA_ERR_DEVICE_CHECK, "a kernel's bounded wait ran out (code 0x%x); its step was not completed", err);
  }
  return MA_OK;
}

void set_epi_coefficients(NsEpiArgs& e, const muon_adamw_config& c, int it);

// The elements of each parameter that this rank updates: all of every
// trainable parameter, or this rank's part of the partition of shard.cu.
void assign_ownership(muon_adamw* h) {
  const size_t n = h->params.size();
  if (h->shard_world <= 1) {
    for (Param& p : h->params) {
      p.own_b = 0;
      p.own_e = p.group == MA_GROUP_FROZEN ? 0 : p.numel;
    }
    return;
  }
  std::vector<int> group(n), owner;
  std::vector<int64_t> numel(n), rows(n), cols(n), b, e;
  for (size_t i = 0; i < n; ++i) {
    const Param& p = h->params[i];
    group[i] = p.group;
    numel[i] = p.numel;
    rows[i] = p.shape.size() == 2 ? p.shape[0] : p.numel;
    cols[i] = p.shape.size() == 2 ? p.shape[1] : 1;
  }
  shard_partition(group, numel, rows, cols, h->shard_world, owner, b, e);
  for (size_t i = 0; i < n; ++i) {
    h->params[i].own_b = b[i * (size_t)h->shard_world + (size_t)h->shard_rank];
    h->params[i].own_e = e[i * (size_t)h->shard_world + (size_t)h->shard_rank];
  }
}

ma_status build_plan(muon_adamw* h) {
  const muon_adamw_config& c = h->cfg;
  if (h->arena) {  // a previous attempt failed part-way
    cudaFree(h->arena);
    h->arena = nullptr;
  }
  // --- ownership (the whole of every trainable parameter unless sharded) ---
  assign_ownership(h);
  // --- classify: the parameters this rank updates ---
  h->muon_params.clear();
  h->adam_params.clear();
  for (int i = 0; i < (int)h->params.size(); ++i) {
    const Param& p = h->params[i];
    if (p.own_e <= p.own_b) continue;
    if (p.group == MA_GROUP_MUON) h->muon_params.push_back(i);
    if (p.group == MA_GROUP_ADAMW) h->adam_params.push_back(i);
  }
  // --- buckets (by padded canonical shape and narrowness, first-seen order; narrow ones moved first below) ---
  std::map<std::pair<std::pair<int, int>, bool>, int> bidx;
  h->buckets.clear();
  for (int pi : h->muon_params) {
    const Param& p = h->params[pi];
    const int64_t m = p.shape[0], n = p.shape[1];
    const int S = (int)pad_up(std::min(m, n), kPad), L = (int)pad_up(std::max(m, n), kPad);
    const bool narrow = std::min(m, n) < kNarrowMinS;
    auto key = std::make_pair(std::make_pair(S, L), narrow);
    auto it = bidx.find(key);
    if (it == bidx.end()) {
      bidx[key] = (int)h->buckets.size();
      Bucket b;
      b.S = S;
      b.L = L;
      b.narrow = narrow;
      h->buckets.push_back(b);
      it = bidx.find(key);
    }
    h->buckets[it->second].params.push_back(pi);
  }
  for (Bucket& B : h->buckets)
    B.fused = c.ns_kernel == MA_NS_TCGEN05 && !(c.reserved[0] & 8) && !B.narrow && B.S == 128 &&
              B.L <= kSmallMaxL;
  // narrow buckets first, the costliest (S^2 L) first: their matrices are then
  // one contiguous, largest-first run of the matrix table, which a single
  // ns_narrow_kernel launch takes (the other buckets keep their order)
  std::stable_sort(h->buckets.begin(), h->buckets.end(), [](const Bucket& a, const Bucket& b) {
    if (a.narrow != b.narrow) return a.narrow;
    return a.narrow && (double)a.S * a.S * a.L > (double)b.S * b.S * b.L;
  });
  int n_narrow = 0;
  for (Bucket& B : h->buckets) {
    if (!B.narrow) continue;
    int64_t mx = 0;
    for (int pi : B.params) {
      const Param& p = h->params[pi];
      mx = std::max(mx, p.numel);
      const int s = (int)std::min(p.shape[0], p.shape[1]), l = (int)std::max(p.shape[0], p.shape[1]);
      if (narrow_cluster_for(s, l) == 0) B.narrow_stream = true;
    }
    B.xf_stride = (size_t)((mx + 63) / 64 * 64);
    n_narrow += (int)B.params.size();
  }
  // --- sizes ---
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  std::vector<size_t> st0_off(h->params.size(), 0), st1_off(h->params.size(), 0);
  for (int pi : h->muon_params) {
    st0_off[pi] = off;
    off += al(h->params[pi].numel * sizeof(float));
  }
  for (int pi : h->adam_params) {
    const int64_t n_own = h->params[pi].own_e - h->params[pi].own_b;
    st0_off[pi] = off;
    off += al(n_own * sizeof(float));
    st1_off[pi] = off;
    off += al(n_own * sizeof(float));
  }
  h->state_bytes = off;
  // per bucket: X ping, X pong (s x l), A, B (s x s), all bf16; a narrow
  // bucket: X (bf16, written by the momentum pass and not read) and its fp32
  // X in place of the other three
  std::vector<size_t> ws_off(h->buckets.size() * 4);
  for (size_t b = 0; b < h->buckets.size(); ++b) {
    const Bucket& B = h->buckets[b];
    const size_t nb = B.params.size();
    const size_t xs = al(nb * (size_t)B.S * B.L * 2), as = al(nb * (size_t)B.S * B.S * 2);
    const size_t sizes[4] = {xs, B.narrow ? (B.narrow_stream ? al(nb * B.xf_stride * 4) : 0) : xs, B.narrow ? 0 : as,
                             B.narrow ? 0 : as};
    for (int q = 0; q < 4; ++q) {
      ws_off[4 * b + q] = off;
      off += sizes[q];
    }
  }
  h->workspace_bytes = off - h->state_bytes;

  // --- counts of the device tables ---
  auto chunks_of = [](int64_t n) { return (size_t)((n + kChunk - 1) / kChunk); };
  size_t n_norm = 0, n_adam = 0, n_tiles = 0, n_mats = 0;
  for (const Param& p : h->params)
    if (p.group != MA_GROUP_FROZEN && p.own_e > p.own_b) n_norm += chunks_of(p.own_e - p.own_b);
  for (int pi : h->adam_params) n_adam += chunks_of(h->params[pi].own_e - h->params[pi].own_b);
  for (int pi : h->muon_params) {
    const Param& p = h->params[pi];
    const bool tall = p.shape[0] > p.shape[1];
    const int64_t tr = tall ? kMomTile : kMomWideRows, tc = tall ? kMomTile : kMomWideCols;
    n_tiles += (size_t)((p.shape[0] + tr - 1) / tr) * (size_t)((p.shape[1] + tc - 1) / tc);
    ++n_mats;
  }
  h->norm_grid = (int)std::max<size_t>(1, std::min<size_t>(n_norm, (size_t)4 * h->num_sms));
  h->adam_grid = (int)std::max<size_t>(1, std::min<size_t>(n_adam, (size_t)8 * h->num_sms));
  h->mom_grid = (int)std::max<size_t>(1, std::min<size_t>(n_tiles, (size_t)8 * h->num_sms));
  const size_t off_norm_chunks = off;
  off += al(n_norm * sizeof(GradChunk));
  const size_t off_norm_part = off;
  off += al(h->norm_grid * sizeof(float));
  const size_t off_adam_chunks = off;
  off += al(n_adam * sizeof(AdamChunk));
  const size_t off_mats = off;
  off += al(n_mats * sizeof(MuonMat));
  const size_t off_pmaps = off;
  off += al(n_mats * 2 * sizeof(CUtensorMap));
  const size_t off_tiles = off;
  off += al(n_tiles * sizeof(MomTile));
  const size_t off_tile_part = off;
  off += al(n_tiles * kMomPartialsPerTile * sizeof(float));
  const size_t off_rscale = off;
  off += al(n_mats * sizeof(float));
  const size_t off_scalars = off;
  off += al(sizeof(StepScalars));
  const size_t off_step = off;
  off += al(sizeof(StepParams));
  const size_t off_err = off;
  off += al(sizeof(int));
  const size_t off_nidx = off;
  off += al((size_t)n_narrow * sizeof(int32_t));
  h->arena_bytes = off;

  // --- allocate and zero (state starts at zero; workspace padding stays zero) ---
  CUDA_TRY(cudaMalloc(&h->arena, h->arena_bytes));
  CUDA_TRY(cudaMemsetAsync(h->arena, 0, h->arena_bytes, h->s0));
  char* base = static_cast<char*>(h->arena);
  for (int pi : h->muon_params) h->params[pi].st0 = reinterpret_cast<float*>(base + st0_off[pi]);
  for (int pi : h->adam_params) {
    h->params[pi].st0 = reinterpret_cast<float*>(base + st0_off[pi]);
    h->params[pi].st1 = reinterpret_cast<float*>(base + st1_off[pi]);
  }
  for (size_t b = 0; b < h->buckets.size(); ++b) {
    Bucket& B = h->buckets[b];
    B.X0 = reinterpret_cast<uint16_t*>(base + ws_off[4 * b + 0]);
    if (B.narrow) {
      B.XF = B.narrow_stream ? reinterpret_cast<float*>(base + ws_off[4 * b + 1]) : nullptr;
      B.X1 = B.A = B.B = nullptr;
    } else {
      B.XF = nullptr;
      B.X1 = reinterpret_cast<uint16_t*>(base + ws_off[4 * b + 1]);
      B.A = reinterpret_cast<uint16_t*>(base + ws_off[4 * b + 2]);
      B.B = reinterpret_cast<uint16_t*>(base + ws_off[4 * b + 3]);
    }
  }
  h->d_norm_chunks = reinterpret_cast<GradChunk*>(base + off_norm_chunks);
  h->n_norm_chunks = (int)n_norm;
  h->d_norm_partials = reinterpret_cast<float*>(base + off_norm_part);
  h->d_adam_chunks = reinterpret_cast<AdamChunk*>(base + off_adam_chunks);
  h->n_adam_chunks = (int)n_adam;
  h->d_mats = reinterpret_cast<MuonMat*>(base + off_mats);
  h->d_pmaps = reinterpret_cast<CUtensorMap*>(base + off_pmaps);
  h->d_tiles = reinterpret_cast<MomTile*>(base + off_tiles);
  h->d_tile_partials = reinterpret_cast<float*>(base + off_tile_part);
  h->d_rscale = reinterpret_cast<float*>(base + off_rscale);
  h->d_scalars = reinterpret_cast<StepScalars*>(base + off_scalars);
  h->d_step = reinterpret_cast<StepParams*>(base + off_step);
  h->d_err = reinterpret_cast<int*>(base + off_err);
  h->d_narrow_idx = reinterpret_cast<int32_t*>(base + off_nidx);

  // --- host tables with device pointers ---
  std::vector<GradChunk> norm_chunks;
  std::vector<AdamChunk> adam_chunks;
  std::vector<MuonMat> mats;
  std::vector<CUtensorMap> pmaps;
  std::vector<MomTile> tiles;
  norm_chunks.reserve(n_norm);
  adam_chunks.reserve(n_adam);
  tiles.reserve(n_tiles);
  h->grad_elems = h->muon_elems = h->adam_elems = 0;
  h->bytes_norm = h->bytes_mom = h->bytes_adam = 0;
  for (size_t i = 0; i < h->params.size(); ++i) {
    const Param& p = h->params[i];
    if (p.group == MA_GROUP_FROZEN || p.own_e <= p.own_b) continue;
    const size_t es = p.gdtype == MA_DT_BF16 ? 2 : 4;
    const int64_t n_own = p.own_e - p.own_b;
    h->grad_elems += n_own;
    h->bytes_norm += (double)n_own * es;
    for (int64_t o = 0; o < n_own; o += kChunk) {
      GradChunk gc;
      gc.g = static_cast<const char*>(p.g) + (p.own_b + o) * es;
      gc.n = std::min<int64_t>(kChunk, n_own - o);
      gc.dtype = p.gdtype == MA_DT_BF16 ? DT_BF16 : DT_F32;
      gc.vec = (reinterpret_cast<uintptr_t>(gc.g) % 16) == 0;
      norm_chunks.push_back(gc);
    }
  }
  // option groups: distinct (lr_scale, wd_scale) pairs, group 0 = (1, 1)
  h->option_groups.assign(1, {1.0, 1.0});
  for (Param& p : h->params) {
    if (p.group == MA_GROUP_FROZEN) continue;
    if (!p.options_set) {
      p.lr_scale = 1.0;
      p.wd_scale = (c.adam_decay_exempt_bias_norm && p.group == MA_GROUP_ADAMW && decay_exempt_name(p.name)) ? 0.0 : 1.0;
    }
    const std::pair<double, double> key{p.lr_scale, p.wd_scale};
    size_t gi = 0;
    while (gi < h->option_groups.size() && h->option_groups[gi] != key) ++gi;
    if (gi == h->option_groups.size()) {
      if ((int)gi == kMaxOptionGroups)
        return fail(MA_ERR_UNSUPPORTED, "more than %d distinct (lr_scale, weight_decay_scale) pairs",
                    kMaxOptionGroups);
      h->option_groups.push_back(key);
    }
    p.og = (int)gi;
  }
  for (int pi : h->adam_params) {
    const Param& p = h->params[pi];
    const size_t es = p.gdtype == MA_DT_BF16 ? 2 : 4;
    const int64_t n_own = p.own_e - p.own_b;
    h->adam_elems += n_own;
    h->bytes_adam += (double)n_own * (es + 24 + (p.shadow ? 2 : 0));
    for (int64_t o = 0; o < n_own; o += kChunk) {
      const int64_t e0 = p.own_b + o;  // element of the parameter; the state holds the owned range only
      AdamChunk a;
      a.p = p.p + e0;
      a.g = static_cast<const char*>(p.g) + e0 * es;
      a.m = p.st0 + o;
      a.v = p.st1 + o;
      a.shadow = p.shadow ? p.shadow + e0 : nullptr;
      a.n = std::min<int64_t>(kChunk, n_own - o);
      a.gdtype = p.gdtype == MA_DT_BF16 ? DT_BF16 : DT_F32;
      const uintptr_t pa = reinterpret_cast<uintptr_t>(a.p), ga = reinterpret_cast<uintptr_t>(a.g),
                      sa = reinterpret_cast<uintptr_t>(a.shadow);
      a.vec = (pa % 16 == 0) && (ga % (a.gdtype == DT_BF16 ? 8 : 16) == 0) && (sa % 8 == 0);
      a.group = p.og;
      a.pad = 0;
      adam_chunks.push_back(a);
    }
  }
  int mat_index = 0;
  h->unit_gram = h->unit_poly = h->unit_update = h->dense_flops = h->unit_fused = h->unit_narrow = 0;
  h->small_units.clear();
  for (size_t b = 0; b < h->buckets.size(); ++b) {
    Bucket& B = h->buckets[b];
    B.mat0 = mat_index;
    double bucket_units = 0;
    for (size_t slot = 0; slot < B.params.size(); ++slot) {
      const Param& p = h->params[B.params[slot]];
      const size_t es = p.gdtype == MA_DT_BF16 ? 2 : 4;
      MuonMat M{};
      M.p = p.p;
      M.g = p.g;
      M.buf = p.st0;
      M.shadow = p.shadow;
      M.x0 = B.X0 + slot * (size_t)B.S * B.L;
      M.m = (int)p.shape[0];
      M.n = (int)p.shape[1];
      M.s = std::min(M.m, M.n);
      M.l = std::max(M.m, M.n);
      M.S = B.S;
      M.L = B.L;
      M.transposed = M.m > M.n;
      M.gdtype = p.gdtype == MA_DT_BF16 ? DT_BF16 : DT_F32;
      M.vec = (M.n % 8 == 0) && (reinterpret_cast<uintptr_t>(p.g) % 16 == 0);
      M.pvec = (M.n % 8 == 0) && (reinterpret_cast<uintptr_t>(p.p) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(p.shadow) % 16 == 0);
      M.lr_mult = (float)(p.lr_scale * c.muon_lr_scale * c.moonlight_coef * sqrt((double)M.l));
      M.group = p.og;
      M.xf = B.XF ? B.XF + slot * B.xf_stride : nullptr;
      pmaps.resize(2 * (size_t)(mat_index + 1));
      M.tma = (c.ns_kernel == MA_NS_TCGEN05 && !(c.reserved[0] & 4) &&
               tc_encode_param_maps(&pmaps[2 * (size_t)mat_index], M))
                  ? 1
                  : 0;
      M.tile_begin = (int)tiles.size();
      const int tr = M.transposed ? kMomTile : kMomWideRows, tcol = M.transposed ? kMomTile : kMomWideCols;
      for (int r0 = 0; r0 < M.m; r0 += tr)
        for (int c0 = 0; c0 < M.n; c0 += tcol) tiles.push_back(MomTile{mat_index, r0, c0, 0});
      M.tile_end = (int)tiles.size();
      mats.push_back(M);
      ++mat_index;
      const double s = M.s, l = M.l;
      h->muon_elems += p.numel;
      h->bytes_mom += (double)p.numel * (es + 8 + 2);
      if (B.fused || B.narrow) {
        bucket_units += (double)c.ns_steps * (s * (s + 1) * l + s * (s + 1) * s + 2 * s * s * l);
      } else {
        h->unit_gram += s * (s + 1) * l;
        h->unit_poly += s * (s + 1) * s;
        h->unit_update += 2 * s * s * l;
      }
      h->dense_flops += (double)c.ns_steps * (4 * s * s * l + 2 * s * s * s);
    }
    if (B.fused) {
      h->small_units.push_back(bucket_units);
      h->unit_fused += bucket_units;
    } else if (B.narrow) {
      h->unit_narrow += bucket_units;
    }
  }
  h->n_mats = mat_index;
  h->n_tiles = (int)tiles.size();
  if (!norm_chunks.empty())
    CUDA_TRY(cudaMemcpyAsync(h->d_norm_chunks, norm_chunks.data(), norm_chunks.size() * sizeof(GradChunk),
                             cudaMemcpyHostToDevice, h->s0));
  if (!adam_chunks.empty())
    CUDA_TRY(cudaMemcpyAsync(h->d_adam_chunks, adam_chunks.data(), adam_chunks.size() * sizeof(AdamChunk),
                             cudaMemcpyHostToDevice, h->s0));
  if (!mats.empty())
    CUDA_TRY(cudaMemcpyAsync(h->d_mats, mats.data(), mats.size() * sizeof(MuonMat), cudaMemcpyHostToDevice, h->s0));
  if (!pmaps.empty())
    CUDA_TRY(cudaMemcpyAsync(h->d_pmaps, pmaps.data(), pmaps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice,
                             h->s0));
  if (!tiles.empty())
    CUDA_TRY(cudaMemcpyAsync(h->d_tiles, tiles.data(), tiles.size() * sizeof(MomTile), cudaMemcpyHostToDevice, h->s0));
  CUDA_TRY(cudaStreamSynchronize(h->s0));

  // --- Newton-Schulz launch descriptions ---
  const int steps = c.ns_steps;
  for (int k = 0; k < 3; ++k) {
    h->tc[k].assign(steps, {});
    h->simt[k].assign(steps, {});
  }
  for (int it = 0; it < steps; ++it) {
    for (int kind = 0; kind < 3; ++kind) {
      std::vector<NsProblem> probs;
      for (Bucket& B : h->buckets) {
        if (B.fused || B.narrow) continue;  // ns_small_kernel or ns_narrow_kernel takes the whole chain
        uint16_t* Xcur = (it % 2 == 0) ? B.X0 : B.X1;
        uint16_t* Xnext = (it % 2 == 0) ? B.X1 : B.X0;
        NsProblem p{};
        p.kind = kind;
        p.S = B.S;
        p.L = B.L;
        p.nmat = (int)B.params.size();
        p.mats = h->d_mats + B.mat0;
        p.rscale = h->d_rscale + B.mat0;
        p.pmaps = h->d_pmaps + 2 * (size_t)B.mat0;
        p.first = it == 0;
        p.last = it == steps - 1;
        p.shadow = 0;
        for (int pi : B.params) p.shadow |= h->params[pi].shadow != nullptr ? 1 : 0;
        if (kind == NS_GRAM) {
          p.P = Xcur;
          p.Q = Xcur;
          p.aux = nullptr;
          p.out = B.A;
          p.M = B.S;
          p.N = B.S;
          p.K = B.L;
        } else if (kind == NS_POLY) {
          p.P = B.A;
          p.Q = B.A;
          p.aux = B.A;
          p.out = B.B;
          p.M = B.S;
          p.N = B.S;
          p.K = B.S;
        } else {
          p.P = B.B;
          p.Q = Xcur;
          p.aux = nullptr;
          p.out = Xnext;
          p.M = B.S;
          p.N = B.L;
          p.K = B.S;
        }
        probs.push_back(p);
      }
      h->simt[kind][it] = probs;
      if (c.ns_kernel == MA_NS_TCGEN05) {
        // X X^T, A A and the last iteration run in CTA pairs (one M = 256 MMA
        // over both CTAs) where their row blocks pair up; X' = B X of the other
        // iterations and unpaired problems run in single CTAs
        const bool allow_pairs = !(c.reserved[0] & 2);
        for (int cl = 2; cl >= 1; --cl) {
          std::vector<NsProblem> group;
          for (const NsProblem& pp : probs) {
            const bool paired = allow_pairs && ns_tc_pairable(pp);
            if ((cl == 2) == paired) group.push_back(pp);
          }
          // longest work units first: the static round-robin then ends on short units
          std::stable_sort(group.begin(), group.end(),
                           [](const NsProblem& a, const NsProblem& b) { return a.K > b.K; });
          for (size_t b0 = 0; b0 < group.size(); b0 += kTcMaxProblems) {
            TcLaunch L;
            memset(&L, 0, sizeof L);
            int tiles_total = 0;
            for (size_t q = 0; q < (size_t)kTcMaxProblems && b0 + q < group.size(); ++q) {
              TcProblem& tp = L.prob[q];
              tp.p = group[b0 + q];
              char eb[256];
              if (!tc_encode_problem(tp, cl, eb, sizeof eb)) return fail(MA_ERR_CUDA, "%s", eb);
              tp.tile_begin = tiles_total;
              tiles_total += tp.tiles_per_mat * tp.p.nmat;
              L.nprob = (int)q + 1;
            }
            L.total_tiles = tiles_total;
            L.err = h->d_err;
            L.cl = cl;
            for (int q = 0; q < L.nprob; ++q) L.shadow |= L.prob[q].p.shadow;
            h->tc[kind][it].push_back(L);
          }
        }
      }
    }
  }
  h->narrow.clear();
  h->narrow_smem.clear();
  h->narrow_units.clear();
  if (n_narrow > 0) {
    // the narrow matrices lead the matrix table (their buckets come first,
    // costliest first); one launch per cluster size, each over its matrices
    // in table order, then the streamed ones
    NarrowLaunch base;
    memset(&base, 0, sizeof base);
    base.mats = h->d_mats;
    base.sc = h->d_scalars;
    base.sp = h->d_step;
    base.steps = c.ns_steps;
    base.nesterov = c.muon_nesterov;
    base.mu = (float)c.muon_momentum;
    base.gscale = c.muon_momentum_form == MA_MOMENTUM_EMA ? (float)(1.0 - c.muon_momentum) : 1.0f;
    base.eps = (float)c.ns_eps;
    for (int it = 0; it < c.ns_steps; ++it) {
      NsEpiArgs e{};
      set_epi_coefficients(e, c, it);
      base.coef[it][0] = e.a;
      base.coef[it][1] = e.b;
      base.coef[it][2] = e.c;
    }
    std::vector<int32_t> idx;
    for (int cl : {8, 4, 2, 1, 0}) {
      const size_t first = idx.size();
      size_t smem = 0;
      double units = 0;
      for (int mi = 0; mi < n_narrow; ++mi) {
        const MuonMat& M = mats[mi];
        if (narrow_cluster_for(M.s, M.l) != cl) continue;
        idx.push_back(mi);
        if (cl > 0) smem = std::max(smem, narrow_resident_smem(M.s, M.l, cl));
        const double sd = M.s, ld = M.l;
        units += (double)c.ns_steps * (sd * (sd + 1) * ld + sd * (sd + 1) * sd + 2 * sd * sd * ld);
      }
      if (idx.size() == first) continue;
      NarrowLaunch nl = base;
      nl.idx = h->d_narrow_idx + first;
      nl.nmat = (int)(idx.size() - first);
      nl.cluster = cl;
      h->narrow.push_back(nl);
      h->narrow_smem.push_back(smem);
      h->narrow_units.push_back(units);
    }
    CUDA_TRY(cudaMemcpy(h->d_narrow_idx, idx.data(), idx.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
    // the resident kernel's shared-memory ceiling at the largest any plan uses:
    // the attribute is per device, and another handle's plan may need more
    // than this one's (it allows, and reserves nothing)
    CUDA_TRY(ns_narrow_prepare(kNarrowMaxSmem, &h->narrow_per_sm));
  }
  h->small.clear();
  for (Bucket& B : h->buckets) {
    if (!B.fused) continue;
    SmallLaunch sl;
    memset(&sl, 0, sizeof sl);
    char eb[256];
    if (!tc_encode_small(sl, B.X0, (int)B.params.size(), B.L, eb, sizeof eb)) return fail(MA_ERR_CUDA, "%s", eb);
    sl.mats = h->d_mats + B.mat0;
    sl.rscale = h->d_rscale + B.mat0;
    sl.sp = h->d_step;
    sl.err = h->d_err;
    sl.nmat = (int)B.params.size();
    sl.L = B.L;
    sl.steps = c.ns_steps;
    for (int it = 0; it < c.ns_steps; ++it) {
      NsEpiArgs e{};
      set_epi_coefficients(e, c, it);
      sl.coef[it][0] = e.a;
      sl.coef[it][1] = e.b;
      sl.coef[it][2] = e.c;
    }
    h->small.push_back(sl);
  }
  if (c.ns_kernel == MA_NS_TCGEN05 && !h->buckets.empty()) {
    CUDA_TRY(ns_tc_prepare(&h->max_pairs));
    if (h->max_pairs < 1) h->max_pairs = 1;
    // each launch's work order, for the clusters that can be resident at once
    std::vector<int32_t> all, one;
    std::vector<size_t> at;
    for (int kind = 0; kind < 3; ++kind)
      for (int it = 0; it < steps; ++it)
        for (TcLaunch& L : h->tc[kind][it]) {
          const int ncl = std::min(L.cl == 2 ? h->max_pairs : h->num_sms, L.total_tiles);
          tc_unit_order(L, ncl, one);
          L.nclusters = ncl;
          // the plain round-robin order needs no table (position = unit)
          bool plain = true;
          for (size_t i = 0; i < one.size() && plain; ++i)
            plain = one[i] == ((int64_t)i < L.total_tiles ? (int32_t)i : -1);
          if (plain) {
            L.npos = L.total_tiles;
            at.push_back(SIZE_MAX);
          } else {
            L.npos = (int32_t)one.size();
            at.push_back(all.size());
            all.insert(all.end(), one.begin(), one.end());
          }
        }
    if (h->d_orders) cudaFree(h->d_orders);
    h->d_orders = nullptr;
    if (!all.empty()) {
      CUDA_TRY(cudaMalloc(&h->d_orders, all.size() * sizeof(int32_t)));
      CUDA_TRY(cudaMemcpy(h->d_orders, all.data(), all.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
    }
    size_t li = 0;
    for (int kind = 0; kind < 3; ++kind)
      for (int it = 0; it < steps; ++it)
        for (TcLaunch& L : h->tc[kind][it]) {
          const size_t a = at[li++];
          L.order = a == SIZE_MAX ? nullptr : h->d_orders + a;
        }
  }
  h->planned = true;
  return MA_OK;
}

// Coefficients of Newton-Schulz iteration `it` (the schedule's, if one is set).
void set_epi_coefficients(NsEpiArgs& e, const muon_adamw_config& c, int it) {
  const bool sched = c.ns_schedule_len > 0;
  e.a = (float)(sched ? c.ns_schedule[it][0] : c.ns_a);
  e.b = (float)(sched ? c.ns_schedule[it][1] : c.ns_b);
  e.c = (float)(sched ? c.ns_schedule[it][2] : c.ns_c);
}



ma_status valid_config(const muon_adamw_config* c) {
  if (c->mode != MA_MODE_MUON_ADAMW && c->mode != MA_MODE_ADAMW_ONLY) return fail(MA_ERR_ARG, "bad mode %d", c->mode);
  if (c->precision != MA_BF16_MIXED && c->precision != MA_FP32_MIXED)
    return fail(MA_ERR_ARG, "bad precision %d", c->precision);
  if (c->ns_steps < 1 || c->ns_steps > 64) return fail(MA_ERR_ARG, "ns_steps must be in [1, 64]");
  if (c->ns_kernel != MA_NS_TCGEN05 && c->ns_kernel != MA_NS_SIMT) return fail(MA_ERR_ARG, "bad ns_kernel");
  if (c->muon_momentum_form != MA_MOMENTUM_SGD && c->muon_momentum_form != MA_MOMENTUM_EMA)
    return fail(MA_ERR_ARG, "bad muon_momentum_form %d", c->muon_momentum_form);
  if (c->adam_decay_exempt_bias_norm != 0 && c->adam_decay_exempt_bias_norm != 1)
    return fail(MA_ERR_ARG, "adam_decay_exempt_bias_norm must be 0 or 1");
  if (c->ns_schedule_len != 0) {
    if (c->ns_schedule_len != c->ns_steps || c->ns_schedule_len > MA_NS_SCHEDULE_MAX)
      return fail(MA_ERR_ARG, "ns_schedule_len must be 0 or equal ns_steps (<= %d)", MA_NS_SCHEDULE_MAX);
    for (int i = 0; i < c->ns_schedule_len; ++i)
      for (int k = 0; k < 3; ++k)
        if (!isfinite(c->ns_schedule[i][k])) return fail(MA_ERR_ARG, "non-finite ns_schedule entry");
  }
  if (c->reserved[0] & ~14) return fail(MA_ERR_ARG, "unknown cross-check bits in reserved[0]");
  for (int i = 1; i < 4; ++i)
    if (c->reserved[i] != 0) return fail(MA_ERR_ARG, "reserved[%d] must be 0", i);
  if (!(c->adam_beta1 >= 0.0 && c->adam_beta1 < 1.0) || !(c->adam_beta2 >= 0.0 && c->adam_beta2 < 1.0))
    return fail(MA_ERR_ARG, "betas must lie in [0, 1)");
  if (!(c->adam_eps >= 0.0) || !(c->ns_eps >= 0.0) || !(c->clip_eps >= 0.0)) return fail(MA_ERR_ARG, "eps < 0");
  if (!isfinite(c->muon_momentum) || !isfinite(c->max_grad_norm) || !isfinite(c->muon_lr_scale) ||
      !isfinite(c->moonlight_coef) || !isfinite(c->ns_a) || !isfinite(c->ns_b) || !isfinite(c->ns_c))
    return fail(MA_ERR_ARG, "non-finite config value");
  return MA_OK;
}

}  // namespace

// The scalars of one step (lr and step count dependent), formed in double and
// rounded once, as the kernels use them.
static void fill_step_params(muon_adamw* h, double lr, StepParams* sp) {
  const muon_adamw_config& c = h->cfg;
  const double t = (double)h->t;
  const double bc1 = 1.0 - pow(c.adam_beta1, t), bc2 = 1.0 - pow(c.adam_beta2, t);
  memset(sp, 0, sizeof *sp);
  for (int g = 0; g < kMaxOptionGroups; ++g) {
    const double ls = g < (int)h->option_groups.size() ? h->option_groups[g].first : 1.0;
    const double ws = g < (int)h->option_groups.size() ? h->option_groups[g].second : 1.0;
    sp->adam_decay[g] = (float)(1.0 - lr * ls * c.adam_weight_decay * ws);
    sp->adam_step[g] = (float)(lr * ls / bc1);
    sp->ns_decay[g] = (float)(1.0 - lr * ls * c.muon_weight_decay * ws);
  }
  sp->adam_inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
  sp->ns_lr = (float)lr;
}

// The gradient-norm pass on s0: per-block partial sums of squares over the
// gradients this rank owns (every trainable gradient unless sharded).
static ma_status enqueue_norm_pass(muon_adamw* h) {
  if (h->n_norm_chunks > 0) {
    timed(h, MA_K_GRAD_NORM, h->s0, h->bytes_norm,
          [&] { launch_grad_sumsq(h->d_norm_chunks, h->n_norm_chunks, h->d_norm_partials, h->norm_grid, h->s0); });
  } else {
    CUDA_TRY(cudaMemsetAsync(h->d_norm_partials, 0, sizeof(float), h->s0));
  }
  return MA_OK;
}

static int norm_partials(const muon_adamw* h) { return h->n_norm_chunks > 0 ? h->norm_grid : 1; }

// The launches of one step that read gradients after the norm and clip: AdamW
// forked onto s1; the momentum pass on s0. Each stream then records its
// grads-consumed event. The per-step scalars are read from h->d_step.
static ma_status enqueue_update_passes(muon_adamw* h) {
  const muon_adamw_config& c = h->cfg;
  const bool have_adam = h->n_adam_chunks > 0;
  if (have_adam) {
    CUDA_TRY(cudaEventRecord(h->ev_fork, h->s0));
    CUDA_TRY(cudaStreamWaitEvent(h->s1, h->ev_fork, 0));
    AdamArgs a;
    a.beta1 = (float)c.adam_beta1;
    a.beta2 = (float)c.adam_beta2;
    a.omb1 = (float)(1.0 - c.adam_beta1);
    a.omb2 = (float)(1.0 - c.adam_beta2);
    a.eps = (float)c.adam_eps;
    a.sp = h->d_step;
    timed(h, MA_K_ADAMW, h->s1, h->bytes_adam,
          [&] { launch_adamw(h->d_adam_chunks, h->n_adam_chunks, h->d_scalars, a, h->adam_grid, h->s1); });
    CUDA_TRY(cudaEventRecord(h->ev_g1, h->s1));
  }
  h->g1_valid = have_adam;
  if (h->n_mats > 0) {
    MomArgs ma_{(float)c.muon_momentum, c.muon_nesterov,
                c.muon_momentum_form == MA_MOMENTUM_EMA ? (float)(1.0 - c.muon_momentum) : 1.0f};
    timed(h, MA_K_MOMENTUM, h->s0, h->bytes_mom, [&] {
      launch_muon_momentum(h->d_tiles, h->n_tiles, h->d_mats, h->d_scalars, ma_, h->d_tile_partials, h->mom_grid,
                           h->s0);
    });
  }
  CUDA_TRY(cudaEventRecord(h->ev_g0, h->s0));  // the last kernel on s0 that reads gradients is done
  return MA_OK;
}

// The Newton-Schulz part of a step on s0: the Frobenius scales, then every
// product of every iteration. It reads no gradient and nothing that changes
// from step to step except h->d_step, so it can be captured once.
static ma_status enqueue_newton_schulz(muon_adamw* h) {
  const muon_adamw_config& c = h->cfg;
  if (h->n_mats == 0) return MA_OK;
  timed(h, MA_K_NS_PREP, h->s0, (double)h->n_tiles * 4,
        [&] { launch_ns_prep(h->d_mats, h->n_mats, h->d_tile_partials, (float)c.ns_eps, h->d_rscale, h->s0); });
  // narrow matrices: fp32 Newton-Schulz on the CUDA cores
  for (size_t i = 0; i < h->narrow.size(); ++i)
    CUDA_TRY(timed(h, MA_K_NS_NARROW, h->s0, h->narrow_units[i], [&] {
      return launch_ns_narrow(h->narrow[i], h->narrow_smem[i], h->num_sms, h->narrow_per_sm, h->s0);
    }));
  // buckets of small matrices: every iteration and the update in one launch each
  for (size_t i = 0; i < h->small.size(); ++i) {
    SmallLaunch& sl = h->small[i];
    sl.stall_test = h->stall_test ? 1 : 0;
    h->stall_test = false;  // one launch only
    CUDA_TRY(timed(h, MA_K_NS_FUSED, h->s0, h->small_units[i], [&] { return launch_ns_small(sl, h->num_sms, h->s0); }));
  }
  NsEpiArgs epi;
  epi.sp = h->d_step;
  const double units[3] = {h->unit_gram, h->unit_poly, h->unit_update};
  for (int it = 0; it < c.ns_steps; ++it) {
    set_epi_coefficients(epi, c, it);
    for (int kind = 0; kind < 3; ++kind) {
      if (c.ns_kernel == MA_NS_TCGEN05) {
        for (TcLaunch& L : h->tc[kind][it]) {
          L.epi = epi;
          L.stall_test = h->stall_test ? 1 : 0;
          h->stall_test = false;  // one launch only
          const int pk = (kind == NS_UPDATE && it == c.ns_steps - 1) ? MA_K_NS_APPLY : MA_K_NS_GRAM + kind;
          CUDA_TRY(timed(h, pk, h->s0, units[kind] / h->tc[kind][it].size(), [&] { return launch_ns_tc(L, h->s0); }));
        }
      } else {
        const int pk = (kind == NS_UPDATE && it == c.ns_steps - 1) ? MA_K_NS_APPLY : MA_K_NS_GRAM + kind;
        timed(h, pk, h->s0, units[kind], [&] {
          for (const NsProblem& p : h->simt[kind][it]) launch_ns_simt(p, epi, h->s0);
        });
      }
    }
  }
  return MA_OK;
}

// Capture the Newton-Schulz part as a CUDA graph (the plan's pointers and
// launch shapes never change after the first step, and the step's scalars are
// read from HBM). Any failure leaves the handle on direct launches.
static void capture_newton_schulz_graph(muon_adamw* h) {
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(h->s0, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    h->graph_broken = true;
    return;
  }
  const bool good = enqueue_newton_schulz(h) == MA_OK;
  const cudaError_t e = cudaStreamEndCapture(h->s0, &g);
  if (!good || e != cudaSuccess || !g || cudaGraphInstantiate(&h->gexec, g, 0) != cudaSuccess) {
    h->gexec = nullptr;
    h->graph_broken = true;
  }
  if (g) cudaGraphDestroy(g);
  cudaGetLastError();  // a failed capture leaves no sticky error behind
  clear_last_error();
}

extern "C" {

void muon_adamw_config_init(muon_adamw_config* cfg) {
  if (!cfg) return;
  memset(cfg, 0, sizeof *cfg);
  cfg->mode = MA_MODE_MUON_ADAMW;
  cfg->precision = MA_BF16_MIXED;
  cfg->muon_momentum = 0.95;
  cfg->muon_nesterov = 1;
  cfg->ns_steps = 5;
  cfg->ns_a = 3.4445;
  cfg->ns_b = -4.7750;
  cfg->ns_c = 2.0315;
  cfg->ns_eps = 1e-7;
  cfg->moonlight_coef = 0.2;
  cfg->muon_lr_scale = 1.0;
  cfg->muon_weight_decay = 0.1;
  cfg->adam_beta1 = 0.9;
  cfg->adam_beta2 = 0.999;
  cfg->adam_eps = 1e-8;
  cfg->adam_weight_decay = 0.1;
  cfg->max_grad_norm = 1.0;
  cfg->clip_eps = 1e-6;
  cfg->ns_kernel = MA_NS_TCGEN05;
}

int muon_adamw_is_muon_param(const char* name, int ndim) { return route_is_muon(name, ndim) ? 1 : 0; }

double muon_adamw_cosine_with_min_lr(int64_t step, int64_t total, int64_t warmup, double min_lr_rate) {
  if (step < warmup) return (double)step / (double)std::max<int64_t>(1, warmup);
  const double progress = (double)(step - warmup) / (double)std::max<int64_t>(1, total - warmup);
  const double cosine = 0.5 * (1.0 + cos(M_PI * progress));
  const double f = cosine * (1.0 - min_lr_rate) + min_lr_rate;
  return f > 0.0 ? f : 0.0;
}

const char* muon_adamw_last_error(void) { return g_last_error.c_str(); }

const char* muon_adamw_version(void) { return "0.1.0 sm_103a"; }

ma_status muon_adamw_create(const muon_adamw_config* cfg, void* cuda_stream, muon_adamw_t** out) {
  if (!cfg || !out) return fail(MA_ERR_ARG, "cfg and out must not be NULL");
  *out = nullptr;
  ma_status st = valid_config(cfg);
  if (st != MA_OK) return st;
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(MA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, prop.major,
                prop.minor);
  muon_adamw* h = new (std::nothrow) muon_adamw();
  if (!h) return fail(MA_ERR_OOM, "host allocation failed");
  h->cfg = *cfg;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->s0 = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaStreamCreateWithFlags(&h->s1, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->s2, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_g0, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_g1, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_slot[0], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_slot[1], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaHostAlloc(&h->h_step, 2 * sizeof(StepParams), cudaHostAllocDefault);
  if (e != cudaSuccess) {
    muon_adamw_destroy(h);
    return fail(MA_ERR_CUDA, "stream/event creation failed: %s", cudaGetErrorString(e));
  }
  *out = h;
  return ok();
}

ma_status muon_adamw_register_param(muon_adamw_t* h, const char* name, int ndim, const int64_t* shape,
                                    float* param_fp32, const void* grad, int grad_dtype, void* param_bf16_shadow,
                                    int group_override, int* assigned, int* index_out) {
  if (!h || !name) return fail(MA_ERR_ARG, "handle and name must not be NULL");
  if (h->planned) return fail(MA_ERR_STATE, "register_param after the first step (plan is frozen)");
  if (ndim < 0 || ndim > 8) return fail(MA_ERR_SHAPE, "ndim %d outside [0, 8]", ndim);
  if (ndim > 0 && !shape) return fail(MA_ERR_ARG, "shape must not be NULL for ndim > 0");
  Param p;
  p.name = name;
  p.numel = 1;
  for (int d = 0; d < ndim; ++d) {
    if (shape[d] < 0) return fail(MA_ERR_SHAPE, "negative size in dim %d", d);
    if (shape[d] > ((int64_t)1 << 40)) return fail(MA_ERR_SHAPE, "size too large in dim %d", d);
    p.shape.push_back(shape[d]);
    p.numel *= shape[d];
  }
  int group;
  switch (group_override) {
    case MA_GROUP_AUTO:
      group = (h->cfg.mode == MA_MODE_MUON_ADAMW && route_is_muon(name, ndim)) ? MA_GROUP_MUON : MA_GROUP_ADAMW;
      break;
    case MA_GROUP_MUON:
    case MA_GROUP_ADAMW:
    case MA_GROUP_FROZEN:
      group = group_override;
      break;
    default:
      return fail(MA_ERR_ARG, "bad group override %d", group_override);
  }
  if (group == MA_GROUP_MUON) {
    if (ndim != 2) return fail(MA_ERR_SHAPE, "Muon parameters must be 2-D (got ndim %d)", ndim);
    if (p.shape[0] >= ((int64_t)1 << 30) || p.shape[1] >= ((int64_t)1 << 30))
      return fail(MA_ERR_SHAPE, "Muon matrix dimension too large");
  }
  if (group != MA_GROUP_FROZEN && p.numel > 0) {
    if (!param_fp32 || !grad) return fail(MA_ERR_ARG, "param and grad must not be NULL for trainable '%s'", name);
    if (grad_dtype != MA_DT_F32 && grad_dtype != MA_DT_BF16) return fail(MA_ERR_DTYPE, "bad grad dtype %d", grad_dtype);
    if (reinterpret_cast<uintptr_t>(param_fp32) % 4) return fail(MA_ERR_ALIGN, "param not 4-byte aligned");
    if (reinterpret_cast<uintptr_t>(grad) % (grad_dtype == MA_DT_BF16 ? 2 : 4))
      return fail(MA_ERR_ALIGN, "grad not aligned to its element size");
    if (reinterpret_cast<uintptr_t>(param_bf16_shadow) % 2) return fail(MA_ERR_ALIGN, "shadow not 2-byte aligned");
  }
  p.p = param_fp32;
  p.g = grad;
  p.gdtype = grad_dtype;
  p.shadow = (h->cfg.precision == MA_BF16_MIXED) ? static_cast<uint16_t*>(param_bf16_shadow) : nullptr;
  p.group = group;
  h->params.push_back(p);
  if (assigned) *assigned = group;
  if (index_out) *index_out = (int)h->params.size() - 1;
  return ok();
}

// Start a step: freeze the plan at the first one, advance t and queue the
// copy of the step's lr- and t-dependent scalars.
static ma_status begin_step(muon_adamw* h, double lr) {
  CUDA_TRY(cudaSetDevice(h->device));
  if (!h->planned) {
    ma_status st = build_plan(h);
    if (st != MA_OK) return st;
  }
  h->t += 1;
  // the step's scalars go through one of two pinned slots; the slot's
  // previous copy (two steps ago) has been read before it is rewritten
  const int slot = (int)(h->t & 1);
  CUDA_TRY(cudaEventSynchronize(h->ev_slot[slot]));
  fill_step_params(h, lr, &h->h_step[slot]);
  CUDA_TRY(cudaMemcpyAsync(h->d_step, &h->h_step[slot], sizeof(StepParams), cudaMemcpyHostToDevice, h->s0));
  CUDA_TRY(cudaEventRecord(h->ev_slot[slot], h->s0));
  return MA_OK;
}

// Finish a step once the clip coefficient is in h->d_scalars: the update
// passes, the Newton-Schulz chain (one graph launch, or its launches one by
// one) and the join of the AdamW stream, before the chain or after it; with
// grad_norm_out, wait and read.
static ma_status finish_step(muon_adamw* h, float* grad_norm_out) {
  const muon_adamw_config& c = h->cfg;
  ma_status st = enqueue_update_passes(h);
  if (st != MA_OK) return st;
  // Where AdamW moves more bytes than the momentum pass, the chain starts
  // once AdamW is done: its long-running blocks hold every SM until they run
  // out of work, so a chain launched earlier would only wait for them inside
  // its first launch. Where AdamW is the smaller stream, its blocks retire
  // one by one and the chain's first CTAs take their SMs as they do, so the
  // join comes at the end of the step instead.
  const bool join_first = h->g1_valid && h->bytes_adam > h->bytes_mom;
  if (join_first) CUDA_TRY(cudaStreamWaitEvent(h->s0, h->ev_g1, 0));
  const bool graph = h->graph_mode && !h->graph_broken && !h->profiling && !h->stall_test &&
                     c.ns_kernel == MA_NS_TCGEN05 && h->n_mats > 0;
  if (graph && !h->gexec) capture_newton_schulz_graph(h);
  if (graph && h->gexec) {
    CUDA_TRY(cudaGraphLaunch(h->gexec, h->s0));
  } else {
    st = enqueue_newton_schulz(h);
    if (st != MA_OK) return st;
  }
  if (h->g1_valid && !join_first) CUDA_TRY(cudaStreamWaitEvent(h->s0, h->ev_g1, 0));
  CUDA_TRY(cudaGetLastError());
  if (h->profiling) h->prof.steps += 1;
  if (grad_norm_out) {
    StepScalars sc;
    CUDA_TRY(cudaMemcpyAsync(&sc, h->d_scalars, sizeof sc, cudaMemcpyDeviceToHost, h->s0));
    CUDA_TRY(cudaStreamSynchronize(h->s0));
    *grad_norm_out = sc.total;
    st = check_device_flag(h);
    if (st != MA_OK) return st;
  }
  return ok();
}

ma_status muon_adamw_step(muon_adamw_t* h, double lr, float* grad_norm_out) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (!isfinite(lr)) return fail(MA_ERR_ARG, "lr is not finite");
  if (h->shard_world > 1)
    return fail(MA_ERR_STATE, "a sharded handle steps with muon_adamw_step_begin / muon_adamw_step_end");
  ma_status st = begin_step(h, lr);
  if (st != MA_OK) return st;
  const muon_adamw_config& c = h->cfg;
  st = enqueue_norm_pass(h);
  if (st != MA_OK) return st;
  timed(h, MA_K_CLIP, h->s0, (double)h->norm_grid * 4, [&] {
    launch_clip_finalize(h->d_norm_partials, norm_partials(h), (float)c.max_grad_norm, (float)c.clip_eps,
                         h->d_scalars, h->s0);
  });
  return finish_step(h, grad_norm_out);
}

ma_status muon_adamw_step_begin(muon_adamw_t* h, double lr, double* local_sumsq) {
  if (!h || !local_sumsq) return fail(MA_ERR_ARG, "NULL handle or local_sumsq");
  if (!isfinite(lr)) return fail(MA_ERR_ARG, "lr is not finite");
  if (h->begun) return fail(MA_ERR_STATE, "step_begin twice without step_end");
  if (reinterpret_cast<uintptr_t>(local_sumsq) % 8) return fail(MA_ERR_ALIGN, "local_sumsq not 8-byte aligned");
  ma_status st = begin_step(h, lr);
  if (st != MA_OK) return st;
  st = enqueue_norm_pass(h);
  if (st != MA_OK) return st;
  timed(h, MA_K_CLIP, h->s0, (double)h->norm_grid * 4,
        [&] { launch_sumsq_partials(h->d_norm_partials, norm_partials(h), local_sumsq, h->s0); });
  CUDA_TRY(cudaGetLastError());
  h->begun = true;
  return ok();
}

ma_status muon_adamw_step_end(muon_adamw_t* h, const double* global_sumsq, float* grad_norm_out) {
  if (!h || !global_sumsq) return fail(MA_ERR_ARG, "NULL handle or global_sumsq");
  if (!h->begun) return fail(MA_ERR_STATE, "step_end without step_begin");
  if (reinterpret_cast<uintptr_t>(global_sumsq) % 8) return fail(MA_ERR_ALIGN, "global_sumsq not 8-byte aligned");
  h->begun = false;
  CUDA_TRY(cudaSetDevice(h->device));
  const muon_adamw_config& c = h->cfg;
  timed(h, MA_K_CLIP, h->s0, 8.0, [&] {
    launch_clip_from_sumsq(global_sumsq, (float)c.max_grad_norm, (float)c.clip_eps, h->d_scalars, h->s0);
  });
  return finish_step(h, grad_norm_out);
}

ma_status muon_adamw_set_shard(muon_adamw_t* h, int rank, int world) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (world < 1 || world > MA_SHARD_MAX_WORLD || rank < 0 || rank >= world)
    return fail(MA_ERR_ARG, "rank %d of world %d: need 0 <= rank < world <= %d", rank, world, MA_SHARD_MAX_WORLD);
  if (h->planned) return fail(MA_ERR_STATE, "set_shard after the first step (plan is frozen)");
  h->shard_rank = rank;
  h->shard_world = world;
  return ok();
}

ma_status muon_adamw_shard_range(muon_adamw_t* h, int index, int rank, int64_t* begin, int64_t* end) {
  if (!h || !begin || !end) return fail(MA_ERR_ARG, "NULL argument");
  if (index < 0 || index >= (int)h->params.size()) return fail(MA_ERR_ARG, "bad parameter index %d", index);
  if (rank < 0 || rank >= h->shard_world) return fail(MA_ERR_ARG, "rank %d outside world %d", rank, h->shard_world);
  const Param& q = h->params[index];
  if (h->shard_world == 1) {
    *begin = 0;
    *end = q.group == MA_GROUP_FROZEN ? 0 : q.numel;
    return ok();
  }
  const size_t n = h->params.size();
  std::vector<int> group(n), owner;
  std::vector<int64_t> numel(n), rows(n), cols(n), b, e;
  for (size_t i = 0; i < n; ++i) {
    const Param& p = h->params[i];
    group[i] = p.group;
    numel[i] = p.numel;
    rows[i] = p.shape.size() == 2 ? p.shape[0] : p.numel;
    cols[i] = p.shape.size() == 2 ? p.shape[1] : 1;
  }
  shard_partition(group, numel, rows, cols, h->shard_world, owner, b, e);
  *begin = b[(size_t)index * (size_t)h->shard_world + (size_t)rank];
  *end = e[(size_t)index * (size_t)h->shard_world + (size_t)rank];
  return ok();
}

ma_status muon_adamw_plan_shards(int n_params, const int32_t* groups, const int64_t* numels, const int64_t* rows,
                                 const int64_t* cols, int world, int32_t* owner_out, int64_t* begin_out,
                                 int64_t* end_out) {
  if (n_params < 0 || (n_params > 0 && (!groups || !numels || !rows || !cols || !owner_out || !begin_out || !end_out)))
    return fail(MA_ERR_ARG, "NULL pointer or negative n_params");
  if (world < 1 || world > MA_SHARD_MAX_WORLD) return fail(MA_ERR_ARG, "world must be 1..%d", MA_SHARD_MAX_WORLD);
  std::vector<int> group((size_t)n_params), owner;
  std::vector<int64_t> numel((size_t)n_params), r((size_t)n_params), cl((size_t)n_params), b, e;
  for (int i = 0; i < n_params; ++i) {
    if (groups[i] != MA_GROUP_MUON && groups[i] != MA_GROUP_ADAMW && groups[i] != MA_GROUP_FROZEN)
      return fail(MA_ERR_ARG, "groups[%d] must be MUON, ADAMW or FROZEN", i);
    if (numels[i] < 0 || rows[i] < 0 || cols[i] < 0) return fail(MA_ERR_SHAPE, "negative size for parameter %d", i);
    if (groups[i] == MA_GROUP_MUON && rows[i] * cols[i] != numels[i])
      return fail(MA_ERR_SHAPE, "Muon parameter %d: rows x cols != numel", i);
    group[(size_t)i] = groups[i];
    numel[(size_t)i] = numels[i];
    r[(size_t)i] = rows[i];
    cl[(size_t)i] = cols[i];
  }
  shard_partition(group, numel, r, cl, world, owner, b, e);
  for (int i = 0; i < n_params; ++i) owner_out[i] = owner[(size_t)i];
  if (!b.empty()) {
    memcpy(begin_out, b.data(), b.size() * sizeof(int64_t));
    memcpy(end_out, e.data(), e.size() * sizeof(int64_t));
  }
  return ok();
}

ma_status muon_adamw_set_graph_mode(muon_adamw_t* h, int enable) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  h->graph_mode = enable != 0;
  return ok();
}

ma_status muon_adamw_record_grads_consumed(muon_adamw_t* h, void* cuda_event) {
  if (!h || !cuda_event) return fail(MA_ERR_ARG, "NULL handle or event");
  if (!h->planned || h->t == 0) return fail(MA_ERR_STATE, "no step taken yet");
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamWaitEvent(h->s2, h->ev_g0, 0));
  if (h->g1_valid) CUDA_TRY(cudaStreamWaitEvent(h->s2, h->ev_g1, 0));
  CUDA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(cuda_event), h->s2));
  return ok();
}

ma_status muon_adamw_set_param_options(muon_adamw_t* h, int index, double lr_scale, double weight_decay_scale) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (index < 0 || index >= (int)h->params.size()) return fail(MA_ERR_ARG, "bad parameter index %d", index);
  if (!(lr_scale >= 0.0) || !isfinite(lr_scale) || !(weight_decay_scale >= 0.0) || !isfinite(weight_decay_scale))
    return fail(MA_ERR_ARG, "scales must be finite and >= 0");
  if (h->planned) return fail(MA_ERR_STATE, "set_param_options after the first step (plan is frozen)");
  Param& p = h->params[index];
  if (p.group == MA_GROUP_FROZEN) return fail(MA_ERR_STATE, "parameter %d is frozen", index);
  // count the distinct explicit pairs with this one (the rule's pairs are checked at the first step)
  std::vector<std::pair<double, double>> seen{{1.0, 1.0}};
  for (size_t i = 0; i < h->params.size(); ++i) {
    const Param& q = h->params[i];
    std::pair<double, double> key;
    if ((int)i == index)
      key = {lr_scale, weight_decay_scale};
    else if (q.options_set && q.group != MA_GROUP_FROZEN)
      key = {q.lr_scale, q.wd_scale};
    else
      continue;
    if (std::find(seen.begin(), seen.end(), key) == seen.end()) seen.push_back(key);
  }
  if ((int)seen.size() > kMaxOptionGroups)
    return fail(MA_ERR_UNSUPPORTED, "more than %d distinct (lr_scale, weight_decay_scale) pairs", kMaxOptionGroups);
  p.lr_scale = lr_scale;
  p.wd_scale = weight_decay_scale;
  p.options_set = true;
  return ok();
}

ma_status muon_adamw_plan_work_order(int nprob, const int64_t* k, const int64_t* units, int nclusters,
                                     int32_t* order, int64_t cap, int64_t* npos) {
  if (!k || !units || !npos || (cap > 0 && !order)) return fail(MA_ERR_ARG, "NULL pointer");
  if (nprob < 1 || nprob > kTcMaxProblems) return fail(MA_ERR_ARG, "nprob must be 1..%d", kTcMaxProblems);
  if (nclusters < 1) return fail(MA_ERR_ARG, "nclusters must be >= 1");
  TcLaunch L;
  memset(&L, 0, sizeof L);
  int64_t total = 0;
  for (int q = 0; q < nprob; ++q) {
    if (k[q] < 64 || k[q] % 64 != 0 || k[q] > INT32_MAX) return fail(MA_ERR_ARG, "k[%d] must be a positive multiple of 64", q);
    if (units[q] < 0 || total + units[q] > INT32_MAX) return fail(MA_ERR_ARG, "bad unit count for problem %d", q);
    L.prob[q].p.K = (int32_t)k[q];
    L.prob[q].p.nmat = 1;
    L.prob[q].tiles_per_mat = (int32_t)units[q];
    L.prob[q].tile_begin = (int32_t)total;
    total += units[q];
  }
  L.nprob = nprob;
  L.total_tiles = (int32_t)total;
  std::vector<int32_t> tab;
  tc_unit_order(L, nclusters, tab);
  *npos = (int64_t)tab.size();
  if ((int64_t)tab.size() > cap) return fail(MA_ERR_SHAPE, "order needs %zu entries, capacity %lld", tab.size(), (long long)cap);
  if (!tab.empty()) memcpy(order, tab.data(), tab.size() * sizeof(int32_t));
  return ok();
}

ma_status muon_adamw_test_arm_stall(muon_adamw_t* h) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (h->cfg.ns_kernel != MA_NS_TCGEN05) return fail(MA_ERR_UNSUPPORTED, "only the tensor-core kernel has waits");
  h->stall_test = true;
  return ok();
}

ma_status muon_adamw_sync(muon_adamw_t* h) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  ma_status st = check_device_flag(h);
  if (st != MA_OK) return st;
  return ok();
}

static ma_status state_ptr(muon_adamw_t* h, int index, int which, float** ptr, int64_t* n) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (index < 0 || index >= (int)h->params.size()) return fail(MA_ERR_ARG, "bad parameter index %d", index);
  const Param& p = h->params[index];
  if (p.group == MA_GROUP_FROZEN) return fail(MA_ERR_STATE, "parameter %d is frozen: no state", index);
  if (which == 0) {
    *ptr = p.st0;
  } else if (which == 1) {
    if (p.group != MA_GROUP_ADAMW) return fail(MA_ERR_ARG, "which=1 (second moment) exists only for AdamW");
    *ptr = p.st1;
  } else {
    return fail(MA_ERR_ARG, "bad which %d", which);
  }
  if (p.numel > 0 && p.own_e <= p.own_b)
    return fail(MA_ERR_STATE, "parameter %d is not updated by this rank (sharded step)", index);
  *n = p.own_e - p.own_b;  // the whole parameter, or this rank's range of an AdamW parameter
  return MA_OK;
}

ma_status muon_adamw_get_state(muon_adamw_t* h, int index, int which, float* dst_host) {
  if (h && !h->planned) return fail(MA_ERR_STATE, "no state before the first step");
  float* src = nullptr;
  int64_t n = 0;
  ma_status st = state_ptr(h, index, which, &src, &n);
  if (st != MA_OK) return st;
  if (!dst_host && n > 0) return fail(MA_ERR_ARG, "dst must not be NULL");
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  if (n > 0) CUDA_TRY(cudaMemcpy(dst_host, src, n * sizeof(float), cudaMemcpyDeviceToHost));
  return ok();
}

ma_status muon_adamw_set_state(muon_adamw_t* h, int index, int which, const float* src_host) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  CUDA_TRY(cudaSetDevice(h->device));
  if (!h->planned) {
    ma_status st = build_plan(h);
    if (st != MA_OK) return st;
  }
  float* dst = nullptr;
  int64_t n = 0;
  ma_status st = state_ptr(h, index, which, &dst, &n);
  if (st != MA_OK) return st;
  if (!src_host && n > 0) return fail(MA_ERR_ARG, "src must not be NULL");
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  if (n > 0) CUDA_TRY(cudaMemcpy(dst, src_host, n * sizeof(float), cudaMemcpyHostToDevice));
  return ok();
}

ma_status muon_adamw_get_step(muon_adamw_t* h, int64_t* t_out) {
  if (!h || !t_out) return fail(MA_ERR_ARG, "NULL argument");
  *t_out = h->t;
  return ok();
}

ma_status muon_adamw_set_step(muon_adamw_t* h, int64_t t) {
  if (!h || t < 0) return fail(MA_ERR_ARG, "NULL handle or negative step");
  h->t = t;
  return ok();
}

ma_status muon_adamw_last_norm(muon_adamw_t* h, float* total_out, float* coef_out) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  if (!h->planned) return fail(MA_ERR_STATE, "no step taken yet");
  CUDA_TRY(cudaSetDevice(h->device));
  StepScalars sc;
  CUDA_TRY(cudaMemcpyAsync(&sc, h->d_scalars, sizeof sc, cudaMemcpyDeviceToHost, h->s0));
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  if (total_out) *total_out = sc.total;
  if (coef_out) *coef_out = sc.coef;
  ma_status st = check_device_flag(h);
  if (st != MA_OK) return st;
  return ok();
}

ma_status muon_adamw_plan_info(muon_adamw_t* h, ma_plan_info* out) {
  if (!h || !out) return fail(MA_ERR_ARG, "NULL argument");
  if (!h->planned) return fail(MA_ERR_STATE, "plan is built by the first step");
  memset(out, 0, sizeof *out);
  out->n_params = (int)h->params.size();
  for (const Param& p : h->params) {
    if (p.group == MA_GROUP_MUON) out->n_muon++;
    if (p.group == MA_GROUP_ADAMW) out->n_adamw++;
    if (p.group == MA_GROUP_FROZEN) out->n_frozen++;
  }
  out->n_buckets = (int)h->buckets.size();
  out->muon_elems = h->muon_elems;
  out->adamw_elems = h->adam_elems;
  out->grad_elems = h->grad_elems;
  out->state_bytes = (int64_t)h->state_bytes;
  out->workspace_bytes = (int64_t)h->workspace_bytes;
  out->ns_flops_per_step =
      h->cfg.ns_steps * (h->unit_gram + h->unit_poly + h->unit_update) + h->unit_fused + h->unit_narrow;
  out->ns_dense_flops_per_step = h->dense_flops;
  out->stream_bytes_per_step = h->bytes_norm + h->bytes_mom + h->bytes_adam;
  return ok();
}

ma_status muon_adamw_set_profiling(muon_adamw_t* h, int enable) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  h->profiling = enable != 0;
  return ok();
}

ma_status muon_adamw_get_profile(muon_adamw_t* h, ma_profile* out) {
  if (!h || !out) return fail(MA_ERR_ARG, "NULL argument");
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  CUDA_TRY(cudaStreamSynchronize(h->s1));
  ma_status st = fold_profile(h);
  if (st != MA_OK) return st;
  *out = h->prof;
  return ok();
}

ma_status muon_adamw_reset_profile(muon_adamw_t* h) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamSynchronize(h->s0));
  CUDA_TRY(cudaStreamSynchronize(h->s1));
  ma_status st = fold_profile(h);
  if (st != MA_OK) return st;
  memset(&h->prof, 0, sizeof h->prof);
  return ok();
}

ma_status muon_adamw_destroy(muon_adamw_t* h) {
  if (!h) return fail(MA_ERR_ARG, "NULL handle");
  cudaSetDevice(h->device);
  if (h->s0 || h->s1) {
    cudaStreamSynchronize(h->s0);
    if (h->s1) cudaStreamSynchronize(h->s1);
  }
  for (const ProfRec& r : h->prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  if (h->arena) cudaFree(h->arena);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_g0) cudaEventDestroy(h->ev_g0);
  if (h->ev_g1) cudaEventDestroy(h->ev_g1);
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->d_orders) cudaFree(h->d_orders);
  for (int k = 0; k < 2; ++k)
    if (h->ev_slot[k]) cudaEventDestroy(h->ev_slot[k]);
  if (h->h_step) cudaFreeHost(h->h_step);
  if (h->s1) cudaStreamDestroy(h->s1);
  if (h->s2) cudaStreamDestroy(h->s2);
  delete h;
  return ok();
}

}  // extern "C"
