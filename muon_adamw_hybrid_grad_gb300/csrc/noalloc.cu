// Allocation-free global gradient norm and clip coefficient.
//
// Some callers cannot call cudaMalloc: for example a host application that
// hands all device memory to its own pool allocator at start-up and forbids
// later allocations, or a latency-critical loop in which cudaMalloc's
// implicit device-wide synchronisation is unacceptable. For them this file
// offers one entry point, muon_adamw_grad_norm_noalloc(), that computes the
// same global gradient norm and clip coefficient as muon_adamw_step() without
// allocating anything: its only scratch is the file-scope device array below,
// which every GPU that loads this library holds until the process exits.
//
// Limits: at most kNoAllocMaxTensors gradient tensors per call (they travel
// as kernel parameters, so no table has to be copied to the device) and at
// most kNoAllocMaxBlocks partial sums (4 KiB of scratch per device).
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "muon_adamw.h"
#include "internal.h"

// The scratch: one fp32 partial sum of squares per block of the reduction.
// Every call writes all the slots it later reads, so nothing has to be
// cleared between calls; its contents are simply those of the last call.
static __device__ __align__(256) float g_noalloc_partials[MA_NOALLOC_MAX_PARTIALS];

namespace ma {
namespace {

constexpr int kNoAllocMaxTensors = MA_NOALLOC_MAX_TENSORS;
constexpr int kNoAllocMaxBlocks = MA_NOALLOC_MAX_PARTIALS;
constexpr int kNoAllocThreads = 512;
constexpr int kMaxDevices = 64;

struct NoAllocTensors {
  const void* ptr[kNoAllocMaxTensors];
  int64_t numel[kNoAllocMaxTensors];
  int64_t chunk_end[kNoAllocMaxTensors];  // inclusive prefix sum of chunk counts
  int32_t dtype[kNoAllocMaxTensors];
  int32_t n;
  int32_t total_chunks;
};

__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  if (isinf(t)) {  // keep an infinite sum infinite instead of producing inf - inf
    s = t;
    c = 0.f;
    return;
  }
  c = (t - s) - y;
  s = t;
}

// Sum of squares of 8 bf16 values packed in a 16-byte vector.
__device__ __forceinline__ float sumsq_bf16x8(const uint4& w) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  float s8 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xFFFF0000u);
    s8 = fmaf(lo, lo, s8);
    s8 = fmaf(hi, hi, s8);
  }
  return s8;
}

__device__ __forceinline__ float sumsq_f32x4(const float4& w) {
  float s4 = w.x * w.x;
  s4 = fmaf(w.y, w.y, s4);
  s4 = fmaf(w.z, w.z, s4);
  return fmaf(w.w, w.w, s4);
}

// One block per 64 Ki-element chunk (grid-stride). Where a tensor's pointer is
// 16-byte aligned (every chunk of it then is too: a chunk is 128 KiB of bf16
// or 256 KiB of fp32), its elements are read as 16-byte vectors, four in
// flight per thread; the rest of the chunk, and unaligned tensors, element by
// element.
__global__ void __launch_bounds__(kNoAllocThreads) noalloc_sumsq_kernel(const __grid_constant__ NoAllocTensors T,
                                                                        float* __restrict__ partials) {
  __shared__ double sh[kNoAllocThreads / 32];
  float s = 0.f, comp = 0.f;
  int t = 0;
  for (int c = blockIdx.x; c < T.total_chunks; c += gridDim.x) {
    while (c >= T.chunk_end[t]) ++t;  // chunks are visited in increasing order
    const int64_t first = (t == 0) ? 0 : T.chunk_end[t - 1];
    const int64_t begin = (int64_t)(c - first) * kChunk;
    const int64_t end = begin + kChunk < T.numel[t] ? begin + kChunk : T.numel[t];
    const bool vec = (reinterpret_cast<uintptr_t>(T.ptr[t]) & 15) == 0;
    if (T.dtype[t] == MA_DT_BF16) {
      const uint16_t* g = static_cast<const uint16_t*>(T.ptr[t]);
      const int64_t nv = vec ? (end - begin) / 8 : 0;  // vectors of 8 from `begin`
      const uint4* gv = reinterpret_cast<const uint4*>(g + begin);
      int64_t i = threadIdx.x;
      for (; i + 3 * kNoAllocThreads < nv; i += 4 * kNoAllocThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = __ldg(gv + i + u * kNoAllocThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) kahan_add(s, comp, sumsq_bf16x8(w[u]));
      }
      for (; i < nv; i += kNoAllocThreads) kahan_add(s, comp, sumsq_bf16x8(__ldg(gv + i)));
      for (int64_t j = begin + nv * 8 + threadIdx.x; j < end; j += kNoAllocThreads) {
        const float x = __uint_as_float(((uint32_t)g[j]) << 16);
        kahan_add(s, comp, x * x);
      }
    } else {
      const float* g = static_cast<const float*>(T.ptr[t]);
      const int64_t nv = vec ? (end - begin) / 4 : 0;  // vectors of 4 from `begin`
      const float4* gv = reinterpret_cast<const float4*>(g + begin);
      int64_t i = threadIdx.x;
      for (; i + 3 * kNoAllocThreads < nv; i += 4 * kNoAllocThreads) {
        float4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = __ldg(gv + i + u * kNoAllocThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) kahan_add(s, comp, sumsq_f32x4(w[u]));
      }
      for (; i < nv; i += kNoAllocThreads) kahan_add(s, comp, sumsq_f32x4(__ldg(gv + i)));
      for (int64_t j = begin + nv * 4 + threadIdx.x; j < end; j += kNoAllocThreads) {
        const float x = g[j];
        kahan_add(s, comp, x * x);
      }
    }
  }
  double v = (double)s - (double)comp;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    double r = threadIdx.x < kNoAllocThreads / 32 ? sh[threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (threadIdx.x == 0) partials[blockIdx.x] = (float)r;
  }
}

__global__ void __launch_bounds__(32) noalloc_finalize_kernel(const float* __restrict__ partials, int n,
                                                              double max_norm, double clip_eps,
                                                              float* __restrict__ out) {
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += 32) s += (double)partials[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (threadIdx.x == 0) {
    const double total = sqrt(s);
    double coef = 1.0;
    if (isnan(total)) {
      coef = total;
    } else if (max_norm > 0.0) {
      coef = max_norm / (total + clip_eps);
      if (coef > 1.0) coef = 1.0;
    }
    out[0] = (float)total;
    out[1] = (float)coef;
  }
}

// Per-device set-up: the device address of the scratch array and the SM count.
struct DeviceSlot {
  std::atomic<int> ready{0};
  float* partials = nullptr;
  int num_sms = 0;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_setup_mutex;

ma_status noalloc_fail(ma_status st, const char* msg) {
  set_last_error(msg);  // read back with muon_adamw_last_error()
  return st;
}

}  // namespace
}  // namespace ma

using namespace ma;

extern "C" MA_API ma_status muon_adamw_grad_norm_noalloc(const void* const* grads, const int64_t* numels,
                                                         const int32_t* dtypes, int n_tensors, double max_norm,
                                                         double clip_eps, float* out_total_coef, void* cuda_stream) {
  char msg[256];
  if (n_tensors < 0 || n_tensors > kNoAllocMaxTensors) {
    snprintf(msg, sizeof msg, "n_tensors = %d: this entry point takes 0 to %d tensors per call", n_tensors,
             kNoAllocMaxTensors);
    return noalloc_fail(MA_ERR_ARG, msg);
  }
  if (!out_total_coef) return noalloc_fail(MA_ERR_ARG, "out_total_coef must not be NULL");
  if (n_tensors > 0 && (!grads || !numels || !dtypes))
    return noalloc_fail(MA_ERR_ARG, "grads, numels and dtypes must not be NULL");
  if (!(clip_eps >= 0.0) || !isfinite(max_norm)) return noalloc_fail(MA_ERR_ARG, "bad max_norm or clip_eps");
  NoAllocTensors T;
  memset(&T, 0, sizeof T);
  int64_t chunks = 0;
  for (int i = 0; i < n_tensors; ++i) {
    if (numels[i] < 0) return noalloc_fail(MA_ERR_SHAPE, "negative numel");
    if (dtypes[i] != MA_DT_F32 && dtypes[i] != MA_DT_BF16) return noalloc_fail(MA_ERR_DTYPE, "bad dtype");
    if (numels[i] > 0 && !grads[i]) return noalloc_fail(MA_ERR_ARG, "NULL gradient pointer");
    if (reinterpret_cast<uintptr_t>(grads[i]) % (dtypes[i] == MA_DT_BF16 ? 2 : 4))
      return noalloc_fail(MA_ERR_ALIGN, "gradient pointer not aligned to its element size");
    T.ptr[i] = grads[i];
    T.numel[i] = numels[i];
    T.dtype[i] = dtypes[i];
    chunks += (numels[i] + kChunk - 1) / kChunk;
    T.chunk_end[i] = chunks;
  }
  if (chunks > (int64_t)1 << 30) return noalloc_fail(MA_ERR_SHAPE, "too many elements");
  T.n = n_tensors;
  T.total_chunks = (int32_t)chunks;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(MA_ERR_CUDA, "no usable current CUDA device");
  DeviceSlot& slot = g_slots[dev];
  if (!slot.ready.load(std::memory_order_acquire)) {
    // First call on this device: resolve the scratch array's device address
    // (a host-side name of a __device__ array is not a device pointer).
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!slot.ready.load(std::memory_order_relaxed)) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_partials);
      if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        return noalloc_fail(MA_ERR_CUDA, msg);
      }
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        return noalloc_fail(MA_ERR_CUDA, msg);
      }
      slot.partials = static_cast<float*>(p);
      slot.num_sms = sms;
      slot.ready.store(1, std::memory_order_release);
    }
  }
  int grid = 4 * slot.num_sms;
  if (grid > kNoAllocMaxBlocks) grid = kNoAllocMaxBlocks;
  if (grid > T.total_chunks) grid = T.total_chunks;
  if (grid < 1) grid = 1;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  noalloc_sumsq_kernel<<<grid, kNoAllocThreads, 0, st>>>(T, slot.partials);
  noalloc_finalize_kernel<<<1, 32, 0, st>>>(slot.partials, grid, max_norm, clip_eps, out_total_coef);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "kernel launch: %s", cudaGetErrorString(e));
    return noalloc_fail(MA_ERR_CUDA, msg);
  }
  clear_last_error();
  return MA_OK;
}
