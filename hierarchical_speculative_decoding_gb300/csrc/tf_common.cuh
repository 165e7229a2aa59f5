// Shared device helpers for the TriForce decode-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "triforce_attn.h"

namespace tf {

constexpr int kHeadDim = 128;
constexpr int kChunk = 8;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- host side

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

// A kernel's one-time setup, kept per device: function attributes (the
// dynamic shared-memory limit, non-portable cluster sizes) and the occupancy
// they allow apply to the current device only.  get() runs `setup` on the
// first call on each device and keeps its result when positive; a failed
// setup (0) is not kept, so the next call tries again.  Threads that race on
// a first call may each run `setup`; it only sets attributes and queries
// occupancy, so they store the same value, and a thread that reads a stored
// value sees the attributes already set (release/acquire).
class DeviceCache {
 public:
  static constexpr int kSlots = 64;  // device ordinals served
  template <class F>
  int get(F&& setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSlots) return 0;
    int v = vals_[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    v = setup();
    if (v > 0) vals_[dev].store(v, std::memory_order_release);
    return v;
  }

 private:
  std::atomic<int> vals_[kSlots]{};
};

// Resident CTAs per SM for a kernel (at least 1).
inline int occupancy_blocks(const void* fn, int threads, size_t dyn_smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, dyn_smem) != cudaSuccess || n < 1) return 1;
  return n;
}

// Split count that fills whole waves: the largest s <= cap with units * s
// CTAs fitting the resident slots, or one wave's worth rounded down.
inline int wave_splits(int units, int slots, int cap) {
  int s = slots / (units > 0 ? units : 1);
  if (s > cap) s = cap;
  return s < 1 ? 1 : s;
}

// Launch with programmatic dependent launch: the grid may be scheduled while
// the previous kernel on the stream drains, so its on-chip set-up overlaps that
// tail.  Every kernel launched this way calls pdl_wait() before it touches
// global memory that earlier work on the stream writes or reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

inline tf_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TF_OK : TF_ERR_CUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- debug build
// Built with -DTF_DEBUG, every kernel checks the data-dependent indices of its
// global-memory gathers (rows of the cache, chunks of the index, tiles and
// pieces of the tensor-core stream, rows of the packed buffer) against the
// extents of their buffers.  A failed check ORs its bit into a word of this
// translation unit's device memory and skips the access (no trap, no assert);
// tf_debug_status() collects the words of every file.  Release builds compile
// each check to `true`.
constexpr uint32_t kDbgCacheRow = 1u;   // a row outside [0, L) of its unit, or L > Lmax
constexpr uint32_t kDbgIndexRow = 2u;   // a chunk-mean row outside [0, Cmax)
constexpr uint32_t kDbgTile = 4u;       // a tensor-core tile or gathered piece outside its unit's rows
constexpr uint32_t kDbgPacked = 8u;     // a packed row outside the resident buffer

#ifdef TF_DEBUG
static __device__ unsigned int g_tf_dbg;  // one word per translation unit
__device__ __forceinline__ bool dbg_ok(bool ok, uint32_t code) {
  if (!ok) atomicOr(&g_tf_dbg, code);
  return ok;
}
#define TF_DBG_OK(cond, code) ::tf::dbg_ok((cond), (code))
#define TF_DBG_READER(name)                                                         \
  uint32_t name(int clear) {                                                        \
    unsigned int v = 0;                                                             \
    if (cudaMemcpyFromSymbol(&v, g_tf_dbg, sizeof(v)) != cudaSuccess) return ~0u;  \
    if (clear) {                                                                    \
      const unsigned int z = 0;                                                     \
      if (cudaMemcpyToSymbol(g_tf_dbg, &z, sizeof(z)) != cudaSuccess) return ~0u;  \
    }                                                                               \
    return v;                                                                       \
  }
#else
#define TF_DBG_OK(cond, code) (true)
#define TF_DBG_READER(name)
#endif
// Readers of the files whose kernels gather (defined in debug builds only).
uint32_t dbg_read_chunk_means(int clear);
uint32_t dbg_read_gather(int clear);
uint32_t dbg_read_verify(int clear);
uint32_t dbg_read_topk(int clear);
uint32_t dbg_read_draft(int clear);
uint32_t dbg_read_pack(int clear);

// ---------------------------------------------------------------- device side

// Wait until the previous kernel on the stream has completed and its writes are
// visible (a no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int clamp_len(int L, int Lmax) { return L < 0 ? 0 : (L > Lmax ? Lmax : L); }

// Eight bf16 values packed in 16 bytes -> fp32 (exact: bf16 is the fp32 top half).
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xffff0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xffff0000u);
}

// 16-byte read-only load that does not allocate in L1 (KV rows are read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving map of an fp32 score to uint32 (larger float -> larger key).
// -0 is folded onto +0 so equal scores get equal keys.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

// Combine two online-softmax states in the log2 domain: (m, l) and o scaled alike.
__device__ __forceinline__ float merge_scale(float m_self, float m_new) {
  return (m_self == -INFINITY) ? 0.0f : exp2f(m_self - m_new);
}

// Final log-sum-exp merge of split-K partial states, run by one CTA.
// ml: [splits][stride][2] (m, l) and o: [splits][stride][D] in global memory
// (written by other CTAs; read with L1-bypassing loads); scratch: shared
// memory for 2 * splits * rows + rows floats.  out(n, d) receives
// sum_s e^{m_s - m} o_s / sum_s e^{m_s - m} l_s  (0 when every split is empty).
// The (m, l) pairs are staged first so that every global load below is
// independent of the others (no chain of round trips per split).
template <typename Out>
__device__ void merge_splits(const float* __restrict__ ml, const float* __restrict__ o, int splits, int rows,
                             int stride, float* scratch, Out out) {
  float* sm_w = scratch;                  // [splits][rows]: m, then the weight e^{m_s - m}
  float* sm_l = scratch + splits * rows;  // [splits][rows]
  float* sm_L = sm_l + splits * rows;     // [rows]
  for (int i = threadIdx.x; i < splits * rows; i += blockDim.x) {
    const int sp = i / rows, n = i % rows;
    const float2 v = __ldcg(reinterpret_cast<const float2*>(ml) + (size_t)sp * stride + n);
    sm_w[i] = v.x;
    sm_l[i] = v.y;
  }
  __syncthreads();
  for (int n = threadIdx.x; n < rows; n += blockDim.x) {
    float mx = -INFINITY;
    for (int sp = 0; sp < splits; ++sp) mx = fmaxf(mx, sm_w[sp * rows + n]);
    float L = 0.0f;
    for (int sp = 0; sp < splits; ++sp) {
      const float w = merge_scale(sm_w[sp * rows + n], mx);
      sm_w[sp * rows + n] = w;
      L = fmaf(w, sm_l[sp * rows + n], L);
    }
    sm_L[n] = L;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rows * kHeadDim; e += blockDim.x) {
    const int n = e / kHeadDim, d = e % kHeadDim;
    const float* on = o + (size_t)n * kHeadDim + d;
    const size_t sstride = (size_t)stride * kHeadDim;
    float acc = 0.0f;
    int sp = 0;
    for (; sp + 4 <= splits; sp += 4) {
      const float v0 = __ldcg(on + (sp + 0) * sstride), v1 = __ldcg(on + (sp + 1) * sstride);
      const float v2 = __ldcg(on + (sp + 2) * sstride), v3 = __ldcg(on + (sp + 3) * sstride);
      acc = fmaf(sm_w[(sp + 0) * rows + n], v0, acc);
      acc = fmaf(sm_w[(sp + 1) * rows + n], v1, acc);
      acc = fmaf(sm_w[(sp + 2) * rows + n], v2, acc);
      acc = fmaf(sm_w[(sp + 3) * rows + n], v3, acc);
    }
    for (; sp < splits; ++sp) acc = fmaf(sm_w[sp * rows + n], __ldcg(on + sp * sstride), acc);
    const float L = sm_L[n];
    out(n, d, L > 0.0f ? acc / L : 0.0f);
  }
}

}  // namespace tf
