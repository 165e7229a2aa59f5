// The retrieval drafter's cache packed into a resident buffer of its own.
//
// "TriForce: Lossless Acceleration of Long Sequence Generation with
// Hierarchical Speculative Decoding", "Abstract (arXiv)": the retrieval-sparse
// KV cache is the middle draft level, and in the offloading setting the full
// cache lives in host memory (the project summary's "How It Works": KV cache
// offloaded to CPU memory).  The retrieval drafter only ever reads the rows of
// its selected chunks, so those rows can stay on the GPU: this call copies the
// valid tokens of every listed chunk, in list order, from row 0 of a
// [kc * 8]-row buffer per (b, g), reading the full cache from device memory or,
// over the host link, from pinned host memory.
//
// Design: a grid of (list slices, units) CTAs.  Every CTA of a unit recomputes
// the unit's packed offsets itself: each thread loads its run of the <= kc
// listed ids at once, and one block-wide scan of their valid row counts gives
// every entry's first packed row (a single round trip, no chain of dependent
// loads); the CTA keeps those of its own slice of 64 entries.  It then copies
// that slice: 8 rows of K and of V per chunk (4 KiB), 16 bytes per thread,
// eight chunks in flight.  No CTA waits on another.
#include "tf_common.cuh"

namespace tf {
namespace {

constexpr int kPackThreads = 256;     // 128 threads for a chunk's K rows, 128 for its V rows
constexpr int kPackMaxList = 4096;    // listed chunks per unit
constexpr int kPackPerThread = kPackMaxList / kPackThreads;  // ids scanned per thread
constexpr int kPackChunksPerCta = 64;
constexpr int kPackInFlight = 8;

// Plain (coherent) 16-byte load: the source may be host memory.
__device__ __forceinline__ uint4 ld_global16(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kPackThreads) pack_kernel(const uint16_t* K, const uint16_t* V,
                                                            const int32_t* __restrict__ seq_lens,
                                                            const int32_t* __restrict__ idx,
                                                            const int32_t* __restrict__ n_sel, int Hkv, int Lmax,
                                                            int kc, uint16_t* __restrict__ Kc,
                                                            uint16_t* __restrict__ Vc, int32_t* __restrict__ lens,
                                                            int32_t* __restrict__ n_chunks) {
  __shared__ int s_c[kPackChunksPerCta];    // chunk id of each entry of this CTA's slice, -1 if not a valid chunk
  __shared__ int s_off[kPackChunksPerCta];  // its first packed row
  __shared__ int s_wsum[kPackThreads / 32];
  const int unit = blockIdx.y;
  const int b = unit / Hkv;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  pdl_wait();
  const int L = clamp_len(seq_lens[b], Lmax);
  const int C = (L + kChunk - 1) / kChunk;
  int ns = n_sel[unit];
  ns = ns < 0 ? 0 : (ns > kc ? kc : ns);
  const int i0 = blockIdx.x * kPackChunksPerCta;
  const int i1 = min(ns, i0 + kPackChunksPerCta);

  // Exclusive scan of the entries' valid row counts: thread t owns entries
  // [t * q, (t + 1) * q), all its ids loaded together.
  const int q = (ns + kPackThreads - 1) / kPackThreads;  // <= kPackPerThread
  int cid[kPackPerThread], rows[kPackPerThread];
  int mine = 0;
#pragma unroll
  for (int k = 0; k < kPackPerThread; ++k) {
    const int e = t * q + k;
    cid[k] = (k < q && e < ns) ? idx[(size_t)unit * kc + e] : -1;
  }
#pragma unroll
  for (int k = 0; k < kPackPerThread; ++k) {
    const int c = cid[k];
    rows[k] = (c >= 0 && c < C) ? min(kChunk, L - c * kChunk) : 0;  // an id outside the context adds no row
    mine += rows[k];
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int run = incl - mine;
  for (int w = 0; w < warp; ++w) run += s_wsum[w];
#pragma unroll
  for (int k = 0; k < kPackPerThread; ++k) {
    const int e = t * q + k;
    if (k < q && e >= i0 && e < i1) {
      s_c[e - i0] = rows[k] > 0 ? cid[k] : -1;
      s_off[e - i0] = run;
    }
    run += rows[k];
  }
  if (t == kPackThreads - 1 && blockIdx.x == 0) {
    lens[unit] = run;  // the last thread's running total is the unit's row count
    n_chunks[unit] = (run + kChunk - 1) / kChunk;
  }
  __syncthreads();

  const bool is_v = t >= kPackThreads / 2;
  const int r = (t >> 4) & 7;  // row within the chunk
  const int piece = t & 15;    // 16-byte piece within the row
  const size_t cap = (size_t)kc * kChunk;
  const uint16_t* src = (is_v ? V : K) + (size_t)unit * Lmax * kHeadDim + piece * 8;
  uint16_t* dst = (is_v ? Vc : Kc) + (size_t)unit * cap * kHeadDim + piece * 8;
  for (int i = i0; i < i1; i += kPackInFlight) {
    uint4 v[kPackInFlight];
    int drow[kPackInFlight];
#pragma unroll
    for (int u = 0; u < kPackInFlight; ++u) {
      const int e = i + u;
      drow[u] = -1;
      if (e < i1) {
        const int c = s_c[e - i0];
        if (c >= 0 && r < min(kChunk, L - c * kChunk) && TF_DBG_OK(c * kChunk + r < L && L <= Lmax, kDbgCacheRow) &&
            TF_DBG_OK(s_off[e - i0] + r < (int)cap, kDbgPacked)) {
          drow[u] = s_off[e - i0] + r;
          v[u] = ld_global16(src + ((size_t)c * kChunk + r) * kHeadDim);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kPackInFlight; ++u)
      if (drow[u] >= 0) *reinterpret_cast<uint4*>(dst + (size_t)drow[u] * kHeadDim) = v[u];
  }
}

// Whether a kernel on the current device may read p: device memory of this
// device, managed memory, or host memory the CUDA runtime pinned or registered
// (reached through the same address under unified addressing).
bool kernel_readable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // a failed query leaves a (non-sticky) error behind: clear it
    return false;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  switch (a.type) {
    case cudaMemoryTypeDevice: return a.device == dev;
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return a.devicePointer == p;
    default: return false;
  }
}

}  // namespace

TF_DBG_READER(dbg_read_pack)

}  // namespace tf

extern "C" tf_status tf_pack_retrieval_cache(const uint16_t* K, const uint16_t* V, const int32_t* seq_lens,
                                             const int32_t* idx, const int32_t* n_sel, int B, int Hkv, int Lmax,
                                             int D, int chunk, int kc, uint16_t* Kc, uint16_t* Vc, int32_t* lens,
                                             int32_t* n_chunks, tf_stream_t stream) {
  using namespace tf;
  if (!K || !V || !seq_lens || !idx || !n_sel || !Kc || !Vc || !lens || !n_chunks) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hkv <= 0 || Lmax < 0 || kc <= 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(Kc) || !aligned16(Vc)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (kc > kPackMaxList) return TF_ERR_UNSUPPORTED;
  const long long units = (long long)B * Hkv;
  if (units == 0) return TF_OK;
  if (units > 65535) return TF_ERR_UNSUPPORTED;
  if (!kernel_readable(K) || !kernel_readable(V)) return TF_ERR_INVALID_ARG;
  const int slices = (kc + kPackChunksPerCta - 1) / kPackChunksPerCta;
  if (launch_pdl(pack_kernel, dim3((unsigned)slices, (unsigned)units), dim3(kPackThreads), 0, (cudaStream_t)stream,
                 K, V, seq_lens, idx, n_sel, Hkv, Lmax, kc, Kc, Vc, lens, n_chunks) != cudaSuccess)
    return TF_ERR_CUDA;
  return launch_status();
}
