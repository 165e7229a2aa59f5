// a2 + a3 -- chunk scores and top-k selection for the Force 2 retrieval drafter.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": Force 2 keeps a small top-k subset of the KV blocks, chosen by
// key-query similarity.  Score of chunk c for (sequence b, KV head g):
//   s = (sum of the group's query heads) . M[b, g, c, :]   (fp32 accumulation)
// Selection: the kc largest scores, equal scores to the lower chunk id, ids
// written in ascending order.
//
// Design: one thread-block cluster per (b, g) unit, S <= 8 CTAs, CTA r owning
// the r-th contiguous slice of the unit's chunks.  Each CTA streams its chunk
// means (a half-warp per 256-byte mean row, 16-byte loads, several in flight)
// and keeps its scores in shared memory as order-preserving uint32 keys with a
// histogram of their top 11 bits.  The selection then runs on the whole
// cluster at once through distributed shared memory: every CTA sums the S
// histograms and finds the bin holding the kc-th largest key (all CTAs reach
// the same answer); each CTA publishes its keys of that bin and its count of
// keys above it; every CTA gathers those few keys, resolves the remaining 21
// bits and every CTA's output offset by itself, and writes its own winners in
// id order.  Three cluster barriers in all; scores never leave the chip and no
// CTA waits on another except at those barriers (hardware, no spinning).
#include "sm100_ptx.cuh"
#include "tf_common.cuh"

namespace tf {
namespace {

using namespace sm100;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 6;
constexpr int kMaxCluster = 8;
constexpr int kMaxSliceKeys = 16384;  // keys per CTA held in shared memory (64 KB)
constexpr int kCandCap = 4096;        // keys of the threshold bin gathered on every CTA

// Thread t owns nb / kThreads bins of h (thread 0 the highest); find the bin
// holding the krem-th largest key.  All threads; result in s_bin / s_krem.
__device__ __forceinline__ void find_bin(const uint32_t* h, int nb, int krem, int* s_wsum, int* s_bin,
                                         int* s_krem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int k = nb / kThreads;
  const int top = nb - (int)threadIdx.x * k;
  int segsum = 0;
  for (int i = top - k; i < top; ++i) segsum += (int)h[i];
  int incl = segsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
  incl += wbase;
  const int excl = incl - segsum;
  if (excl < krem && krem <= incl) {
    int run = excl;
    for (int i = top - 1; i >= top - k; --i) {
      const int c = (int)h[i];
      if (run + c >= krem) {
        *s_bin = i;
        *s_krem = krem - run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// tot[i] = sum over the cluster's CTAs of their local[i], i < nb (nb a multiple
// of 4, arrays 16-byte aligned): 16-byte remote loads, all ranks in flight.
__device__ __forceinline__ void cluster_sum(const uint32_t* local, uint32_t* tot, int nb, int S) {
  for (int i = 4 * threadIdx.x; i < nb; i += 4 * kThreads) {
    uint4 v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) v[r] = r < S ? dsmem_ld_v4(local + i, (uint32_t)r) : make_uint4(0, 0, 0, 0);
    uint4 t = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      t.x += v[r].x;
      t.y += v[r].y;
      t.z += v[r].z;
      t.w += v[r].w;
    }
    *reinterpret_cast<uint4*>(tot + i) = t;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 2) scores_topk_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ M, const int32_t* __restrict__ seq_lens,
    int Hq, int Hkv, int Lmax, int kc, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    float* __restrict__ s_cut) {
  extern __shared__ uint32_t keys[];  // this CTA's slice of score keys
  __shared__ float qs[kHeadDim];
  __shared__ __align__(16) uint32_t hist1[2048], hist2[2048], hist3[1024], tot[2048];
  __shared__ uint32_t cand[kCandCap];   // this CTA's keys of the threshold bin (read by the cluster)
  __shared__ uint32_t gcand[kCandCap];  // the cluster's keys of the threshold bin
  __shared__ int s_ncand, s_above, s_roff[kMaxCluster + 1], s_rgt[kMaxCluster], s_req[kMaxCluster];
  __shared__ int s_wsum[kWarps], s_bin, s_krem;
  __shared__ uint32_t s_counts[2];  // keys > T and keys == T in this slice (or the slice's min key)
  __shared__ int s_wgt[kWarps], s_weq[kWarps];

  const int S = (int)gridDim.x;  // the cluster spans grid x
  const uint32_t rank = cluster_ctarank();
  const int unit = blockIdx.y;
  const int b = unit / Hkv, g = unit % Hkv;
  const int G = Hq / Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;

  for (int i = threadIdx.x; i < 2048; i += kThreads) {
    hist1[i] = 0;
    hist2[i] = 0;
  }
  for (int i = threadIdx.x; i < 1024; i += kThreads) hist3[i] = 0;
  pdl_wait();
  const int L = clamp_len(seq_lens[b], Lmax);
  const int C = (L + kChunk - 1) / kChunk;
  const int per = (C + S - 1) / S;
  const int c0 = min(C, (int)rank * per);
  const int c1 = min(C, c0 + per);
  const int n = c1 - c0;

  if (threadIdx.x < kHeadDim) {
    float s = 0.0f;
    for (int h = 0; h < G; ++h)
      s += __uint_as_float((uint32_t)q[((size_t)b * Hq + (size_t)g * G + h) * kHeadDim + threadIdx.x] << 16);
    qs[threadIdx.x] = s;
  }
  __syncthreads();

  // ---- scoring of this CTA's slice into shared memory
  {
    const int half = (threadIdx.x >> 4) & 1, l16 = threadIdx.x & 15, wid = threadIdx.x >> 5;
    float qv[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) qv[d] = qs[l16 * 8 + d];
    const uint16_t* Mu = M + (size_t)unit * Cmax * kHeadDim + l16 * 8;
    constexpr int kHalfWarps = kThreads / 16;
    // The loop bound is warp-uniform (the shuffles need the whole warp); each
    // half-warp owns chunk base + half + u * kHalfWarps.
    for (int base = c0 + 2 * wid; base < c1; base += kHalfWarps * kUnroll) {
      const int cb = base + half;
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = cb + u * kHalfWarps;
        v[u] = (c < c1) ? ld_stream16(Mu + (size_t)c * kHeadDim) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float f[8];
        unpack8(v[u], f);
        float s = 0.0f;
#pragma unroll
        for (int d = 0; d < 8; ++d) s = fmaf(qv[d], f[d], s);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        const int c = cb + u * kHalfWarps;
        if (l16 == 0 && c < c1) {
          const uint32_t key = score_key(s);
          keys[c - c0] = key;
          atomicAdd(&hist1[key >> 21], 1u);
        }
      }
    }
  }
  __syncthreads();
  int32_t* out = idx + (size_t)unit * kc;

  if (C <= kc) {
    // Every chunk is selected: ids in order, slots past C hold -1, s_cut = min score.
    uint32_t mn = 0xffffffffu;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      out[c0 + i] = c0 + i;
      mn = min(mn, keys[i]);
    }
    if (rank == 0)
      for (int i = C + (int)threadIdx.x; i < kc; i += kThreads) out[i] = -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if (threadIdx.x == 0) s_counts[0] = 0xffffffffu;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicMin(&s_counts[0], mn);
    cluster_sync();
    if (rank == 0 && threadIdx.x == 0) {
      uint32_t m = 0xffffffffu;
      for (int r = 0; r < S; ++r) m = min(m, dsmem_ld_u32(&s_counts[0], (uint32_t)r));
      n_sel[unit] = C;
      if (s_cut) s_cut[unit] = (C > 0) ? key_score(m) : -INFINITY;
    }
    cluster_sync();  // keep shared memory alive until rank 0 has read it
    return;
  }

  // ---- round 1: the cluster's histogram of the top 11 key bits -> bin b1
  cluster_sync();
  cluster_sum(hist1, tot, 2048, S);
  find_bin(tot, 2048, kc, s_wsum, &s_bin, &s_krem);
  const uint32_t b1 = (uint32_t)s_bin;
  const int krem1 = s_krem;
  const int ncand_tot = (int)tot[b1];  // keys of bin b1 over the cluster (same on every CTA)

  uint32_t T;
  int take_eq;
  int cta_eq = 0, cta_sel = 0;  // equal keys and selected ids in the CTAs before this one
  if (ncand_tot <= kCandCap) {
    // ---- round 2: publish this slice's keys of bin b1 and its count of keys
    // above the bin; every CTA gathers all lists and resolves the last 21 bits
    // and all output offsets by itself.
    if (threadIdx.x == 0) {
      s_ncand = 0;
      s_above = 0;
    }
    __syncthreads();
    {
      int above = 0;
      constexpr int k4 = 2048 / kThreads;
      for (int i = threadIdx.x * k4; i < ((int)threadIdx.x + 1) * k4; ++i) above += (uint32_t)i > b1 ? (int)hist1[i] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
      if ((threadIdx.x & 31) == 0) atomicAdd(&s_above, above);
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        if ((key >> 21) == b1) cand[atomicAdd(&s_ncand, 1)] = key;  // at most ncand_tot <= kCandCap
      }
    }
    cluster_sync();
    if (threadIdx.x < 32) {
      const int r = threadIdx.x;
      const int nc = r < S ? (int)dsmem_ld_u32(&s_ncand, (uint32_t)r) : 0;
      int incl = nc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (r >= o) incl += v;
      }
      if (r < S) {
        s_roff[r] = incl - nc;
        s_rgt[r] = (int)dsmem_ld_u32(&s_above, (uint32_t)r);
        s_req[r] = 0;
      }
      if (r == S - 1) s_roff[S] = incl;
    }
    __syncthreads();
    // one remote load per gathered key, all ranks at once
    for (int i = threadIdx.x; i < ncand_tot; i += kThreads) {
      int r = 0;
      while (r + 1 < S && i >= s_roff[r + 1]) ++r;
      gcand[i] = dsmem_ld_u32(cand + (i - s_roff[r]), (uint32_t)r);
    }
    __syncthreads();
    // bits 20..10, then 9..0, among the gathered keys (all of them are in bin b1)
    for (int i = threadIdx.x; i < ncand_tot; i += kThreads) atomicAdd(&hist2[(gcand[i] >> 10) & 2047u], 1u);
    __syncthreads();
    find_bin(hist2, 2048, krem1, s_wsum, &s_bin, &s_krem);
    const uint32_t pre2 = (b1 << 11) | (uint32_t)s_bin;
    const int krem2 = s_krem;
    for (int i = threadIdx.x; i < ncand_tot; i += kThreads) {
      const uint32_t key = gcand[i];
      if ((key >> 10) == pre2) atomicAdd(&hist3[key & 1023u], 1u);
    }
    __syncthreads();
    find_bin(hist3, 1024, krem2, s_wsum, &s_bin, &s_krem);
    T = (pre2 << 10) | (uint32_t)s_bin;
    take_eq = s_krem;
    // per-CTA counts of keys > T and == T among the gathered keys
    for (int i = threadIdx.x; i < ncand_tot; i += kThreads) {
      const uint32_t key = gcand[i];
      int r = 0;
      while (r + 1 < S && i >= s_roff[r + 1]) ++r;
      if (key > T) atomicAdd(&s_rgt[r], 1);
      if (key == T) atomicAdd(&s_req[r], 1);
    }
    __syncthreads();
    for (int r = 0; r < (int)rank; ++r) {
      cta_sel += s_rgt[r] + min(max(take_eq - cta_eq, 0), s_req[r]);
      cta_eq += s_req[r];
    }
  } else {
    // ---- rare (huge ties or a flat score range): resolve the last 21 bits with
    // two more cluster-wide histogram rounds, then exchange exact counts.
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key >> 21) == b1) atomicAdd(&hist2[(key >> 10) & 2047u], 1u);
    }
    cluster_sync();
    cluster_sum(hist2, tot, 2048, S);
    find_bin(tot, 2048, krem1, s_wsum, &s_bin, &s_krem);
    const uint32_t pre2 = (b1 << 11) | (uint32_t)s_bin;
    const int krem2 = s_krem;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key >> 10) == pre2) atomicAdd(&hist3[key & 1023u], 1u);
    }
    cluster_sync();
    cluster_sum(hist3, tot, 1024, S);
    find_bin(tot, 1024, krem2, s_wsum, &s_bin, &s_krem);
    T = (pre2 << 10) | (uint32_t)s_bin;
    take_eq = s_krem;
    {
      int ngt = 0, neq = 0;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        ngt += key > T;
        neq += key == T;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
        neq += __shfl_xor_sync(0xffffffffu, neq, o);
      }
      if (threadIdx.x == 0) {
        s_counts[0] = 0;
        s_counts[1] = 0;
      }
      __syncthreads();
      if ((threadIdx.x & 31) == 0) {
        atomicAdd(&s_counts[0], (uint32_t)ngt);
        atomicAdd(&s_counts[1], (uint32_t)neq);
      }
    }
    cluster_sync();
    for (int r = 0; r < (int)rank; ++r) {
      const int gt_r = (int)dsmem_ld_u32(&s_counts[0], (uint32_t)r);
      const int eq_r = (int)dsmem_ld_u32(&s_counts[1], (uint32_t)r);
      cta_sel += gt_r + min(max(take_eq - cta_eq, 0), eq_r);
      cta_eq += eq_r;
    }
  }

  // ---- id-order compaction of this slice: warp w owns local ids [w * seg, (w + 1) * seg)
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int w0 = warp * seg, w1 = min(n, w0 + seg);
    const unsigned lt = (1u << lane) - 1u;
    int ngt = 0, neq = 0;
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      const uint32_t key = i < w1 ? keys[i] : 0u;
      ngt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > T));
      neq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == T));
    }
    if (lane == 0) {
      s_wgt[warp] = ngt;
      s_weq[warp] = neq;
    }
    __syncthreads();
    int eq_base = cta_eq, sel_base = cta_sel;
    for (int w = 0; w < warp; ++w) {
      sel_base += s_wgt[w] + min(max(take_eq - eq_base, 0), s_weq[w]);
      eq_base += s_weq[w];
    }
    for (int base = w0; base < w1; base += 32) {
      const int i = base + lane;
      const uint32_t key = i < w1 ? keys[i] : 0u;
      const bool gt = i < w1 && key > T;
      const bool eq = i < w1 && key == T;
      const unsigned beq = __ballot_sync(0xffffffffu, eq);
      const bool sel = gt || (eq && eq_base + __popc(beq & lt) < take_eq);
      const unsigned bsel = __ballot_sync(0xffffffffu, sel);
      const int pos = sel_base + __popc(bsel & lt);
      if (sel && pos < kc) out[pos] = c0 + i;
      eq_base += __popc(beq);
      sel_base += __popc(bsel);
    }
  }
  if (rank == 0 && threadIdx.x == 0) {
    n_sel[unit] = kc;
    if (s_cut) s_cut[unit] = key_score(T);
  }
  cluster_sync();  // no CTA leaves while another may still read its counts
}

}  // namespace
}  // namespace tf

extern "C" size_t tf_chunk_scores_topk_workspace(int B, int Hkv, int Lmax, int chunk) {
  (void)B;
  (void)Hkv;
  (void)Lmax;
  (void)chunk;
  return 0;  // scores and the selection stay in (distributed) shared memory
}

extern "C" tf_status tf_chunk_scores_topk(const uint16_t* q, const uint16_t* M, const int32_t* seq_lens, int B,
                                          int Hq, int Hkv, int Lmax, int D, int chunk, int kc, int32_t* idx,
                                          int32_t* n_sel, float* s_cut, void* ws, size_t ws_bytes,
                                          tf_stream_t stream) {
  using namespace tf;
  (void)ws;
  (void)ws_bytes;
  if (!q || !M || !seq_lens || !idx || !n_sel) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv != 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(M)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const int units = B * Hkv;
  if (units > 65535) return TF_ERR_UNSUPPORTED;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;

  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(scores_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSliceKeys * (int)sizeof(uint32_t)) != cudaSuccess)
      return TF_ERR_CUDA;
    configured = true;
  }
  // Cluster size: the largest S <= 8 (at most one CTA per 64 chunks) whose
  // units x S CTAs fit one wave at the occupancy their slice size allows; at
  // least enough CTAs that every slice fits on chip.
  const int sms = num_sms();
  const int need = (Cmax + kMaxSliceKeys - 1) / kMaxSliceKeys;
  if (need > kMaxCluster) return TF_ERR_UNSUPPORTED;  // context beyond 8 x 16384 chunks
  int most = (Cmax + 63) / 64;
  if (most > kMaxCluster) most = kMaxCluster;
  int S = need;
  for (int cand_s = most; cand_s >= need; --cand_s) {
    const int sl = (Cmax + cand_s - 1) / cand_s;
    const int occ = occupancy_blocks((const void*)scores_topk_kernel, kThreads, (size_t)sl * sizeof(uint32_t));
    if ((long long)units * cand_s <= (long long)sms * occ) {
      S = cand_s;
      break;
    }
  }
  if (S < 1) S = 1;
  const int slice = (Cmax + S - 1) / S;
  const size_t dyn = (size_t)slice * sizeof(uint32_t);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, scores_topk_kernel, q, M, seq_lens, Hq, Hkv, Lmax, kc, idx, n_sel, s_cut) !=
      cudaSuccess)
    return TF_ERR_CUDA;
  return launch_status();
}
