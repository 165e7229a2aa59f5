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
#include "topk_select.cuh"

namespace tf {
namespace {

using namespace sm100;
using topk::kThreads;
using topk::kMaxCluster;
using topk::kMaxSliceKeys;

constexpr int kCandCap = 4096;  // keys of the threshold bin gathered on every CTA

__global__ void __launch_bounds__(kThreads, 2) scores_topk_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ M, const int32_t* __restrict__ seq_lens,
    int Hq, int Hkv, int Lmax, int kc, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
    float* __restrict__ s_cut) {
  extern __shared__ uint32_t keys[];  // this CTA's slice of score keys
  __shared__ float qs[kHeadDim];
  __shared__ __align__(16) uint32_t hist1[2048], hist2[2048], hist3[1024], tot[2048];
  __shared__ uint32_t cand[kCandCap], gcand[kCandCap];
  __shared__ uint32_t s_min;

  const topk::Arrays a{keys, hist1, hist2, hist3, tot, cand, gcand, kCandCap};
  const int S = (int)gridDim.x;  // the cluster spans grid x
  const uint32_t rank = cluster_ctarank();
  const int unit = blockIdx.y;
  const int b = unit / Hkv, g = unit % Hkv;
  const int G = Hq / Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;

  topk::zero_hists(a);
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
  topk::score_slice(qs, M + (size_t)unit * Cmax * kHeadDim, c0, c1, a, Cmax);
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
    if (threadIdx.x == 0) s_min = 0xffffffffu;
    __syncthreads();
    if ((threadIdx.x & 31) == 0) atomicMin(&s_min, mn);
    cluster_sync();
    if (rank == 0 && threadIdx.x == 0) {
      uint32_t m = 0xffffffffu;
      for (int r = 0; r < S; ++r) m = min(m, dsmem_ld_u32(&s_min, (uint32_t)r));
      n_sel[unit] = C;
      if (s_cut) s_cut[unit] = (C > 0) ? key_score(m) : -INFINITY;
    }
    cluster_sync();  // keep shared memory alive until rank 0 has read it
    return;
  }

  const topk::Round1 r1 = topk::round1(a, kc, S);
  const topk::Cut cut = r1.ncand_tot <= kCandCap ? topk::fast_cut(a, n, S, rank, r1, topk::CtaBar())
                                                 : topk::fallback_cut(a, n, S, rank, r1);
  topk::compact(a, n, kc, cut, topk::CtaBar(), [&](int i, int pos, bool) { out[pos] = c0 + i; });
  if (rank == 0 && threadIdx.x == 0) {
    n_sel[unit] = kc;
    if (s_cut) s_cut[unit] = key_score(cut.T);
  }
  cluster_sync();  // no CTA leaves while another may still read its counts
}

}  // namespace
TF_DBG_READER(dbg_read_topk)

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

  static DeviceCache configured;
  if (!configured.get([] {
        return cudaFuncSetAttribute(scores_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kMaxSliceKeys * (int)sizeof(uint32_t)) == cudaSuccess;
      }))
    return TF_ERR_CUDA;
  // Cluster size: the largest S <= 8 (at most one CTA per 64 chunks) whose
  // units x S CTAs fit one wave at the occupancy their slice size allows; at
  // least enough CTAs that every slice fits on chip.
  const int sms = num_sms();
  const int need = (Cmax + kMaxSliceKeys - 1) / kMaxSliceKeys;
  if (need > topk::kMaxPortableCluster) return TF_ERR_UNSUPPORTED;  // context beyond 8 x 16384 chunks
  int most = (Cmax + 63) / 64;
  if (most > topk::kMaxPortableCluster) most = topk::kMaxPortableCluster;
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
