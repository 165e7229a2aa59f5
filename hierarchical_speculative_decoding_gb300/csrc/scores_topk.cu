// a2 + a3 -- chunk scores and top-k selection for the Force 2 retrieval drafter.
//
// "TriForce: Hierarchical Speculative Decoding for LLMs", "The Three Forces of
// TriForce": Force 2 keeps a small top-k subset of the KV blocks, chosen by
// key-query similarity.  Score of chunk c for (sequence b, KV head g):
//   s = (sum of the group's query heads) . M[b, g, c, :]   (fp32 accumulation)
// Selection: the kc largest scores, equal scores to the lower chunk id, ids
// written in ascending order.
//
// Design: one kernel.  The (b, g) units are few (32 at batch 1) while each
// holds up to ~16K chunks, so every unit is split over several CTAs that stream
// the chunk means (a half-warp per 256-byte mean row, 16-byte loads), write fp32
// scores to the workspace and add the top 11 bits of each order-preserving
// uint32 score key to a per-unit histogram.  The last CTA of a unit to finish
// (an atomic ticket; no CTA ever waits) reads that histogram to find the bin
// holding the kc-th largest key, pulls the unit's keys into shared memory while
// collecting the few keys of that bin, resolves the remaining 21 bits on those
// candidates alone, and then compacts the winners in id order with two
// warp-segmented ballot walks, so ties resolve to the lower id without a sort.
#include "tf_common.cuh"

namespace tf {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;
constexpr int kBins = 2048;       // histogram over the top 11 key bits
constexpr int kSmemKeys = 16384;  // keys the selecting CTA keeps in shared memory (128K tokens)
constexpr int kCandCap = 2048;    // keys of the threshold bin resolved in shared memory

inline size_t tickets_bytes(int units) { return align_up((size_t)units * sizeof(int), 256); }
inline size_t hist_bytes(int units) { return (size_t)units * kBins * sizeof(uint32_t); }

// Warp 0 scans hist[0, nb) from the top and finds the bin holding the krem-th
// largest key; writes the bin and how many keys are still needed from it.
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int krem, int* s_bin, int* s_krem) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int seg = nb / 32;
    const int top = nb - lane * seg;  // lane 0 owns the highest bins
    int segsum = 0;
    for (int i = top - seg; i < top; ++i) segsum += (int)hist[i];
    int incl = segsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - segsum;
    if (excl < krem && krem <= incl) {
      int run = excl;
      for (int i = top - 1; i >= top - seg; --i) {
        const int h = (int)hist[i];
        if (run + h >= krem) {
          *s_bin = i;
          *s_krem = krem - run;
          break;
        }
        run += h;
      }
    }
  }
}

template <bool kSmem>
__device__ __forceinline__ uint32_t key_at(const uint32_t* keys, const float* scores, int c) {
  return kSmem ? keys[c] : score_key(__ldcg(scores + c));
}

// Select the kc largest of C > kc keys (ties to the lower id) and write their ids
// ascending.  hist holds the unit's top-11-bit histogram on entry.
template <bool kSmem>
__device__ __noinline__ void select_and_compact(const uint32_t* keys, const float* scores, int C, int kc, uint32_t* hist,
                                   uint32_t* cand, int32_t* out, uint32_t* thresh_out) {
  __shared__ int s_bin, s_krem, s_ncand;
  __shared__ int s_wgt[kWarps], s_weq[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // 1. the top-11-bit bin of the kc-th largest key
  find_bin(hist, kBins, kc, &s_bin, &s_krem);
  if (threadIdx.x == 0) s_ncand = 0;
  __syncthreads();
  const uint32_t b1 = (uint32_t)s_bin;
  int krem = s_krem;

  // 2. collect the keys of that bin
  for (int c = threadIdx.x; c < C; c += kThreads) {
    const uint32_t key = key_at<kSmem>(keys, scores, c);
    if ((key >> 21) == b1) {
      const int slot = atomicAdd(&s_ncand, 1);
      if (slot < kCandCap) cand[slot] = key;
    }
  }
  __syncthreads();
  const int ncand = s_ncand;
  const bool in_cand = ncand <= kCandCap;

  // 3. remaining 11 + 10 bits, on the candidates (or on all keys if the bin is huge)
  uint32_t prefix = b1 << 21, pmask = 0xFFE00000u;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0, nb = pass == 0 ? 2048 : 1024;
    const uint32_t mask = (uint32_t)nb - 1u;
    for (int i = threadIdx.x; i < nb; i += kThreads) hist[i] = 0;
    __syncthreads();
    const int n = in_cand ? ncand : C;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = in_cand ? cand[i] : key_at<kSmem>(keys, scores, i);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & mask], 1u);
    }
    __syncthreads();
    find_bin(hist, nb, krem, &s_bin, &s_krem);
    __syncthreads();
    prefix |= (uint32_t)s_bin << shift;
    pmask |= mask << shift;
    krem = s_krem;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const int take_eq = krem;

  // 4. id-order compaction: warp w owns ids [w * seg, (w + 1) * seg)
  const int seg = ((C + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = warp * seg, w1 = min(C, w0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  int ngt = 0, neq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int c = base + lane;
    const uint32_t key = c < w1 ? key_at<kSmem>(keys, scores, c) : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, c < w1 && key > T));
    neq += __popc(__ballot_sync(0xffffffffu, c < w1 && key == T));
  }
  if (lane == 0) {
    s_wgt[warp] = ngt;
    s_weq[warp] = neq;
  }
  __syncthreads();
  int eq_base = 0, sel_base = 0;
  for (int w = 0; w < warp; ++w) {
    const int take = min(max(take_eq - eq_base, 0), s_weq[w]);
    sel_base += s_wgt[w] + take;
    eq_base += s_weq[w];
  }
  for (int base = w0; base < w1; base += 32) {
    const int c = base + lane;
    const uint32_t key = c < w1 ? key_at<kSmem>(keys, scores, c) : 0u;
    const bool gt = c < w1 && key > T;
    const bool eq = c < w1 && key == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_base + __popc(beq & lt) < take_eq);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    const int pos = sel_base + __popc(bsel & lt);
    if (sel && pos < kc) out[pos] = c;
    eq_base += __popc(beq);
    sel_base += __popc(bsel);
  }
  *thresh_out = T;
}

__global__ void __launch_bounds__(kThreads, 2) scores_topk_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ M, const int32_t* __restrict__ seq_lens,
    int Hq, int Hkv, int Lmax, int kc, int splits, int smem_keys, int32_t* __restrict__ idx,
    int32_t* __restrict__ n_sel, float* __restrict__ s_cut, int* __restrict__ tickets,
    uint32_t* __restrict__ hist_ws, float* __restrict__ scores_ws) {
  extern __shared__ uint32_t keys_smem[];
  __shared__ float qs[kHeadDim];
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t cand[kCandCap];
  __shared__ int s_last;
  __shared__ float s_min[kWarps];

  const int unit = blockIdx.y;
  const int b = unit / Hkv, g = unit % Hkv;
  const int G = Hq / Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  const int L = clamp_len(seq_lens[b], Lmax);
  const int C = (L + kChunk - 1) / kChunk;
  float* scores = scores_ws + (size_t)unit * Cmax;
  uint32_t* hist_g = hist_ws + (size_t)unit * kBins;

  if (threadIdx.x < kHeadDim) {
    float s = 0.0f;
    for (int h = 0; h < G; ++h)
      s += __uint_as_float((uint32_t)q[((size_t)b * Hq + (size_t)g * G + h) * kHeadDim + threadIdx.x] << 16);
    qs[threadIdx.x] = s;
  }
  for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
  __syncthreads();

  // ---- scoring: this CTA's slice of the unit's chunks
  const int per = (C + splits - 1) / splits;
  const int c0 = blockIdx.x * per;
  const int c1 = min(C, c0 + per);
  const int half = (threadIdx.x >> 4) & 1, l16 = threadIdx.x & 15, wid = threadIdx.x >> 5;
  float qv[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) qv[d] = qs[l16 * 8 + d];
  const uint16_t* Mu = M + (size_t)unit * Cmax * kHeadDim + l16 * 8;
  constexpr int kHalfWarps = kThreads / 16;
  // The loop bound is warp-uniform (the shuffles below need the whole warp);
  // each half-warp owns chunk base + half + u * kHalfWarps.
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
        scores[c] = s;
        atomicAdd(&hist[score_key(s) >> 21], 1u);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (hist[i]) atomicAdd(&hist_g[i], hist[i]);

  // ---- ticket: the last CTA of this unit selects
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&tickets[unit], 1) == splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // the unit's histogram -> shared memory; leave the workspace copy zeroed
  for (int i = threadIdx.x; i < kBins; i += kThreads) {
    hist[i] = __ldcg(hist_g + i);
    hist_g[i] = 0u;
  }
  __syncthreads();

  int32_t* out = idx + (size_t)unit * kc;
  if (C <= kc) {
    float mn = INFINITY;
    for (int c = threadIdx.x; c < kc; c += kThreads) {
      out[c] = (c < C) ? c : -1;
      if (c < C) mn = fminf(mn, __ldcg(scores + c));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    if ((threadIdx.x & 31) == 0) s_min[threadIdx.x >> 5] = mn;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = INFINITY;
      for (int w = 0; w < kWarps; ++w) m = fminf(m, s_min[w]);
      n_sel[unit] = C;
      if (s_cut) s_cut[unit] = (C > 0) ? m : -INFINITY;
      tickets[unit] = 0;
    }
    return;
  }

  uint32_t T = 0;
  if (C <= smem_keys) {
    for (int c = threadIdx.x; c < C; c += kThreads) keys_smem[c] = score_key(__ldcg(scores + c));
    __syncthreads();
    select_and_compact<true>(keys_smem, scores, C, kc, hist, cand, out, &T);
  } else {
    select_and_compact<false>(keys_smem, scores, C, kc, hist, cand, out, &T);
  }
  if (threadIdx.x == 0) {
    n_sel[unit] = kc;
    if (s_cut) s_cut[unit] = key_score(T);
    tickets[unit] = 0;
  }
}

}  // namespace
}  // namespace tf

namespace {
int scores_splits(int units, int Cmax) {
  const int target = tf::num_sms() * 2;
  int s = (target + units - 1) / units;
  const int max_s = (Cmax + 63) / 64;
  if (s > max_s) s = max_s;
  return s < 1 ? 1 : s;
}
}  // namespace

extern "C" size_t tf_chunk_scores_topk_workspace(int B, int Hkv, int Lmax, int chunk) {
  if (B <= 0 || Hkv <= 0 || Lmax <= 0 || chunk != tf::kChunk) return 0;
  const size_t units = (size_t)B * Hkv;
  const size_t Cmax = (size_t)(Lmax + chunk - 1) / chunk;
  return tf::tickets_bytes((int)units) + tf::hist_bytes((int)units) + units * Cmax * sizeof(float);
}

extern "C" tf_status tf_chunk_scores_topk(const uint16_t* q, const uint16_t* M, const int32_t* seq_lens, int B,
                                          int Hq, int Hkv, int Lmax, int D, int chunk, int kc, int32_t* idx,
                                          int32_t* n_sel, float* s_cut, void* ws, size_t ws_bytes,
                                          tf_stream_t stream) {
  using namespace tf;
  if (!q || !M || !seq_lens || !idx || !n_sel) return TF_ERR_INVALID_ARG;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Lmax < 0 || kc <= 0 || Hq % Hkv != 0) return TF_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(M)) return TF_ERR_INVALID_ARG;
  if (D != kHeadDim || chunk != kChunk) return TF_ERR_UNSUPPORTED;
  if (B == 0 || Lmax == 0) return TF_OK;
  const size_t need = tf_chunk_scores_topk_workspace(B, Hkv, Lmax, chunk);
  if (!ws || ws_bytes < need || !aligned16(ws)) return TF_ERR_WORKSPACE;
  const int units = B * Hkv;
  const int Cmax = (Lmax + kChunk - 1) / kChunk;
  const int splits = scores_splits(units, Cmax);
  const int smem_keys = Cmax <= kSmemKeys ? Cmax : 0;
  const size_t dyn = (size_t)smem_keys * sizeof(uint32_t);
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(scores_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemKeys * (int)sizeof(uint32_t)) != cudaSuccess)
      return TF_ERR_CUDA;
    configured = true;
  }
  char* w = static_cast<char*>(ws);
  int* tickets = reinterpret_cast<int*>(w);
  uint32_t* hist = reinterpret_cast<uint32_t*>(w + tickets_bytes(units));
  float* scores = reinterpret_cast<float*>(w + tickets_bytes(units) + hist_bytes(units));
  dim3 grid(splits, units);
  scores_topk_kernel<<<grid, kThreads, dyn, stream>>>(q, M, seq_lens, Hq, Hkv, Lmax, kc, splits, smem_keys, idx,
                                                      n_sel, s_cut, tickets, hist, scores);
  return launch_status();
}
